"""Pins the oracle's dense-and-sparse outliers (CPU only).

Source: KV-cache quantization guide (pigeon), "KVQuant adds": a small share
of the values (about one in a hundred) is kept in fp16 in a sparse table
beside the low-bit codes.  The readings fixed here: per frozen key block and
value block the n = ceil(permille G d / 1000) values of largest magnitude are
outliers (ties to the smaller flat index t d + c); they take no part in the
dense min and max, get code 0, are stored as rows by token (u16 row
pointers, then {u8 t, u8 c, fp16 x} entries in flat order), and dequantize
to x exactly.

The pins do not restate the quantizer: blocks whose dense part lies on a
2-bit grid reconstruct exactly only if the selection, the exclusion from the
ranges, the table and the override are all right; the tie order is worked by
hand; attention over an exactly reconstructed cache is the textbook softmax
of the raw keys and values.
"""
import numpy as np
import pytest


def P(oracle, **kw):
    base = dict(bits=2, group=16, residual=32, sinks=0, h_q=2, h_kv=1, head_dim=64, batch=1,
                max_tokens=400, window=0, outlier_permille=10)
    base.update(kw)
    return oracle.Params(**base)


def grid_block(rng, G, d):
    """Keys and values of one group whose every vector lies on its own 2-bit
    grid {min + k delta}, with k = 0 and k = 3 present at tokens 0, 1 (keys,
    per channel) and channels 0, 1 (values, per token): exact under a 2-bit
    quantizer over those vectors."""
    kd = 2.0 ** -rng.integers(0, 4, d)            # per-channel step
    kmn = -kd * rng.integers(0, 4, d)
    kk = rng.integers(0, 4, (G, d))
    kk[0], kk[1] = 0, 3
    K = kmn[None, :] + kk * kd[None, :]
    vd = 2.0 ** -rng.integers(0, 4, G)            # per-token step
    vmn = -vd * rng.integers(0, 4, G)
    vk = rng.integers(0, 4, (G, d))
    vk[:, 0], vk[:, 1] = 0, 3
    V = vmn[:, None] + vk * vd[:, None]
    return K, V


def plant(rng, X, n, rows, cols, base):
    """n distinct large values at distinct positions (row >= rows[0], col >=
    cols[0]); returns their flat positions."""
    G, d = X.shape
    pos = set()
    while len(pos) < n:
        pos.add((int(rng.integers(rows, G)), int(rng.integers(cols, d))))
    pos = sorted(pos, key=lambda tc: tc[0] * d + tc[1])
    mags = rng.permutation(n) + base
    for (t, c), m in zip(pos, mags):
        X[t, c] = m * (1 if rng.random() < 0.5 else -1)
    return pos


def stream_with(p, blocks, rng, tail):
    """A [1, 1, T, d] stream: the given groups, then `tail` N(0,1) tokens."""
    K = np.concatenate([b[0] for b in blocks] + [rng.standard_normal((tail, p.head_dim))])
    V = np.concatenate([b[1] for b in blocks] + [rng.standard_normal((tail, p.head_dim))])
    return K[None, None].astype(np.float16), V[None, None].astype(np.float16)


def table(c, slot, which, G=16):
    """The entries of a block's table; its row pointers are checked against
    them (row t holds exactly the entries of token t)."""
    L = c.layout
    blk = c.unit(0, 0)[L["groups"] + slot * L["block_bytes"]:][:L["block_bytes"]]
    off = L["blk_ko"] if which == "k" else L["blk_vo"]
    ptr = blk[off:off + 2 * (G + 1)].copy().view(np.uint16)
    raw = blk[off + L["out_entries"]:off + L["out_entries"] + 4 * L["n_outliers"]].reshape(-1, 4)
    vals = raw[:, 2:].copy().view(np.float16)[:, 0]
    ent = [(int(t), int(ch), float(x)) for (t, ch), x in zip(raw[:, :2], vals)]
    assert ptr[0] == 0 and ptr[G] == len(ent)
    for t in range(G):
        assert all(e[0] == t for e in ent[ptr[t]:ptr[t + 1]]), (t, ptr)
    return ent


def test_entry_count_and_layout(oracle_lib):
    L0 = oracle_lib.layout(P(oracle_lib, outlier_permille=0))
    L = oracle_lib.layout(P(oracle_lib))
    assert L0["n_outliers"] == 0 and L0["blk_ko"] == L0["blk_vo"] == L0["block_bytes"]
    assert L["n_outliers"] == 11                          # ceil(10 * 16 * 64 / 1000) = ceil(10.24)
    assert L["blk_ko"] == L0["block_bytes"]               # tables after the value scales
    assert L["out_entries"] == 36                         # 17 u16 row pointers, to a 4-byte boundary
    assert L["blk_vo"] - L["blk_ko"] == 80                # 36 + 44 bytes, padded to 16
    assert L["block_bytes"] == L0["block_bytes"] + 160
    assert oracle_lib.layout(P(oracle_lib, group=32, head_dim=128, outlier_permille=1))["n_outliers"] == 5
    assert oracle_lib.validate(P(oracle_lib, outlier_permille=50)) == 0
    for bad in (-1, 51):
        assert oracle_lib.validate(P(oracle_lib, outlier_permille=bad)) != 0


def test_grid_blocks_with_planted_outliers_reconstruct_exactly(oracle_lib):
    """Two frozen groups whose dense parts lie on 2-bit grids, with 11 planted
    key and 11 planted value outliers each: every frozen value comes back
    exactly and the tables hold the planted entries in flat order."""
    bits = 2
    rng = np.random.default_rng(5)
    p = P(oracle_lib, bits=bits)
    G, d = p.group, p.head_dim
    blocks, planted = [], []
    for g in range(2):
        K, V = grid_block(rng, G, d)
        pk = plant(rng, K, 11, 2, 0, 40 + 20 * g)
        pv = plant(rng, V, 11, 0, 2, 40 + 20 * g)
        blocks.append((K, V))
        planted.append((pk, pv))
    k, v = stream_with(p, blocks, rng, tail=30)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    assert c.n_groups == 2
    Kh, Vh, vis = c.dequant_unit(0, 0)
    assert vis.all()
    frozen = slice(0, 2 * G)
    np.testing.assert_array_equal(Kh[frozen], k[0, 0, frozen].astype(np.float64))
    np.testing.assert_array_equal(Vh[frozen], v[0, 0, frozen].astype(np.float64))
    for g in range(2):
        pk, pv = planted[g]
        Kg, Vg = blocks[g]
        assert table(c, g, "k") == [(t, ch, float(np.float16(Kg[t, ch]))) for t, ch in pk]
        assert table(c, g, "v") == [(t, ch, float(np.float16(Vg[t, ch]))) for t, ch in pv]
    # without the side table the planted values stretch the ranges: not exact
    c0 = oracle_lib.Cache(P(oracle_lib, bits=bits, outlier_permille=0))
    assert c0.append(k, v) == 0
    K0, _, _ = c0.dequant_unit(0, 0)
    assert np.abs(K0[frozen] - k[0, 0, frozen]).max() > 1.0


def test_ties_go_to_the_smaller_flat_index(oracle_lib):
    """Worked by hand: keys of magnitude 1 everywhere except -2 at (5, 7), 2 at
    (9, 0) and 2 at (12, 63).  With 11 outliers the three of magnitude 2 come
    first, then the 8 smallest flat indices among the ties: token 0, channels
    0..7.  The table lists all 11 in flat order."""
    rng = np.random.default_rng(1)
    p = P(oracle_lib)
    G, d = p.group, p.head_dim
    K = np.where(rng.random((G, d)) < 0.5, -1.0, 1.0)
    K[5, 7], K[9, 0], K[12, 63] = -2.0, 2.0, 2.0
    V = rng.standard_normal((G, d)) * 0.1
    k, v = stream_with(p, [(K, V)], rng, tail=32)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups == 1
    want = [(0, ch, K[0, ch]) for ch in range(8)] + [(5, 7, -2.0), (9, 0, 2.0), (12, 63, 2.0)]
    assert table(c, 0, "k") == want
    # row pointers worked by hand: 8 entries in row 0, one each in rows 5, 9, 12
    L = c.layout
    ptr = c.unit(0, 0)[L["groups"] + L["blk_ko"]:][:34].copy().view(np.uint16)
    assert ptr.tolist() == [0] + [8] * 5 + [9] * 4 + [10] * 3 + [11] * 4


def test_a_channel_of_outliers_only_gets_zero_scales(oracle_lib):
    """17 outliers (permille 16: ceil(16.384)), 16 of them the whole of key
    channel 5: that channel has no dense value left, its (delta, min) are 0
    and its codes 0, and it still comes back exactly."""
    rng = np.random.default_rng(2)
    p = P(oracle_lib, outlier_permille=16)
    G, d = p.group, p.head_dim
    K, V = grid_block(rng, G, d)
    K[:, 5] = 100.0 + np.arange(G)
    K[3, 40] = -300.0
    k, v = stream_with(p, [(K, V)], rng, tail=32)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups == 1
    L = c.layout
    blk = c.unit(0, 0)[L["groups"]:][:L["block_bytes"]]
    ks = blk[L["blk_ks"]:L["blk_ks"] + 4 * d].view(np.uint16)
    assert ks[5] == 0 and ks[d + 5] == 0
    row = d * p.bits // 8   # key codes: one packed row of d codes per token
    for t in range(G):
        codes = oracle_lib.unpack_row(blk[L["blk_kq"] + t * row:][:row], d, p.bits)
        assert codes[5] == 0
    Kh, _, _ = c.dequant_unit(0, 0)
    np.testing.assert_array_equal(Kh[:G], k[0, 0, :G].astype(np.float64))


def test_attention_over_an_exact_cache_is_the_textbook_softmax(oracle_lib):
    rng = np.random.default_rng(9)
    p = P(oracle_lib)
    G, d = p.group, p.head_dim
    blocks = []
    for g in range(3):
        K, V = grid_block(rng, G, d)
        plant(rng, K, 11, 2, 0, 8)
        plant(rng, V, 11, 0, 2, 8)
        blocks.append((K, V))
    k, v = stream_with(p, blocks, rng, tail=20)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups == 3
    q = rng.standard_normal((1, p.h_q, d)).astype(np.float16)
    out = c.decode_attn(q)
    Kr, Vr = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64)
    for h in range(p.h_q):
        s = Kr @ q[0, h].astype(np.float64) / np.sqrt(d)
        w = np.exp(s - s.max())
        np.testing.assert_allclose(out[0, h], (w[:, None] * Vr).sum(0) / w.sum(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_side_table_lowers_the_error_on_spiky_data(oracle_lib, bits):
    """N(0,1) keys and values with 1 % spikes of x20: keeping 1 % of the
    values exactly lowers the RMS reconstruction error of the frozen keys and
    values at least twice, and the attention error against fp64 attention
    over the raw values."""
    rng = np.random.default_rng(4)
    T, d = 16 * 12 + 32, 64
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    for X in (K, V):
        X[rng.random((T, d)) < 0.01] *= 20
    k = K[None, None].astype(np.float16)
    v = V[None, None].astype(np.float16)
    q = (rng.standard_normal((1, 2, d)) * 0.3).astype(np.float16)
    Kr, Vr = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64)
    exact = []
    for h in range(2):
        s = Kr @ q[0, h].astype(np.float64) / np.sqrt(d)
        w = np.exp(s - s.max())
        exact.append((w[:, None] * Vr).sum(0) / w.sum())
    exact = np.array(exact)
    res = {}
    for pm in (0, 10):
        c = oracle_lib.Cache(P(oracle_lib, bits=bits, outlier_permille=pm))
        assert c.append(k, v) == 0
        Kh, Vh, _ = c.dequant_unit(0, 0)
        n = c.n_groups * 16
        rms = lambda a, b: np.sqrt(((a[:n] - b[:n]) ** 2).mean())
        res[pm] = (rms(Kh, Kr), rms(Vh, Vr), np.abs(c.decode_attn(q)[0] - exact).max())
    assert res[10][0] * 2 < res[0][0] and res[10][1] * 2 < res[0][1], res
    assert res[10][2] < res[0][2], res
