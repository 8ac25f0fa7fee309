"""Pins the oracle's cache state machine and byte layout (CPU only).

Sources: KV-cache quantization guide (pigeon), "How it works", steps 1, 2, 4;
tract #2458 "quantized KV-cache storage op (int8/int4)": f32 sinks (sink
commit); its unit tests that a stream accumulated in pieces equals the stream
concatenated, and that per-channel blocks stay consistent while the range
grows (description); key-block scales that never change once written.
"""
import numpy as np
import pytest

from conftest import read_table


def P(oracle, **kw):
    base = dict(bits=4, group=32, residual=32, sinks=4, h_q=2, h_kv=2, head_dim=64, batch=2,
                max_tokens=512, window=0)
    base.update(kw)
    return oracle.Params(**base)


def stream(p, T, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    shape = (p.batch, p.h_kv, T, p.head_dim)
    k = (rng.standard_normal(shape) * scale).astype(np.float16)
    k[..., 3] *= 20  # an outlier channel
    v = (rng.standard_normal(shape) * scale).astype(np.float16)
    return k, v


def closed_form(T, S, R, G):
    """Test-side restatement of the lazy-flush state (derivation in
    tests/golden/cache_states.txt)."""
    m = max(T - S, 0)
    ng = 0 if m <= R else -(-(m - R) // G)
    return min(T, S), ng, m - ng * G


@pytest.mark.parametrize("row", read_table("cache_states.txt"), ids=lambda r: r[0])
def test_cache_state_golden(oracle_lib, row):
    name, T, S, R, G, W, ns, ng, nr, vq, slots = row
    T, S, R, G, W = int(T), int(S), int(R), int(G), int(W)
    p = P(oracle_lib, sinks=S, residual=R, group=G, window=W, batch=1, h_kv=1, h_q=1,
          max_tokens=0 if W else T)
    assert oracle_lib.state_of(p, T) == (int(ns), int(ng), int(nr))
    c = oracle_lib.Cache(p)
    k, v = stream(p, T, seed=1)
    assert c.append(k, v) == 0
    assert (c.T, c.n_groups, c.n_res) == (T, int(ng), int(nr))
    if slots != "-":
        assert c.layout["n_slots"] == int(slots)
    _, _, vis = c.dequant_unit(0, 0)
    q_tokens = np.arange(T)
    quantized = (q_tokens >= S) & (q_tokens < S + int(ng) * G)
    assert int((vis & quantized).sum()) == int(vq)


@pytest.mark.parametrize("S,R,G", [(0, 16, 16), (4, 32, 32), (4, 64, 16), (1, 48, 16), (7, 32, 16)])
def test_counters_match_closed_form_every_T(oracle_lib, S, R, G):
    p = P(oracle_lib, sinks=S, residual=R, group=G, batch=1, h_kv=1, h_q=1, max_tokens=600)
    c = oracle_lib.Cache(p)
    k, v = stream(p, 600, seed=2)
    for T in range(1, 601):
        assert c.append(k[:, :, T - 1:T], v[:, :, T - 1:T]) == 0
        assert (min(T, S), c.n_groups, c.n_res) == closed_form(T, S, R, G), T
        if T - S > R:
            assert R - G + 1 <= c.n_res <= R


@pytest.mark.parametrize("chunks", [[1] * 300, [300], [7, 64, 1, 128, 100], [36, 1, 263], [4, 33, 31, 232]])
@pytest.mark.parametrize("window", [0, 64])
def test_bulk_equals_sequential(oracle_lib, chunks, window):
    """tract #2458 (its test that accumulating a stream matches concatenating
    it): any chunking of the same stream yields the same bytes."""
    p = P(oracle_lib, window=window, max_tokens=0 if window else 300)
    k, v = stream(p, 300, seed=3)
    ref = oracle_lib.Cache(p)
    for t in range(300):
        assert ref.append(k[:, :, t:t + 1], v[:, :, t:t + 1]) == 0
    c = oracle_lib.Cache(p)
    t = 0
    for n in chunks:
        assert c.append(k[:, :, t:t + n], v[:, :, t:t + n]) == 0
        t += n
    assert np.array_equal(c.arena(), ref.arena())
    assert (c.T, c.n_groups, c.n_res) == (ref.T, ref.n_groups, ref.n_res)


def test_frozen_groups_never_change(oracle_lib):
    """tract #2458: key blocks keep frozen scales; bytes of a written group
    never change as the stream grows."""
    p = P(oracle_lib, max_tokens=700)
    k, v = stream(p, 700, seed=4)
    c = oracle_lib.Cache(p)
    L = c.layout
    seen = {}
    for t in range(700):
        c.append(k[:, :, t:t + 1], v[:, :, t:t + 1])
        arena = c.arena()
        for g in range(c.n_groups):
            for u in range(p.batch * p.h_kv):
                off = u * L["unit_bytes"] + L["groups"] + g * L["block_bytes"]
                blk = arena[off:off + L["block_bytes"]].copy()
                if (g, u) in seen:
                    assert np.array_equal(seen[(g, u)], blk), (t, g, u)
                else:
                    seen[(g, u)] = blk


def test_sinks_and_ring_hold_inputs(oracle_lib):
    p = P(oracle_lib, sinks=5, max_tokens=200)
    k, v = stream(p, 200, seed=5)
    c = oracle_lib.Cache(p)
    c.append(k, v)
    L = c.layout
    d = p.head_dim
    ar = c.arena()
    for b in range(p.batch):
        for h in range(p.h_kv):
            u = ar[(b * p.h_kv + h) * L["unit_bytes"]:][:L["unit_bytes"]]
            sk = u[L["sink_k"]:L["sink_k"] + 5 * d * 4].view(np.float32).reshape(5, d)
            sv = u[L["sink_v"]:L["sink_v"] + 5 * d * 4].view(np.float32).reshape(5, d)
            assert np.array_equal(sk, k[b, h, :5].astype(np.float32))
            assert np.array_equal(sv, v[b, h, :5].astype(np.float32))
            rk = u[L["res_k"]:L["res_k"] + p.residual * d * 2].view(np.float16).reshape(p.residual, d)
            rv = u[L["res_v"]:L["res_v"] + p.residual * d * 2].view(np.float16).reshape(p.residual, d)
            # the ring holds the last R tokens of the stream at slot (a - S) mod R
            for a in range(200 - p.residual, 200):
                s = (a - 5) % p.residual
                assert np.array_equal(rk[s], k[b, h, a]) and np.array_equal(rv[s], v[b, h, a])


# --- an independent, test-side decoder of the documented byte layout -------
def _unpack(packed, L, bits):
    if bits not in (2, 4, 8):   # bit stream: element j at bits [b j, b j + b), LSB first
        flat = np.unpackbits(packed, bitorder="little")[:L * bits].reshape(L, bits).astype(np.int64)
        return (flat << np.arange(bits)[None, :]).sum(axis=1)
    words = packed.view("<u4")
    per = 32 // bits
    j = np.arange(per)
    shifts = 16 * (j & 1) + bits * (j >> 1)
    codes = (words[:, None] >> shifts[None, :].astype(np.uint32)) & ((1 << bits) - 1)
    return codes.reshape(-1)[:L].astype(np.int64)


def decode_unit_numpy(arena_unit, p, L, T, n_groups):
    d, G, b, S, R = p.head_dim, p.group, p.bits, p.sinks, p.residual
    K = np.zeros((T, d))
    V = np.zeros((T, d))
    f16 = lambda off, n: arena_unit[off:off + 2 * n].view("<f2").astype(np.float64)
    for a in range(T):
        if a < S:
            K[a] = arena_unit[L["sink_k"] + a * d * 4:][:d * 4].view("<f4")
            V[a] = arena_unit[L["sink_v"] + a * d * 4:][:d * 4].view("<f4")
            continue
        g = (a - S) // G
        if g < n_groups:
            if n_groups - 1 - g >= L["n_slots"]:
                continue
            blk = L["groups"] + (g % L["n_slots"]) * L["block_bytes"]
            t = (a - S) - g * G
            row = _unpack(arena_unit[blk + L["blk_kq"] + t * d * b // 8:][:d * b // 8], d, b)
            dq = f16(blk + L["blk_ks"], d)
            mn = f16(blk + L["blk_ks"] + 2 * d, d)
            K[a] = mn + row * dq
            vs = f16(blk + L["blk_vs"] + 4 * t, 2)
            for ch in range(d):
                vr = _unpack(arena_unit[blk + L["blk_vq"] + ch * G * b // 8:][:G * b // 8], G, b)
                V[a, ch] = vs[1] + vr[t] * vs[0]
        else:
            s = (a - S) % R
            K[a] = f16(L["res_k"] + s * d * 2, d)
            V[a] = f16(L["res_v"] + s * d * 2, d)
    return K, V


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("G,d", [(16, 64), (32, 128)])
def test_independent_decoder_agrees(oracle_lib, bits, G, d):
    p = P(oracle_lib, bits=bits, group=G, residual=2 * G, head_dim=d, batch=1, h_kv=2, h_q=2, max_tokens=200)
    k, v = stream(p, 200, seed=6 + bits)
    c = oracle_lib.Cache(p)
    c.append(k, v)
    for h in range(2):
        K, V, vis = c.dequant_unit(0, h)
        K2, V2 = decode_unit_numpy(c.unit(0, h), p, c.layout, c.T, c.n_groups)
        assert np.array_equal(K, K2) and np.array_equal(V, V2)
        # and the decoded keys are within half a step of their inputs, where the
        # step is the channel's range over its group / (2^b - 1)
        kin = k[0, h].astype(np.float64)
        for g in range(c.n_groups):
            sl = slice(p.sinks + g * G, p.sinks + (g + 1) * G)
            step = (kin[sl].max(0) - kin[sl].min(0)) / ((1 << bits) - 1)
            assert np.all(np.abs(K[sl] - kin[sl]) <= 0.5 * step * (1 + 2.0 ** -9) + 1e-6)
        assert np.array_equal(K[c.p.sinks + c.n_groups * G:], kin[c.p.sinks + c.n_groups * G:])
        # values are quantized per token: half a step of the token's own range
        vin = v[0, h].astype(np.float64)
        q0, q1 = p.sinks, p.sinks + c.n_groups * G
        vstep = (vin[q0:q1].max(1) - vin[q0:q1].min(1)) / ((1 << bits) - 1)
        assert np.all(np.abs(V[q0:q1] - vin[q0:q1]) <= 0.5 * vstep[:, None] * (1 + 2.0 ** -9) + 1e-6)
        assert np.array_equal(V[q1:], vin[q1:]) and np.array_equal(V[:q0], vin[:q0])


def test_layout_sizes_closed_form(oracle_lib):
    # tiny workload: d=64, G=32, b=4, R=32, S=4, T_max=256 -> 7 slots
    p = P(oracle_lib, bits=4, group=32, residual=32, sinks=4, head_dim=64, batch=1, h_kv=4, h_q=4, max_tokens=256)
    L = oracle_lib.layout(p)
    block = 32 * 64 * 4 // 8 + 2 * 64 * 2 + 64 * 32 * 4 // 8 + 32 * 4
    assert L["block_bytes"] == block == 2432
    assert L["unit_bytes"] == 2 * 4 * 64 * 4 + 2 * 32 * 64 * 2 + 7 * block
    assert L["cache_bytes"] == 4 * L["unit_bytes"]
    for k in ("sink_v", "res_k", "res_v", "groups", "blk_ks", "blk_vq", "blk_vs", "block_bytes", "unit_bytes"):
        assert L[k] % 16 == 0, k   # every region starts on a 16-byte boundary


def test_window_slot_reuse_and_visibility(oracle_lib):
    p = P(oracle_lib, window=100, residual=32, group=16, sinks=3, batch=1, h_kv=1, h_q=1, max_tokens=0)
    c = oracle_lib.Cache(p)
    assert c.layout["n_slots"] == -(-100 // 16) + 1
    k, v = stream(p, 1000, seed=8)
    for t0 in range(0, 1000, 37):
        n = min(37, 1000 - t0)
        c.append(k[:, :, t0:t0 + n], v[:, :, t0:t0 + n])
        T = c.T
        K, V, vis = c.dequant_unit(0, 0)
        expect = np.zeros(T, bool)
        expect[:min(T, 3)] = True
        expect[max(T - 100, 0):] = True
        assert np.array_equal(vis, expect)
        # a visible quantized token is never in a slot that was overwritten:
        # it decodes to within half a step of its own input
        kin = k[0, 0, :T].astype(np.float64)
        for a in np.flatnonzero(vis):
            g = (a - 3) // 16
            if a < 3 or g >= c.n_groups:
                assert np.array_equal(K[a], kin[a])
                continue
            sl = slice(3 + g * 16, 3 + (g + 1) * 16)
            step = (kin[sl].max(0) - kin[sl].min(0)) / 15
            assert np.all(np.abs(K[a] - kin[a]) <= 0.5 * step * (1 + 2.0 ** -9) + 1e-6)


def test_capacity_and_validation(oracle_lib):
    p = P(oracle_lib, max_tokens=40)
    c = oracle_lib.Cache(p)
    k, v = stream(p, 41, seed=9)
    assert c.append(k[:, :, :40], v[:, :, :40]) == 0
    before = c.arena()
    assert c.append(k[:, :, 40:41], v[:, :, 40:41]) == 3
    assert c.T == 40 and np.array_equal(before, c.arena())
    bad = [dict(bits=0), dict(bits=9), dict(head_dim=96), dict(group=8), dict(group=24),
           dict(residual=16), dict(residual=48), dict(sinks=-1), dict(h_q=3), dict(window=16),
           dict(window=-1), dict(batch=0)]
    for kw in bad:
        assert oracle_lib.validate(P(oracle_lib, **kw)) == 1, kw
    assert oracle_lib.validate(P(oracle_lib)) == 0
