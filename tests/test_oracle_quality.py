"""Quality and sizing pins of the oracle against what the pages state.

  * int8 is near-lossless for attention ("~0.5%" deviation) — tract #2329,
    "The idea" table; on synthetic keys with outlier channels the pin is
    int8 < 2% plus the table's ratios between bit widths.
  * per-channel keys beat per-token keys on outlier channels — tract #2329,
    "The idea"; KV-cache quantization guide (pigeon), "When it breaks".
  * 2 bits without a residual window loses precision on the recent tokens —
    pigeon guide, "When it breaks".
  * fp16 KV of a 7B model is 2 * 32 * 4096 * 2 B = 512 KiB per token —
    pigeon guide, "The idea".
  * packed u8 saves > 3x versus f32 — tract #2329, "Correctness & gates";
    memory is about bits/16 of the f16 cache — tract #2329 commit message.
  * a 4096-token window of a Mistral-shaped layer drops from ~33 MB (f32) to
    ~8 MB with int8 — tract #2329, "Relationship to other PRs".
The real GPT-2 / OpenELM figures need model weights and are not reproduced
(parity unpinned for those numbers).
"""
import numpy as np
import pytest


def deviation(o, ref):
    """‖o − o_ref‖₂ / ‖o_ref‖₂ per row, maximum over rows."""
    o = o.reshape(-1, o.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    return float((np.linalg.norm(o - ref, axis=1) / np.linalg.norm(ref, axis=1)).max())


def full_precision(q, k, v, rep):
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for hq in range(Hq):
            K = k[b, hq // rep].astype(np.float64)
            V = v[b, hq // rep].astype(np.float64)
            s = K @ q[b, hq].astype(np.float64) / np.sqrt(d)
            w = np.exp(s - s.max())
            out[b, hq] = (w[:, None] * V).sum(0) / w.sum()
    return out


def outlier_stream(B, H, T, d, seed, n_out=4, lo=10, hi=30):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, H, T, d))
    for h in range(H):
        for ch, sc in zip(rng.choice(d, n_out, replace=False), rng.uniform(lo, hi, size=n_out)):
            k[:, h, :, ch] *= sc
    v = rng.standard_normal((B, H, T, d)) * np.exp(0.5 * rng.standard_normal((B, H, T, 1)))
    q = rng.standard_normal((B, H, d))
    return k.astype(np.float16), v.astype(np.float16), q.astype(np.float16)


def run(oracle, bits, k, v, q, R=32, G=32, S=4):
    B, H, T, d = k.shape
    p = oracle.Params(bits=bits, group=G, residual=R, sinks=S, h_q=H, h_kv=H, head_dim=d, batch=B,
                      max_tokens=T)
    c = oracle.Cache(p)
    c.append(k, v)
    return c.decode_attn(q, threads=4), c


def mean_deviation(o, ref):
    o = o.reshape(-1, o.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    return float((np.linalg.norm(o - ref, axis=1) / np.linalg.norm(ref, axis=1)).mean())


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_int8_near_lossless(oracle_lib, seed):
    """The page's table: int8 ~0.5%, int4 ~7-10%, int2 ~41-51% on GPT-2.  The
    synthetic keys (N(0,1) queries against x10-30 outlier channels) give a
    sharper softmax than GPT-2, so absolute deviations run about twice the
    page's; the pin is int8 < 2% (mean over rows) and the page's ratios
    between widths, int4/int8 14-20x and int2/int4 4.1-7.3x (from 7-10% /
    0.5% and 41-51% / 7-10%), each held to within a factor 1.5 of the
    page's range on this synthetic stand-in."""
    k, v, q = outlier_stream(2, 4, 512, 64, seed=seed)
    ref = full_precision(q, k, v, 1)
    dev = {}
    for bits in (8, 4, 3, 2):
        o, _ = run(oracle_lib, bits, k, v, q)
        dev[bits] = mean_deviation(o, ref)
    assert dev[8] < 0.02
    # kvquant++ README: 3 bits sits between 2 (some loss) and 4 (near-lossless)
    assert dev[4] < dev[3] < dev[2]
    assert deviation(run(oracle_lib, 8, k, v, q)[0], ref) < 0.05
    assert 14.0 / 1.5 < dev[4] / dev[8] < 20.0 * 1.5
    assert 4.1 / 1.5 < dev[2] / dev[4] < 7.3 * 1.5


def _attend_dequant(q, K, V):
    d = q.shape[-1]
    s = K @ q / np.sqrt(d)
    w = np.exp(s - s.max())
    return (w[:, None] * V).sum(0) / w.sum()


def test_per_channel_keys_beat_per_token_keys(oracle_lib):
    """Same values path; only the key scale axis changes.  The per-token key
    variant uses the oracle's own quantizer over each token's channels."""
    B, H, T, d, bits = 1, 4, 512, 64, 4
    k, v, q = outlier_stream(B, H, T, d, seed=2)
    ref = full_precision(q, k, v, 1)
    out_pc, c = run(oracle_lib, bits, k, v, q)
    out_pt = np.zeros_like(out_pc)
    for h in range(H):
        K, V, vis = c.dequant_unit(0, h)
        Kpt = K.copy()
        for a in range(c.p.sinks, c.p.sinks + c.n_groups * c.p.group):
            codes, d16, m16 = oracle_lib.quantize(k[0, h, a], bits)
            dq = np.float64(np.uint16(d16).view(np.float16))
            mn = np.float64(np.uint16(m16).view(np.float16))
            Kpt[a] = mn + codes * dq
        out_pt[0, h] = _attend_dequant(q[0, h].astype(np.float64), Kpt, V)
    dev_pc, dev_pt = deviation(out_pc, ref), deviation(out_pt, ref)
    assert dev_pc < dev_pt
    assert dev_pt / dev_pc > 1.5   # the pages report 1.75-1.9x on real activations


def test_two_bits_needs_the_residual_window(oracle_lib):
    """Queries aligned with the most recent keys: quantizing the recent tokens
    too (no fp16 window) is worse than keeping them in fp16."""
    B, H, T, d, bits, R, G = 1, 4, 512, 64, 2, 128, 32
    k, v, q = outlier_stream(B, H, T, d, seed=3)
    # recency-weighted attention: the most recent 96 keys share a component
    # along q that lifts their scores by ~4 (in q·k/sqrt(d) units)
    qf = q.astype(np.float64)
    kf = k.astype(np.float64)
    for h in range(H):
        qhat = qf[0, h] / np.linalg.norm(qf[0, h])
        # adding beta * qhat raises q·k by beta*|q|; beta*|q|/sqrt(d) = 4
        kf[0, h, -96:] += (4.0 * np.sqrt(d) / np.linalg.norm(qf[0, h])) * qhat
    k = kf.astype(np.float16)
    ref = full_precision(q, k, v, 1)
    out_r, c = run(oracle_lib, bits, k, v, q, R=R, G=G)
    out_nr = np.zeros_like(out_r)
    for h in range(H):
        K, V, vis = c.dequant_unit(0, h)
        K2, V2 = K.copy(), V.copy()
        first = c.p.sinks + c.n_groups * G
        a = first
        while a < T:   # quantize the residual tokens as well, group by group
            hi = min(a + G, T)
            for ch in range(d):
                codes, d16, m16 = oracle_lib.quantize(k[0, h, a:hi, ch].copy(), bits)
                K2[a:hi, ch] = np.float64(np.uint16(m16).view(np.float16)) + codes * np.float64(np.uint16(d16).view(np.float16))
            for t in range(a, hi):
                codes, d16, m16 = oracle_lib.quantize(v[0, h, t], bits)
                V2[t] = np.float64(np.uint16(m16).view(np.float16)) + codes * np.float64(np.uint16(d16).view(np.float16))
            a = hi
        out_nr[0, h] = _attend_dequant(q[0, h].astype(np.float64), K2, V2)
    assert mean_deviation(out_r, ref) < 0.7 * mean_deviation(out_nr, ref)


def test_7b_fp16_sizing(oracle_lib):
    """512 KiB per token for a 7B model in fp16 (32 layers, 32 heads x 128):
    the cache's fp16 residual rows are exactly that size per token."""
    p = oracle_lib.Params(bits=4, group=32, residual=128, sinks=0, h_q=32, h_kv=32, head_dim=128,
                          batch=1, max_tokens=128)
    L = oracle_lib.layout(p)
    per_token_layer = 2 * (L["res_v"] - L["res_k"]) // p.residual * p.h_kv   # K + V rows, all heads
    assert per_token_layer * 32 == 2 * 32 * 4096 * 2 == 512 * 1024
    assert per_token_layer * 32 * 4096 == 2 * 1024 ** 3     # 2 GiB per 4096-token sequence


@pytest.mark.parametrize("bits,ratio_f16_lo,ratio_f16_hi", [(8, 1.8, 2.0), (4, 3.3, 4.0), (2, 5.5, 8.0)])
def test_bits_over_16_of_fp16(oracle_lib, bits, ratio_f16_lo, ratio_f16_hi):
    """Frozen-group bytes per token vs fp16 K+V: bits/16 plus the scale rows."""
    p = oracle_lib.Params(bits=bits, group=32, residual=32, sinks=0, h_q=1, h_kv=1, head_dim=128,
                          batch=1, max_tokens=32 * 100 + 32)
    L = oracle_lib.layout(p)
    per_token = L["block_bytes"] / p.group
    fp16 = 2 * 2 * p.head_dim
    assert ratio_f16_lo <= fp16 / per_token <= ratio_f16_hi
    if bits == 8:
        assert (2 * 4 * p.head_dim) / per_token > 3.0   # "> 3x vs f32"


def test_mistral_window_sizing(oracle_lib):
    """4096-token window, 8 kv heads x 128: ~33 MB in f32 -> ~8 MB with int8."""
    f32 = 2 * 8 * 128 * 4096 * 4
    assert 33e6 <= f32 <= 34e6
    p = oracle_lib.Params(bits=8, group=64, residual=64, sinks=0, h_q=32, h_kv=8, head_dim=128,
                          batch=1, max_tokens=0, window=4096)
    L = oracle_lib.layout(p)
    int8_window = 4096 / p.group * L["block_bytes"] * p.h_kv
    assert 7.5e6 <= int8_window <= 9.5e6
