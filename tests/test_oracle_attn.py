"""Pins the oracle's fp64 decode attention (CPU only).

Sources: KV-cache quantization guide (pigeon), "How it works", step 5
(softmax(q Kᵀ / sqrt(d)) V over the dequantized values); tract #2329 "What's
in the PR" (grouped-query heads; an output shaped like the query); tract #2329
"Relationship to other PRs" (sliding-window cache composed with quantization).
"""
import numpy as np
import pytest


def P(oracle, **kw):
    base = dict(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=2, head_dim=64, batch=2,
                max_tokens=400, window=0)
    base.update(kw)
    return oracle.Params(**base)


def make(oracle, p, T, seed=0):
    rng = np.random.default_rng(seed)
    shape = (p.batch, p.h_kv, T, p.head_dim)
    k = rng.standard_normal(shape).astype(np.float16)
    v = rng.standard_normal(shape).astype(np.float16)
    q = rng.standard_normal((p.batch, p.h_q, p.head_dim)).astype(np.float16)
    c = oracle.Cache(p)
    if T:
        assert c.append(k, v) == 0
    return c, k, v, q


def textbook(q, K, V, visible=None):
    """softmax(q Kᵀ / sqrt(d)) V in fp64 for one query row."""
    d = q.shape[-1]
    s = (K @ q) / np.sqrt(d)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    w = np.exp(s - s.max())
    return (w[:, None] * V).sum(0) / w.sum()


@pytest.mark.parametrize("T", [1, 3, 4, 20, 36])
def test_unquantized_prefix_is_textbook_attention(oracle_lib, T):
    """While T <= S + R nothing is quantized: the result is plain softmax
    attention over the fp16 inputs (sinks are exact fp32 widenings)."""
    p = P(oracle_lib)
    c, k, v, q = make(oracle_lib, p, T, seed=T)
    assert c.n_groups == 0
    out = c.decode_attn(q)
    rep = p.h_q // p.h_kv
    for b in range(p.batch):
        for hq in range(p.h_q):
            ref = textbook(q[b, hq].astype(np.float64), k[b, hq // rep].astype(np.float64),
                           v[b, hq // rep].astype(np.float64))
            assert np.allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("window", [0, 48])
@pytest.mark.parametrize("T", [37, 100, 257])
def test_matches_bruteforce_on_dequantized(oracle_lib, bits, window, T):
    p = P(oracle_lib, bits=bits, window=window, max_tokens=0 if window else 400)
    c, k, v, q = make(oracle_lib, p, T, seed=bits * 31 + T)
    out = c.decode_attn(q, threads=3)
    rep = p.h_q // p.h_kv
    for b in range(p.batch):
        for h in range(p.h_kv):
            K, V, vis = c.dequant_unit(b, h)
            exp_vis = np.zeros(T, bool)
            exp_vis[:min(T, p.sinks)] = True
            exp_vis[max(0, T - window) if window else 0:] = True
            assert np.array_equal(vis, exp_vis)
            for r in range(rep):
                hq = h * rep + r
                ref = textbook(q[b, hq].astype(np.float64), K, V, vis)
                assert np.allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_gqa_uses_contiguous_groups(oracle_lib):
    """Query head hq reads kv head floor(hq / (H_q / H_kv)).  The kv heads are
    made very different so that any other mapping changes the output."""
    p = P(oracle_lib, h_q=6, h_kv=3, batch=1)
    T = 30
    rng = np.random.default_rng(3)
    k = rng.standard_normal((1, 3, T, 64)).astype(np.float16)
    v = np.zeros((1, 3, T, 64), np.float16)
    for h in range(3):
        v[0, h] = 10 * (h + 1)   # each kv head's values are a distinct constant
    q = rng.standard_normal((1, 6, 64)).astype(np.float16)
    c = oracle_lib.Cache(p)
    c.append(k, v)
    out = c.decode_attn(q)
    for hq in range(6):
        assert np.allclose(out[0, hq], 10 * (hq // 2 + 1))


def test_threads_do_not_change_result(oracle_lib):
    p = P(oracle_lib, batch=3, h_kv=4, h_q=8)
    c, k, v, q = make(oracle_lib, p, 200, seed=11)
    a = c.decode_attn(q, threads=1)
    b = c.decode_attn(q, threads=7)
    assert np.array_equal(a, b)


def test_output_is_convex_combination(oracle_lib):
    # every output channel lies within [min, max] of the visible V̂ values
    p = P(oracle_lib, bits=2)
    c, k, v, q = make(oracle_lib, p, 300, seed=12)
    out = c.decode_attn(q)
    rep = p.h_q // p.h_kv
    for b in range(p.batch):
        for hq in range(p.h_q):
            K, V, vis = c.dequant_unit(b, hq // rep)
            assert np.all(out[b, hq] <= V[vis].max(0) + 1e-12)
            assert np.all(out[b, hq] >= V[vis].min(0) - 1e-12)


def test_decode_bytes_closed_form(oracle_lib):
    # mha7b-shaped unit count at T=4096: 124 groups, 124 residual, 4 sinks
    p = oracle_lib.Params(bits=4, group=32, residual=128, sinks=4, h_q=1, h_kv=1, head_dim=128,
                          batch=1, max_tokens=4096)
    c = oracle_lib.Cache(p)
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 1, 4096, 128)).astype(np.float16)
    c.append(k, k)
    tq = 124 * 32
    expect = 2 * tq * 128 * 4 // 8 + 4 * 128 * 124 + 4 * tq + 4 * 128 * 124 + 8 * 128 * 4 + 4 * 128
    assert c.decode_bytes() == expect == 654848 + 512
