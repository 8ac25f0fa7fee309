"""Pins the oracle's causal multi-token attention (CPU only).

Sources: kvquant++ README, long-document example (prefill_chunk_size: the
context is processed in chunks, each chunk's attention step covers the chunk
while the whole context accumulates in the cache); KV-cache quantization guide
(pigeon), "How it works", step 5 (softmax(q Kᵀ / sqrt(d)) V over dequantized
values); tract #2329 "Relationship to other PRs" (sliding window).

Reading pinned here: after a chunk of M tokens is appended, query j of the
chunk sits at position P = T - M + j and attends to the tokens the cache
still holds with position <= P; with a window W, to the sinks and to the W
tokens ending at P.
"""
import ctypes

import numpy as np
import pytest


def P(oracle, **kw):
    base = dict(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=2, head_dim=64, batch=2,
                max_tokens=400, window=0)
    base.update(kw)
    return oracle.Params(**base)


def stream(p, T, seed):
    rng = np.random.default_rng(seed)
    shape = (p.batch, p.h_kv, T, p.head_dim)
    return rng.standard_normal(shape).astype(np.float16), rng.standard_normal(shape).astype(np.float16)


def queries(p, M, seed):
    rng = np.random.default_rng(1000 + seed)
    return rng.standard_normal((p.batch, M, p.h_q, p.head_dim)).astype(np.float16)


def textbook(q, K, V, visible):
    d = q.shape[-1]
    s = np.where(visible, (K @ q) / np.sqrt(d), -np.inf)
    w = np.exp(s - s.max())
    return (w[:, None] * V).sum(0) / w.sum()


@pytest.mark.parametrize("T,M", [(1, 1), (5, 5), (20, 7), (36, 36), (36, 1)])
def test_unquantized_prefix_is_textbook_causal_attention(oracle_lib, T, M):
    """While T <= S + R nothing is quantized: query j is plain softmax
    attention over the raw fp16 inputs at positions 0..T-M+j."""
    p = P(oracle_lib)
    k, v = stream(p, T, seed=T)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups == 0
    q = queries(p, M, seed=T)
    out = c.prefill_attn(q)
    rep = p.h_q // p.h_kv
    pos = np.arange(T)
    for b in range(p.batch):
        for j in range(M):
            for hq in range(p.h_q):
                ref = textbook(q[b, j, hq].astype(np.float64), k[b, hq // rep].astype(np.float64),
                               v[b, hq // rep].astype(np.float64), pos <= T - M + j)
                assert np.allclose(out[b, j, hq], ref, rtol=1e-12, atol=1e-12)


def resident(p, T, n_groups):
    """Positions the cache still holds: sinks, ring, and the last n_slots
    frozen groups (every group without a window)."""
    pos = np.arange(T)
    if p.window == 0:
        return np.ones(T, bool)
    n_slots = -(-p.window // p.group) + 1
    first = max(0, n_groups - n_slots)
    return (pos < p.sinks) | (pos >= p.sinks + first * p.group)


@pytest.mark.parametrize("window,T,M", [(0, 150, 40), (0, 150, 150), (48, 200, 33), (48, 200, 120),
                                        (64, 333, 200)])
def test_zero_keys_average_the_visible_positions(oracle_lib, window, T, M):
    """K = 0 makes every score equal, so query j returns the mean of the
    visible values.  V rows are constant across channels (Δ = 0, the value is
    its own fp16 min) with value a + 256 u for token a of unit u, exact in
    fp16: the output is the mean visible position plus 256 u, a closed form
    that checks the causal bound, the window bound, sinks, the ring, frozen
    groups, evicted slots and the GQA head-to-unit map."""
    p = P(oracle_lib, window=window, max_tokens=400, residual=32, group=16, sinks=3)
    c = oracle_lib.Cache(p)
    k = np.zeros((p.batch, p.h_kv, T, p.head_dim), np.float16)
    v = np.zeros_like(k)
    for b in range(p.batch):
        for h in range(p.h_kv):
            v[b, h] = (np.arange(T) + 256 * (b * p.h_kv + h))[:, None]
    assert c.append(k, v) == 0
    q = queries(p, M, seed=M)
    out = c.prefill_attn(q)
    res = resident(p, T, c.n_groups)
    pos = np.arange(T)
    rep = p.h_q // p.h_kv
    for j in range(M):
        Pj = T - M + j
        vis = res & (pos <= Pj)
        if window:
            vis &= (pos < p.sinks) | (pos >= Pj + 1 - window)
        mean = pos[vis].mean()
        for b in range(p.batch):
            for hq in range(p.h_q):
                exp = mean + 256 * (b * p.h_kv + hq // rep)
                assert np.allclose(out[b, j, hq], exp, rtol=0, atol=1e-9), (j, b, hq)


@pytest.mark.parametrize("window", [0, 48])
def test_newest_query_is_the_decode_query(oracle_lib, window):
    """The last query of a chunk sits at T - 1: the same result as decode."""
    p = P(oracle_lib, window=window, bits=2)
    k, v = stream(p, 180, seed=3)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    q = queries(p, 9, seed=3)
    out = c.prefill_attn(q)
    dec = c.decode_attn(q[:, -1])
    assert np.array_equal(out[:, -1], dec)
    one = c.prefill_attn(q[:, -1:])
    assert np.array_equal(one[:, 0], dec)


def test_future_tokens_do_not_reach_earlier_queries(oracle_lib):
    """Two streams that differ only in their last 5 tokens (all in the ring):
    queries before them return identical results, later ones differ."""
    p = P(oracle_lib, bits=4)
    k, v = stream(p, 150, seed=9)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, -5:] = (k2[:, :, -5:].astype(np.float32) * -1.5).astype(np.float16)
    v2[:, :, -5:] = (v2[:, :, -5:].astype(np.float32) + 2.0).astype(np.float16)
    c1, c2 = oracle_lib.Cache(p), oracle_lib.Cache(p)
    assert c1.append(k, v) == 0 and c2.append(k2, v2) == 0
    assert c1.n_res >= 5
    q = queries(p, 12, seed=9)
    o1, o2 = c1.prefill_attn(q), c2.prefill_attn(q)
    assert np.array_equal(o1[:, :7], o2[:, :7])
    assert not np.allclose(o1[:, 7:], o2[:, 7:])


@pytest.mark.parametrize("bits", [2, 8])
def test_matches_bruteforce_on_dequantized(oracle_lib, bits):
    """Each query row equals softmax attention over the dequantized unit with
    the causal mask (no window: every token is resident)."""
    p = P(oracle_lib, bits=bits)
    k, v = stream(p, 211, seed=bits)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups > 0
    M = 50
    q = queries(p, M, seed=bits)
    out = c.prefill_attn(q)
    rep = p.h_q // p.h_kv
    pos = np.arange(211)
    for b in range(p.batch):
        for h in range(p.h_kv):
            K, V, _ = c.dequant_unit(b, h)
            for j in range(0, M, 7):
                for r in range(rep):
                    ref = textbook(q[b, j, h * rep + r].astype(np.float64), K, V, pos <= 211 - M + j)
                    assert np.allclose(out[b, j, h * rep + r], ref, rtol=1e-12, atol=1e-12)


def test_threads_do_not_change_result(oracle_lib):
    p = P(oracle_lib, h_q=8, h_kv=4)
    k, v = stream(p, 120, seed=4)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    q = queries(p, 16, seed=4)
    assert np.array_equal(c.prefill_attn(q, threads=1), c.prefill_attn(q, threads=5))


def test_query_count_outside_one_to_T_is_invalid(oracle_lib):
    p = P(oracle_lib)
    k, v = stream(p, 10, seed=1)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    L = oracle_lib.lib()
    q = np.zeros((p.batch, 11, p.h_q, p.head_dim), np.uint16)
    out = np.zeros(q.shape, np.float64)
    qp = q.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))
    op = out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    assert L.ko_prefill_attn(c._h, qp, 0, op, 1) == 1
    assert L.ko_prefill_attn(c._h, qp, 11, op, 1) == 1
    assert L.ko_prefill_attn(c._h, qp, 10, op, 1) == 0
