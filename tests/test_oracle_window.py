"""Pins the oracle's two readings of a sliding window composed with sinks
(CPU only).

tract #2329, "Relationship to other PRs", composes a bounded sliding-window
cache with the quantized storage but gives no rule for the sink tokens of
tract #2458.  The oracle keeps both readings: window_mode 0 (the CUDA
library's) keeps the sinks visible beside the most recent W tokens;
window_mode 1 is a pure window, in which the sinks expire like any other
token.  These pins fix both readings against closed forms and textbook
attention, so that neither reading can drift into the other.
"""
import numpy as np
import pytest


def params(oracle, **kw):
    base = dict(bits=4, group=16, residual=32, sinks=4, h_q=2, h_kv=1, head_dim=64, batch=1,
                max_tokens=0, window=48)
    base.update(kw)
    return oracle.Params(**base)


def position_stream(T, d):
    """Keys all zero and each token's values equal to its position: exact
    under quantization (every key channel and value token is constant, so
    Δ = 0 and min is the value itself; positions below 2048 are exact fp16),
    and the attention is the mean position of the visible tokens."""
    k = np.zeros((1, 1, T, d), np.float16)
    v = np.broadcast_to(np.arange(T, dtype=np.float16)[None, None, :, None], (1, 1, T, d)).copy()
    return k, v


def visible_positions(T, P, S, W, mode):
    lo = P + 1 - W
    return [a for a in range(T) if a <= P and (a >= lo or (mode == 0 and a < S))]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T", [1, 4, 30, 52, 53, 100, 161, 400, 777])
def test_decode_mean_position_closed_form(oracle_lib, mode, T):
    """Decode at position T - 1 sees [T - W, T - 1], plus the sinks in mode 0."""
    p = params(oracle_lib, window_mode=mode)
    c = oracle_lib.Cache(p)
    k, v = position_stream(T, p.head_dim)
    assert c.append(k, v) == 0
    q = np.ones((1, 2, p.head_dim), np.float16)
    out = c.decode_attn(q)
    expect = np.mean(visible_positions(T, T - 1, p.sinks, p.window, mode))
    assert np.allclose(out, expect, rtol=0, atol=1e-9), (out[0, 0, 0], expect)


@pytest.mark.parametrize("mode", [0, 1])
def test_causal_queries_mean_position_closed_form(oracle_lib, mode):
    """Causal queries of a chunk: query j at P = T - M + j sees [P + 1 - W, P]
    (among the tokens the cache still holds), plus the sinks in mode 0."""
    p = params(oracle_lib, window_mode=mode)
    T, M = 300, 40
    c = oracle_lib.Cache(p)
    k, v = position_stream(T, p.head_dim)
    assert c.append(k, v) == 0
    q = np.ones((1, M, 2, p.head_dim), np.float16)
    out = c.prefill_attn(q)
    for j in range(M):
        P = T - M + j
        expect = np.mean(visible_positions(T, P, p.sinks, p.window, mode))
        assert np.allclose(out[0, j], expect, rtol=0, atol=1e-9), (j, out[0, j, 0, 0], expect)


def textbook(q, K, V):
    s = (K @ q) / np.sqrt(q.shape[-1])
    w = np.exp(s - s.max())
    return (w[:, None] * V).sum(0) / w.sum()


@pytest.mark.parametrize("mode", [0, 1])
def test_unquantized_window_is_textbook_attention(oracle_lib, mode):
    """S = 4, R = W = 32, T = S + R = 36: nothing is quantized and the window
    is [4, 35], so a pure window drops exactly the four sinks."""
    p = params(oracle_lib, window_mode=mode, window=32, residual=32)
    T = 36
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    q = rng.standard_normal((1, 2, 64)).astype(np.float16)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    assert c.n_groups == 0
    out = c.decode_attn(q)
    first = p.sinks if mode == 1 else 0
    for h in range(2):
        ref = textbook(q[0, h].astype(np.float64), k[0, 0, first:].astype(np.float64),
                       v[0, 0, first:].astype(np.float64))
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-12)


def test_readings_agree_while_the_window_holds_the_sinks(oracle_lib):
    """Until T exceeds W every sink lies in the window: both readings give the
    same output, bit for bit."""
    rng = np.random.default_rng(9)
    T = 48
    k = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    q = rng.standard_normal((1, 2, 64)).astype(np.float16)
    outs = []
    for mode in (0, 1):
        c = oracle_lib.Cache(params(oracle_lib, window_mode=mode))
        assert c.append(k, v) == 0
        outs.append(c.decode_attn(q))
    assert np.array_equal(outs[0], outs[1])
    # one token later the first sink leaves a pure window: the outputs differ
    outs = []
    k2 = rng.standard_normal((1, 1, 1, 64)).astype(np.float16)
    for mode in (0, 1):
        c = oracle_lib.Cache(params(oracle_lib, window_mode=mode))
        assert c.append(k, v) == 0 and c.append(k2, k2) == 0
        outs.append(c.decode_attn(q))
    assert not np.array_equal(outs[0], outs[1])


def test_window_mode_is_validated(oracle_lib):
    assert oracle_lib.validate(params(oracle_lib, window_mode=2)) != 0
    assert oracle_lib.validate(params(oracle_lib, window_mode=1)) == 0
