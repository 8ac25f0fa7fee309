"""Pins the oracle's pre-RoPE keys (CPU only).

Source: KV-cache quantization guide (pigeon), "KVQuant adds": keys are
quantized before the rotary position embedding, which would otherwise mix
channel pairs and smear the per-channel structure.  Readings fixed here:
keys are stored (and quantized) as they arrive, before RoPE; attention
rotates each dequantized key at its own position a with the rotate-half
pairing (channel i with i + d/2) and angle a * base^(-2i/d); the query
arrives already rotated.

The pins do not restate the rotation: a closed form whose weights are
cos/sin of the position (keys and values chosen so that quantization is
exact), and a textbook comparison whose rotation is written as a complex
multiplication.
"""
import numpy as np
import pytest


def P(oracle, **kw):
    base = dict(bits=4, group=16, residual=32, sinks=2, h_q=2, h_kv=1, head_dim=64, batch=1,
                max_tokens=400, window=0, rope_base=10000.0)
    base.update(kw)
    return oracle.Params(**base)


def softmax_avg(s, v):
    w = np.exp(s - s.max())
    return (w[:, None] * v).sum(0) / w.sum()


def rotate_complex(K, base):
    """RoPE as complex multiplication: z_i = k_i + j k_{i+h} times e^{j a theta_i}."""
    T, d = K.shape
    h = d // 2
    theta = base ** (-np.arange(h) * 2.0 / d)
    z = (K[:, :h] + 1j * K[:, h:]) * np.exp(1j * np.arange(T)[:, None] * theta[None, :])
    return np.concatenate([z.real, z.imag], axis=1)


def test_bytes_do_not_depend_on_rope(oracle_lib):
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 1, 150, 64)).astype(np.float16)
    v = rng.standard_normal((1, 1, 150, 64)).astype(np.float16)
    arenas = []
    for base in (0.0, 10000.0, 500000.0):
        c = oracle_lib.Cache(P(oracle_lib, rope_base=base))
        assert c.append(k, v) == 0
        arenas.append(c.arena())
    assert np.array_equal(arenas[0], arenas[1]) and np.array_equal(arenas[0], arenas[2])
    assert oracle_lib.validate(P(oracle_lib, rope_base=1.0)) != 0
    assert oracle_lib.validate(P(oracle_lib, rope_base=-5.0)) != 0


@pytest.mark.parametrize("i,d", [(0, 64), (0, 128), (1, 64), (5, 128)])
def test_closed_form_through_frozen_groups(oracle_lib, i, d):
    """Keys kappa e_i at every position (constant per channel: exact codes),
    values equal to the position (constant per token: exact), query
    alpha e_i + beta e_{i+d/2}: the score at position a is
    (alpha cos(a theta_i) + beta sin(a theta_i)) kappa / sqrt(d), theta_0 = 1,
    and the output is the softmax average of the positions."""
    T, kappa, alpha, beta = 300, 3.0, 1.5, -2.0
    p = P(oracle_lib, head_dim=d)
    h = d // 2
    K = np.zeros((T, d))
    K[:, i] = kappa
    V = np.repeat(np.arange(T, dtype=np.float64)[:, None], d, axis=1)
    c = oracle_lib.Cache(p)
    assert c.append(K[None, None].astype(np.float16), V[None, None].astype(np.float16)) == 0
    assert c.n_groups > 5
    q = np.zeros((1, 2, d))
    q[0, :, i], q[0, :, i + h] = alpha, beta
    out = c.decode_attn(q.astype(np.float16))
    theta = 1.0 if i == 0 else 10000.0 ** (-2.0 * i / d)
    a = np.arange(T)
    s = (alpha * np.cos(a * theta) + beta * np.sin(a * theta)) * kappa / np.sqrt(d)
    exp = softmax_avg(s, V)
    np.testing.assert_allclose(out[0, 0], exp, rtol=0, atol=1e-9)
    np.testing.assert_allclose(out[0, 1], exp, rtol=0, atol=1e-9)


@pytest.mark.parametrize("base,window", [(10000.0, 0), (500000.0, 0), (10000.0, 48)])
def test_textbook_while_nothing_is_quantized(oracle_lib, base, window):
    """T <= S + R: every key is exact, so the oracle's attention equals the
    textbook softmax over the raw keys rotated by the complex formula."""
    rng = np.random.default_rng(3)
    p = P(oracle_lib, rope_base=base, window=window, max_tokens=0 if window else 400)
    T = p.sinks + p.residual
    k = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0 and c.n_groups == 0
    q = rng.standard_normal((1, 2, 64)).astype(np.float16)
    out = c.decode_attn(q)
    Kr = rotate_complex(k[0, 0].astype(np.float64), base)
    for hq in range(2):
        s = Kr @ q[0, hq].astype(np.float64) / 8.0
        np.testing.assert_allclose(out[0, hq], softmax_avg(s, v[0, 0].astype(np.float64)), rtol=0, atol=1e-12)


def test_causal_queries_rotate_keys_at_their_positions(oracle_lib):
    """The multi-query attention rotates keys the same way: each query of a
    chunk against the complex-rotated raw keys at or before its position."""
    rng = np.random.default_rng(4)
    p = P(oracle_lib)
    T, M = 30, 6
    k = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, 64)).astype(np.float16)
    c = oracle_lib.Cache(p)
    assert c.append(k, v) == 0
    q = rng.standard_normal((1, M, 2, 64)).astype(np.float16)
    out = c.prefill_attn(q)
    Kr = rotate_complex(k[0, 0].astype(np.float64), p.rope_base)
    for j in range(M):
        P_ = T - M + j
        s = Kr[:P_ + 1] @ q[0, j, 0].astype(np.float64) / 8.0
        np.testing.assert_allclose(out[0, j, 0], softmax_avg(s, v[0, 0, :P_ + 1].astype(np.float64)),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pre_rope_quantization_keeps_outlier_channels(oracle_lib, bits):
    """Keys with fixed large-magnitude channels (an offset of 20 on two
    channels): quantizing them before RoPE (this mode) gives a smaller
    attention error than quantizing the rotated keys, in which each such
    channel turns with the position and spreads over itself and its partner
    (a range of +-20 in both), against fp64 attention over the exact rotated
    keys."""
    rng = np.random.default_rng(11)
    T, d = 16 * 20 + 32, 64
    K = rng.standard_normal((T, d))
    K[:, [3, 17]] += 20
    V = rng.standard_normal((T, d))
    k = K.astype(np.float16)
    v = V.astype(np.float16)
    Kr = rotate_complex(k.astype(np.float64), 10000.0)
    q = rng.standard_normal((1, 2, d)).astype(np.float16)
    exact = np.array([softmax_avg(Kr @ q[0, hq].astype(np.float64) / 8.0, v.astype(np.float64))
                      for hq in range(2)])
    pre = oracle_lib.Cache(P(oracle_lib, bits=bits, sinks=0))
    assert pre.append(k[None, None], v[None, None]) == 0
    post = oracle_lib.Cache(P(oracle_lib, bits=bits, sinks=0, rope_base=0.0))
    assert post.append(Kr.astype(np.float16)[None, None], v[None, None]) == 0
    e_pre = np.abs(pre.decode_attn(q)[0] - exact).max()
    e_post = np.abs(post.decode_attn(q)[0] - exact).max()
    assert e_pre < e_post, (e_pre, e_post)
