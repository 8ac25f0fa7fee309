"""Pre-RoPE keys through the C ABI against the oracle.

Source: KV-cache quantization guide (pigeon), "KVQuant adds": keys are
quantized before the rotary position embedding.  The cache stores the keys
as they arrive (the bytes are those of any cache: the oracle's, byte for
byte), and the decode rotates every dequantized key at its own position
(rotate-half pairs (i, i + d/2), angle position * base^(-2i/d)) before its
dot product with the rotated query: within 2e-3 of the oracle's fp64
attention.  Cases span every code width, head dims 64 and 128, GQA, sinks,
windows whose slot ring wraps, chunked appends, fused steps across group
freezes and ragged lengths.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, Pair, oparams, random_q, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = [
    dict(bits=4, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=700),
    dict(bits=2, group=64, residual=64, sinks=0, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=700),
    dict(bits=3, group=32, residual=32, sinks=2, h_q=16, h_kv=2, head_dim=128, batch=2, max_tokens=700),
    dict(bits=8, group=64, residual=64, sinks=4, h_q=6, h_kv=2, head_dim=128, batch=2, max_tokens=0, window=160),
    dict(bits=5, group=32, residual=32, sinks=1, h_q=2, h_kv=1, head_dim=64, batch=3, max_tokens=700),
    dict(bits=1, group=32, residual=64, sinks=3, h_q=4, h_kv=1, head_dim=128, batch=1, max_tokens=700,
         rope_base=500000.0),
]


@pytest.mark.parametrize("shape", CASES)
def test_pre_rope_cache_bytes_and_decode(shape):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**{"rope_base": 10000.0, **shape})
    p = Pair(cfg)
    k, v = random_stream(cfg, 700, seed=21)
    t = 0
    for i, n in enumerate([1, 2, 40, 100, 7, 300]):
        p.append(k[:, :, t:t + n].contiguous(), v[:, :, t:t + n].contiguous())
        t += n
        err = p.decode_err(random_q(cfg, i))
        assert err <= TOL, (i, t, err)
    assert p.bytes_equal()
    for i in range(70):   # fused steps, crossing group freezes
        kk = k[:, :, t:t + 1].contiguous()
        vv = v[:, :, t:t + 1].contiguous()
        q = random_q(cfg, 100 + i)
        out = p.gpu.append_decode(kk.cuda(), vv.cuda(), q.cuda()).float().cpu().numpy()
        assert p.ref.append(kk.numpy(), vv.numpy()) == 0
        t += 1
        assert row_rel_err(out, p.ref.decode_attn(q.numpy(), threads=8)) <= TOL, i
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0


def test_rotation_changes_the_result():
    """The same stream with and without RoPE at attention differs by far more
    than the tolerance: the rotation is applied."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    base = dict(bits=4, group=32, residual=32, sinks=0, h_q=4, h_kv=4, head_dim=128, batch=1, max_tokens=300)
    k, v = random_stream(KiviConfig(**base), 300, seed=8)
    outs = []
    for rb in (0.0, 10000.0):
        c = KiviCache(KiviConfig(**base, rope_base=rb))
        c.append(k.cuda(), v.cuda())
        outs.append(c.decode(random_q(KiviConfig(**base), 1).cuda()).float().cpu().numpy())
    assert row_rel_err(outs[1], outs[0]) > 20 * TOL


def test_ragged_lengths_with_pre_rope_keys():
    import oracle
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=32, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=3, max_tokens=400,
                     rope_base=10000.0)
    gpu = KiviCache(cfg)
    refs = [oracle.Cache(oparams(cfg, batch=1)) for _ in range(3)]
    streams = [random_stream(KiviConfig(**{**cfg.__dict__, "batch": 1}), 400, seed=60 + b) for b in range(3)]
    pos = [0, 0, 0]
    for counts in ([100, 37, 0], [64, 64, 130], [1, 90, 5]):
        n_max = max(counts)
        k = torch.zeros((3, 2, n_max, 128), dtype=torch.float16)
        v = torch.zeros_like(k)
        for b, n in enumerate(counts):
            ks, vs = streams[b]
            k[b, :, :n] = ks[0, :, pos[b]:pos[b] + n]
            v[b, :, :n] = vs[0, :, pos[b]:pos[b] + n]
            if n:
                assert refs[b].append(k[b:b + 1, :, :n].numpy(), v[b:b + 1, :, :n].numpy()) == 0
            pos[b] += n
        gpu.append_ragged(k.cuda(), v.cuda(), counts)
        q = random_q(cfg, sum(counts))
        out = gpu.decode(q.cuda()).float().cpu().numpy()
        for b in range(3):
            exp = refs[b].decode_attn(q[b:b + 1].numpy(), threads=8)
            assert row_rel_err(out[b:b + 1], exp) <= TOL, (counts, b)
    region = gpu.cache_region().cpu().numpy()
    per_seq = gpu.layout()["unit_bytes"] * cfg.h_kv
    for b in range(3):
        assert np.array_equal(region[b * per_seq:(b + 1) * per_seq], refs[b].arena()), b
    assert gpu.read_error() == 0


@pytest.mark.parametrize("shape", [CASES[0], CASES[1], CASES[3], CASES[4]])
def test_prefill_with_pre_rope_keys(shape):
    """Chunked prefill (each query token attends causally over the cache)
    over pre-RoPE keys: every row within 2e-3 of the oracle's causal
    attention, chunks shorter and longer than the ring, bytes identical."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**{"rope_base": 10000.0, **shape})
    p = Pair(cfg)
    k, v = random_stream(cfg, 700, seed=23)
    g = torch.Generator().manual_seed(11)
    t = 0
    for m in (150, 9, 100, 1, 64):
        p.append(k[:, :, t:t + m].contiguous(), v[:, :, t:t + m].contiguous())
        t += m
        q = torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=g).half()
        out = p.gpu.prefill(q.cuda()).float().cpu().numpy()
        assert row_rel_err(out, p.ref.prefill_attn(q.numpy(), threads=8)) <= TOL, m
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0


def test_long_positions_with_pre_rope_keys():
    """Positions past 2^17 (a 32-token window over a stream of 140000 tokens,
    base angles reduced mod 2π from large multiples): decode within 2e-3."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=32, sinks=2, h_q=4, h_kv=1, head_dim=128, batch=1, max_tokens=0,
                     window=64, rope_base=10000.0)
    p = Pair(cfg)
    k, v = random_stream(cfg, 4000, seed=5)
    # 35 passes over the same 4000 tokens: positions reach 140000
    for rnd in range(35):
        p.append(k, v)
    assert p.gpu.tokens == 140000
    assert p.bytes_equal()
    assert p.decode_err(random_q(cfg, 9)) <= TOL
