"""Dense-and-sparse outliers through the C ABI against the oracle.

Source: KV-cache quantization guide (pigeon), "KVQuant adds": a small share
of the values kept in fp16 in a sparse table beside the codes.  The CUDA
flush must write the same bytes as the oracle (selection, tie order, dense
ranges without the outliers, tables), and the decode must add each table
entry's difference from its dense dequantization to the scores (keys) and to
the outputs (values): within 2e-3 of the oracle's fp64 attention over the
exactly restored values.  The streams carry 1 % spikes of x30 on top of the
fixed outlier channels, so that the corrections are large.
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


def spiky_stream(cfg, T, seed):
    k, v = random_stream(cfg, T, seed)
    g = torch.Generator().manual_seed(seed + 5)
    for x in (k, v):
        m = torch.rand(x.shape, generator=g) < 0.01
        x[m] = (x[m].float() * 30).half()
    return k, v


CASES = [
    # 4 bits, d 128, GQA rep 4, 1 %
    dict(bits=4, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=700,
         outlier_permille=10),
    # 2 bits, d 64, MHA, 2 %
    dict(bits=2, group=32, residual=32, sinks=2, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=700,
         outlier_permille=20),
    # 3 bits (bit stream), d 128, GQA rep 8, 1 %, no sinks
    dict(bits=3, group=32, residual=64, sinks=0, h_q=16, h_kv=2, head_dim=128, batch=2, max_tokens=700,
         outlier_permille=10),
    # 4 bits, G 64, sliding window (slot ring wraps), GQA rep 3, 0.5 %
    dict(bits=4, group=64, residual=64, sinks=2, h_q=6, h_kv=2, head_dim=128, batch=2, max_tokens=0, window=160,
         outlier_permille=5),
    # 2 bits at the largest share, d 128, many entries per 32-token chunk
    dict(bits=2, group=32, residual=32, sinks=1, h_q=4, h_kv=1, head_dim=128, batch=3, max_tokens=700,
         outlier_permille=50),
]


@pytest.mark.parametrize("shape", CASES)
def test_outlier_cache_bytes_and_decode(shape):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    assert p.gpu.layout()["n_outliers"] == p.ref.layout["n_outliers"] > 0
    k, v = spiky_stream(cfg, 700, seed=3)
    t = 0
    for i, n in enumerate([1, 40, 100, 7, 300]):
        p.append(k[:, :, t:t + n].contiguous(), v[:, :, t:t + n].contiguous())
        t += n
        err = p.decode_err(random_q(cfg, i))
        assert err <= TOL, (i, err)
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


def test_outliers_change_the_result():
    """The same stream with and without the tables: the attention differs by
    far more than the tolerance, so the corrections are not a no-op."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    base = dict(bits=2, group=32, residual=32, sinks=0, h_q=4, h_kv=4, head_dim=128, batch=1, max_tokens=300)
    k, v = spiky_stream(KiviConfig(**base), 300, seed=8)
    outs = []
    for pm in (0, 10):
        c = KiviCache(KiviConfig(**base, outlier_permille=pm))
        c.append(k.cuda(), v.cuda())
        outs.append(c.decode(random_q(KiviConfig(**base), 1).cuda()).float().cpu().numpy())
    assert row_rel_err(outs[1], outs[0]) > 20 * TOL


def test_ragged_lengths_with_outliers():
    """Sequences of different lengths: the ragged decode with corrections."""
    import oracle
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=32, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=3, max_tokens=400,
                     outlier_permille=10)
    gpu = KiviCache(cfg)
    refs = [oracle.Cache(oparams(cfg, batch=1)) for _ in range(3)]
    streams = [spiky_stream(KiviConfig(**{**cfg.__dict__, "batch": 1}), 400, seed=40 + b) for b in range(3)]
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


@pytest.mark.parametrize("shape", [
    # 4 bits, d 128, GQA rep 4 (a head pass of four rows spans one query token)
    dict(bits=4, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=700,
         outlier_permille=10),
    # 3 bits at head dim 64 (bit stream), MHA (a pass of four rows spans four query tokens), 2 %
    dict(bits=3, group=32, residual=32, sinks=2, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=700,
         outlier_permille=20),
    # 2 bits, d 128, GQA rep 3, a wrapping window
    dict(bits=2, group=64, residual=64, sinks=1, h_q=6, h_kv=2, head_dim=128, batch=1, max_tokens=0, window=160,
         outlier_permille=5),
])
def test_prefill_with_outliers(shape):
    """Chunked prefill (the causal attention of a chunk's queries) over a cache
    with outlier tables: every row within 2e-3 of the oracle's causal
    attention, chunks shorter and longer than the ring (so some chunk tokens
    are read from codes and their tables), bytes identical after each chunk."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    k, v = spiky_stream(cfg, 700, seed=21)
    t = 0
    g = torch.Generator().manual_seed(4)
    for m in (130, 9, 100, 1, 70):
        p.append(k[:, :, t:t + m].contiguous(), v[:, :, t:t + m].contiguous())
        t += m
        assert p.bytes_equal()
        q = torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=g).half()
        out = p.gpu.prefill(q.cuda()).float().cpu().numpy()
        exp = p.ref.prefill_attn(q.numpy(), threads=8)
        assert row_rel_err(out, exp) <= TOL, m
    assert p.gpu.read_error() == 0


def test_outlier_tables_at_head_dim_64_three_bits():
    """3 bits (bit stream) at head dim 64 with 1 % outlier tables: bytes and
    decode against the oracle, through fused steps across group freezes."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=3, group=64, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=64, batch=2, max_tokens=700,
                     outlier_permille=10)
    p = Pair(cfg)
    k, v = spiky_stream(cfg, 600, seed=12)
    p.append(k[:, :, :500].contiguous(), v[:, :, :500].contiguous())
    assert p.bytes_equal()
    assert p.decode_err(random_q(cfg, 2)) <= TOL
    for i in range(100):
        kk, vv = k[:, :, 500 + i:501 + i].contiguous(), v[:, :, 500 + i:501 + i].contiguous()
        q = random_q(cfg, 200 + i)
        out = p.gpu.append_decode(kk.cuda(), vv.cuda(), q.cuda()).float().cpu().numpy()
        assert p.ref.append(kk.numpy(), vv.numpy()) == 0
        assert row_rel_err(out, p.ref.decode_attn(q.numpy(), threads=8)) <= TOL, i
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0
