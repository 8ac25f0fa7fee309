"""Code widths outside {2, 4, 8} (tract #2329: configurable 1..16 bits; the
kvquant++ README recommends 3) against the oracle, through the C ABI.

These widths pack as a plain bit stream and decode on the tensor cores at
head dims 64 and 128 (two codes unpacked into one fp16x2 operand register).
Bytes must equal the oracle's; decode, fused steps and multi-query attention
within 2e-3.  Streams cross sinks, the filling ring, group freezes, a wrapping
window and ragged lengths.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, Pair, random_q, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = [
    dict(bits=3, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=600),
    dict(bits=1, group=32, residual=32, sinks=1, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=600),
    dict(bits=5, group=64, residual=64, sinks=0, h_q=16, h_kv=2, head_dim=128, batch=1, max_tokens=600),
    dict(bits=6, group=32, residual=64, sinks=3, h_q=6, h_kv=2, head_dim=64, batch=2, max_tokens=600),
    dict(bits=7, group=32, residual=32, sinks=2, h_q=4, h_kv=1, head_dim=128, batch=3, max_tokens=0, window=96),
]


@pytest.mark.parametrize("shape", CASES, ids=lambda s: f"b{s['bits']}")
def test_bit_stream_widths_match_oracle(shape):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    k, v = random_stream(cfg, 560, seed=shape["bits"])
    t = 0
    for n in (1, 3, 60, 1, 200):
        p.append(k[:, :, t:t + n].contiguous(), v[:, :, t:t + n].contiguous())
        t += n
        assert p.bytes_equal()
        assert p.decode_err(random_q(cfg, t)) <= TOL
    for i in range(40):   # fused steps through at least one group freeze
        kt, vt = k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous()
        q = random_q(cfg, 1000 + i)
        out = p.gpu.append_decode(kt.cuda(), vt.cuda(), q.cuda()).float().cpu().numpy()
        assert p.ref.append(kt.numpy(), vt.numpy()) == 0
        exp = p.ref.decode_attn(q.numpy(), threads=8)
        err = (np.abs(out - exp).max(axis=-1) / np.maximum(np.abs(exp).max(axis=-1), 1e-30)).max()
        assert err <= TOL
        t += 1
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0


def test_three_bits_ragged_and_prefill():
    """3 bits at head dims 128 and 64: a ragged batch decodes per sequence and
    chunked prefill matches the oracle (at head dim 64 a lane's quarter of a
    3-bit key row starts on a 16-bit boundary, which the kernel aligns)."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    import oracle
    from gpu_util import oparams
    for d in (128, 64):
        cfg = KiviConfig(bits=3, group=32, residual=64, sinks=4, h_q=4, h_kv=4, head_dim=d, batch=3, max_tokens=600)
        c = KiviCache(cfg)
        refs = [oracle.Cache(oparams(cfg, batch=1)) for _ in range(3)]
        k, v = random_stream(cfg, 500, seed=33)
        counts = [400, 123, 7]
        c.append_ragged(k[:, :, :400].contiguous().cuda(), v[:, :, :400].contiguous().cuda(), counts)
        for b, n in enumerate(counts):
            assert refs[b].append(k[b:b + 1, :, :n].numpy(), v[b:b + 1, :, :n].numpy()) == 0
        q = random_q(cfg, 5)
        out = c.decode(q.cuda()).float().cpu().numpy()
        for b in range(3):
            assert row_rel_err(out[b:b + 1], refs[b].decode_attn(q[b:b + 1].numpy())) <= TOL, (d, b)
        g = torch.Generator().manual_seed(9)
        qq = torch.randn((3, 7, 4, d), generator=g).half()
        pout = c.prefill_ragged(qq.cuda(), [7, 7, 7]).float().cpu().numpy()
        for b in range(3):
            assert row_rel_err(pout[b:b + 1], refs[b].prefill_attn(qq[b:b + 1].numpy())) <= TOL, (d, b)
        assert c.read_error() == 0


@pytest.mark.parametrize("bits", [1, 5, 6, 7])
def test_prefill_at_head_dim_64_bit_streams(bits):
    """Chunked prefill of the other bit-stream widths at head dim 64 (quarters
    of 2 b bytes: aligned at 6 bits, on a 16-bit boundary at 1, 5 and 7)."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=bits, group=32, residual=32, sinks=3, h_q=8, h_kv=2, head_dim=64, batch=2, max_tokens=500)
    p = Pair(cfg)
    k, v = random_stream(cfg, 400, seed=bits)
    g = torch.Generator().manual_seed(bits)
    t = 0
    for m in (200, 48, 1):
        p.append(k[:, :, t:t + m].contiguous(), v[:, :, t:t + m].contiguous())
        t += m
        q = torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=g).half()
        out = p.gpu.prefill(q.cuda()).float().cpu().numpy()
        assert row_rel_err(out, p.ref.prefill_attn(q.numpy(), threads=8)) <= TOL, m
    assert p.bytes_equal()
