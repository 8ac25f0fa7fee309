"""Code widths outside {2, 4, 8} (tract #2329: configurable 1..16 bits; the
kvquant++ README recommends 3) against the oracle, through the C ABI.

These widths pack as a plain bit stream and decode on the tensor cores at
head dim 128 (two codes unpacked into one fp16x2 operand register) and on
CUDA cores at head dim 64 (decode_simt.cuh).  Bytes must equal the oracle's; decode and fused steps
within 2e-3.  Streams cross sinks, the filling ring, group freezes, a wrapping
window and ragged lengths.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, Pair, random_q, random_stream

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
    """3 bits at head dim 128 (the tensor-core path): a ragged batch decodes
    per sequence and chunked prefill matches the oracle; at head dim 64 (the
    CUDA-core path) multi-query attention is refused."""
    import ctypes
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi
    import oracle
    from gpu_util import oparams, row_rel_err
    cfg = KiviConfig(bits=3, group=32, residual=64, sinks=4, h_q=4, h_kv=4, head_dim=128, batch=3, max_tokens=600)
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
        assert row_rel_err(out[b:b + 1], refs[b].decode_attn(q[b:b + 1].numpy())) <= TOL
    g = torch.Generator().manual_seed(9)
    qq = torch.randn((3, 7, 4, 128), generator=g).half()
    pout = c.prefill_ragged(qq.cuda(), [7, 7, 7]).float().cpu().numpy()
    for b in range(3):
        assert row_rel_err(pout[b:b + 1], refs[b].prefill_attn(qq[b:b + 1].numpy())) <= TOL
    assert c.read_error() == 0
    small = KiviConfig(bits=3, group=32, residual=64, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=1, max_tokens=64)
    c64 = KiviCache(small)
    z = torch.zeros((1, 4, 8, 64), dtype=torch.float16, device="cuda")
    c64.append(z, z)
    sc = torch.empty(c64.prefill_scratch_bytes(4), dtype=torch.uint8, device="cuda")
    q4 = torch.zeros((1, 4, 4, 64), dtype=torch.float16, device="cuda")
    vp = ctypes.c_void_p
    assert _abi.lib().kivi_prefill_attn(c64._h, vp(q4.data_ptr()), vp(q4.data_ptr()), 4, vp(sc.data_ptr()),
                                        sc.numel(), None) == _abi.KIVI_EINVAL
