"""kivi_prefill_attn (causal attention of a chunk's newest tokens) against the
oracle, through the C ABI.

Chunked prefill: each chunk of M tokens is appended, then its M queries
attend, each to the tokens at or before its own position.  The streams below
run chunks through the sinks, the filling ring, chunks longer than the ring
(so a chunk's early tokens are read from frozen codes), GQA groups whose head
passes span several query tokens (rep 3 and 8), a sliding window whose slot
ring wraps and evicts part of a long chunk's early windows, and every bit
width.  The bar is the decode's: row-scaled max error <= 2e-3.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, Pair, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def chunk_q(cfg, m: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed + 7717)
    return torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=g).half()


def prefill_err(p: Pair, q: torch.Tensor) -> float:
    out = p.gpu.prefill(q.to(p.dev)).float().cpu().numpy()
    exp = p.ref.prefill_attn(q.numpy(), threads=16)
    assert np.isfinite(out).all()
    return row_rel_err(out, exp)


CASES = [
    # MHA d 64, sinks, chunks shorter and longer than the ring
    (dict(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=400),
     [5, 30, 64, 17, 1, 100]),
    # GQA rep 8 (two head passes per query token), 2-bit, d 128
    (dict(bits=2, group=32, residual=64, sinks=1, h_q=16, h_kv=2, head_dim=128, batch=2, max_tokens=400),
     [40, 33, 128, 3]),
    # GQA rep 3: a pass of four rows spans two query tokens; 8-bit, no sinks
    (dict(bits=8, group=32, residual=32, sinks=0, h_q=6, h_kv=2, head_dim=128, batch=2, max_tokens=400),
     [7, 64, 50, 90]),
    # 5 bits (bit-stream packing) at head dim 128, GQA rep 4
    (dict(bits=5, group=32, residual=64, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=400),
     [9, 70, 33]),
    # sliding window, ring of group slots wrapping; the 150-token chunk loses
    # the evicted start of its first queries' windows
    (dict(bits=4, group=16, residual=32, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=0, window=48),
     [20, 50, 70, 33, 150, 9]),
]


@pytest.mark.parametrize("shape,chunks", CASES)
def test_chunked_prefill_matches_oracle(shape, chunks):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    k, v = random_stream(cfg, sum(chunks), seed=31)
    t = 0
    for i, m in enumerate(chunks):
        p.append(k[:, :, t:t + m].contiguous(), v[:, :, t:t + m].contiguous())
        t += m
        err = prefill_err(p, chunk_q(cfg, m, seed=i))
        assert err <= TOL, (i, m, err)
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0


def test_single_query_is_the_decode():
    """n_queries = 1 is the decode (same kernel, same split): equal bits."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=64, sinks=4, h_q=16, h_kv=4, head_dim=128, batch=3, max_tokens=600)
    p = Pair(cfg)
    k, v = random_stream(cfg, 555, seed=2)
    p.append(k, v)
    q = chunk_q(cfg, 1, seed=5).cuda()
    a = p.gpu.prefill(q)
    b = p.gpu.decode(q[:, 0].contiguous())
    assert torch.equal(a[:, 0], b)


def test_full_size_chunk_against_oracle():
    """A 64-token chunk after a 4032-token context at the mha7b shape (B 8,
    32 heads, d 128, 4-bit, G 32, R 128, S 4): every row against the oracle."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=128, sinks=4, h_q=32, h_kv=32, head_dim=128, batch=8,
                     max_tokens=4096)
    p = Pair(cfg)
    k, v = random_stream(cfg, 4096, seed=8)
    p.append(k[:, :, :4032].contiguous(), v[:, :, :4032].contiguous())
    p.append(k[:, :, 4032:].contiguous(), v[:, :, 4032:].contiguous())
    assert prefill_err(p, chunk_q(cfg, 64, seed=8)) <= TOL
    assert p.gpu.read_error() == 0


def test_prefill_errors():
    import ctypes
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=1, max_tokens=64)
    c = KiviCache(cfg)
    k = torch.zeros((1, 4, 10, 64), dtype=torch.float16, device="cuda")
    c.append(k, k)
    L = _abi.lib()
    q = torch.zeros((1, 11, 4, 64), dtype=torch.float16, device="cuda")
    need = c.prefill_scratch_bytes(11)
    assert need > 0 and c.prefill_scratch_bytes(0) == 0
    sc = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    vp = ctypes.c_void_p

    def call(m, scratch=sc, nbytes=need, qp=q.data_ptr()):
        return L.kivi_prefill_attn(c._h, vp(qp), vp(out.data_ptr()), m, vp(scratch.data_ptr()), nbytes, None)

    assert call(11) == _abi.KIVI_EINVAL           # more queries than tokens
    assert call(0) == _abi.KIVI_EINVAL
    assert call(10, nbytes=c.prefill_scratch_bytes(10) - 1) == _abi.KIVI_ENOSPC
    assert call(10, qp=q.data_ptr() + 2) == _abi.KIVI_EALIGN
    assert L.kivi_prefill_attn(c._h, None, vp(out.data_ptr()), 10, vp(sc.data_ptr()), need, None) == _abi.KIVI_ENULL
    assert call(10) == _abi.KIVI_OK
    assert L.kivi_prefill_bytes(c._h, 11) == -1 and L.kivi_prefill_bytes(c._h, 10) > 0
    torch.cuda.synchronize()
    assert c.read_error() == 0
