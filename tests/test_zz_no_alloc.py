"""kivi_decode_attn_noalloc: decode attention for callers that cannot obtain
device memory while decoding (for instance a plugin inside a host runtime that
owns all device memory and forbids allocation during execution).

The entry point keeps its split-K scratch in a fixed 4 MiB array inside the
library.  These tests call it through the C ABI and compare it with
kivi_decode_attn, the entry point that uses the caller's arena workspace,
within the tolerance the parity tests use, on two calls in a row (the second
call must not see the first call's leftovers).  This file is collected last so
that a failure here does not hide the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import TOL, random_q, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _filled_cache(cfg, T, seed):
    from kivi_quantized_kv_gb300 import KiviCache
    c = KiviCache(cfg)
    k, v = random_stream(cfg, T, seed=seed)
    c.append(k.cuda(), v.cuda())
    return c


@pytest.mark.parametrize("shape", [
    dict(bits=4, group=32, residual=128, sinks=4, h_q=32, h_kv=8, head_dim=128, batch=4, max_tokens=3000),
    dict(bits=2, group=32, residual=64, sinks=1, h_q=8, h_kv=8, head_dim=64, batch=2, max_tokens=0, window=300),
    # a bit-stream width at head dim 64 (unaligned key quarters), with a
    # split count the fixed scratch clamps
    dict(bits=3, group=32, residual=64, sinks=4, h_q=8, h_kv=4, head_dim=64, batch=3, max_tokens=3000),
])
@pytest.mark.parametrize("ragged", [False, True])
def test_noalloc_matches_workspace_decode_twice(shape, ragged):
    from kivi_quantized_kv_gb300 import KiviConfig, _abi
    L = _abi.lib()
    cfg = KiviConfig(**shape)
    cache = _filled_cache(cfg, 2900, seed=3)
    if ragged:   # every sequence a different length: the ragged launches share the scratch
        k, v = random_stream(cfg, 60, seed=4)
        n = [(37 * b) % 60 for b in range(cfg.batch)]
        cache.append_ragged(k.cuda(), v.cuda(), n)
        assert len(set(cache.tokens_per_sequence())) == cfg.batch
    refs = []
    qs = [random_q(cfg, s).cuda() for s in (1, 2)]
    for q in qs:
        ref = cache.decode(q)                       # existing entry: arena workspace
        refs.append(ref.float().cpu().numpy())
    torch.cuda.synchronize()
    out = [torch.full_like(qs[0], float("nan")) for _ in qs]
    reserved, allocated = torch.cuda.memory_reserved(), torch.cuda.memory_allocated()
    for q, o in zip(qs, out):                       # two calls in a row
        st = L.kivi_decode_attn_noalloc(cache._h, _ptr(q), _ptr(o), _stream())
        assert st == _abi.KIVI_OK, _abi.status_string(st)
        torch.cuda.synchronize()
    # nothing went through the caller's allocator (the library itself calls
    # no allocating routine: its scratch is a fixed device array)
    assert (torch.cuda.memory_reserved(), torch.cuda.memory_allocated()) == (reserved, allocated)
    for o, ref in zip(out, refs):
        got = o.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert row_rel_err(got, ref) <= TOL
    assert cache.read_error() == 0


def test_noalloc_timeouts_reach_the_caches_error_word():
    """The bounded copy waits of a no-allocation decode report into the
    cache's own error word (in the arena the caller owns), which
    kivi_read_error reads: with the wait limit at 1 ns a wait whose copy has
    not landed at the first look gives up, and the bit shows.  The cache
    (gqa8b_b4, 155 MB) is larger than L2 and L2 is flushed before each call,
    so first block copies come from DRAM.  At the default limit the next call
    gives the output of a call made before, to within rounding."""
    from kivi_quantized_kv_gb300 import _abi
    from gpu_util import dram_resident_cache, flush_l2
    L = _abi.lib()
    cache, q = dram_resident_cache()
    o = torch.empty_like(q)
    flush_l2()
    assert L.kivi_decode_attn_noalloc(cache._h, _ptr(q), _ptr(o), _stream()) == _abi.KIVI_OK
    before = o.clone()
    assert cache.read_error() == 0
    flags = 0
    try:
        assert L.kivi_debug_set_wait_limit(1) == 0
        for _ in range(5):
            flush_l2()
            assert L.kivi_decode_attn_noalloc(cache._h, _ptr(q), _ptr(o), _stream()) == _abi.KIVI_OK
            flags |= cache.read_error()
            if flags & 1:
                break
    finally:
        assert L.kivi_debug_set_wait_limit(0) == 0
    assert flags & 1, flags
    flush_l2()
    assert L.kivi_decode_attn_noalloc(cache._h, _ptr(q), _ptr(o), _stream()) == _abi.KIVI_OK
    torch.cuda.synchronize()
    assert row_rel_err(o.float().cpu().numpy(), before.float().cpu().numpy()) <= 1e-3
    assert cache.read_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    """3 * B * h_q * (d + 4) * 4 bytes must fit in 4 MiB: 3 * 128 * 64 * 132 * 4 does not."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi
    L = _abi.lib()
    cfg = KiviConfig(bits=4, group=32, residual=128, sinks=4, h_q=64, h_kv=8, head_dim=128, batch=128,
                     max_tokens=64)
    cache = KiviCache(cfg)
    q = torch.zeros((128, 64, 128), dtype=torch.float16, device="cuda")
    o = torch.full_like(q, 7.0)
    st = L.kivi_decode_attn_noalloc(cache._h, _ptr(q), _ptr(o), _stream())
    assert st == _abi.KIVI_ESCRATCH
    assert "4 MiB" in _abi.status_string(st)
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())                   # nothing ran
    assert L.kivi_decode_attn_noalloc(None, _ptr(q), _ptr(o), _stream()) == _abi.KIVI_ENULL
