"""Checkpoint / resume and injected launch failures, through the C ABI.

A cache's state is its arena bytes, its parameters and its token counts: a
handle restored over a byte copy of the arena continues exactly like the
original.  Launch failures are injected on the host (the armed launch is
never made), so no GPU fault is involved: the call reports ECUDA, the token
counts stay, and retrying the call gives the oracle's bytes and outputs.
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


@pytest.mark.parametrize("window", [0, 64])
def test_restored_handle_continues_like_the_original(window):
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=3, h_q=8, h_kv=2, head_dim=128, batch=3,
                     max_tokens=0 if window else 400, window=window)
    a = KiviCache(cfg)
    k, v = random_stream(cfg, 300, seed=4)
    a.append(k[:, :, :200].cuda().contiguous(), v[:, :, :200].cuda().contiguous())
    a.append_ragged(k[:, :, 200:240].cuda().contiguous(), v[:, :, 200:240].cuda().contiguous(), [40, 7, 0])
    torch.cuda.synchronize()
    snap = a.arena.clone()
    b = KiviCache(cfg, arena=snap, restore_tokens=a.tokens_per_sequence())
    assert b.tokens_per_sequence() == [240, 207, 200]
    q = random_q(cfg, 3).cuda()
    assert torch.equal(a.decode(q), b.decode(q))
    for c in (a, b):
        c.append_ragged(k[:, :, 240:280].cuda().contiguous(), v[:, :, 240:280].cuda().contiguous(), [1, 33, 40])
    torch.cuda.synchronize()
    assert torch.equal(a.cache_region(), b.cache_region())
    assert torch.equal(a.decode(q), b.decode(q))
    assert a.read_error() == 0 and b.read_error() == 0


def test_injected_launch_failures_leave_counts_and_allow_retry():
    from kivi_quantized_kv_gb300 import KiviConfig, KiviError, _abi
    L = _abi.lib()
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=300)
    p = Pair(cfg)
    k, v = random_stream(cfg, 200, seed=6)
    p.append(k[:, :, :40].contiguous(), v[:, :, :40].contiguous())
    # an append that freezes groups: flush, then write; the write fails
    kt, vt = k[:, :, 40:90].contiguous().cuda(), v[:, :, 40:90].contiguous().cuda()
    assert L.kivi_debug_inject_launch_failure(2) == 0
    with pytest.raises(KiviError) as e:
        p.gpu.append(kt, vt)
    assert e.value.status == _abi.KIVI_ECUDA
    assert p.gpu.tokens == 40
    p.append(k[:, :, 40:90].contiguous(), v[:, :, 40:90].contiguous())   # the retry
    assert p.bytes_equal()
    # a decode whose launch fails writes nothing
    q = random_q(cfg, 1).cuda()
    out = torch.full((2, 4, 64), 7.0, dtype=torch.float16, device="cuda")
    assert L.kivi_debug_inject_launch_failure(1) == 0
    with pytest.raises(KiviError):
        p.gpu.decode(q, out=out)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    assert p.decode_err(q.cpu()) <= TOL
    # a fused step whose token freezes a group: flush made, decode fails
    import oracle
    t = 90
    while oracle.state_of(p.ref.p, t + 1)[1] == oracle.state_of(p.ref.p, t)[1]:
        p.append(k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous())
        t += 1
    kt, vt = k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous()
    assert L.kivi_debug_inject_launch_failure(2) == 0
    with pytest.raises(KiviError):
        p.gpu.append_decode(kt.cuda(), vt.cuda(), q)
    assert p.gpu.tokens == t
    out = p.gpu.append_decode(kt.cuda(), vt.cuda(), q).float().cpu().numpy()   # the retry
    assert p.ref.append(kt.numpy(), vt.numpy()) == 0
    exp = p.ref.decode_attn(q.cpu().numpy())
    assert np.abs(out - exp).max() / np.abs(exp).max() <= TOL
    assert p.bytes_equal()
    assert L.kivi_debug_inject_launch_failure(0) == 0
    assert p.gpu.read_error() == 0


def test_expired_copy_wait_sets_the_error_bit_and_the_next_call_is_exact():
    """Every decode wait for a copy is bounded.  With the limit set to 1 ns
    (kivi_debug_set_wait_limit) a wait gives up unless its copy has already
    landed at the first look; every copy still arrives, the warps that give up
    let their copies land, the launch ends, and bit 0 of the error word is
    set.  The cache (gqa8b_b4, 155 MB) is larger than L2 and L2 is flushed
    before each launch, so each warp's first group block comes from DRAM
    while its first look is a few hundred nanoseconds after the copy's issue.
    The next call at the default limit gives the output of a call made before
    to within rounding (which warp claims which position, and so the order of
    the fp32 sums, varies from call to call) and sets no bit; that output's
    parity with the oracle is checked at this shape in test_gpu_workloads."""
    from kivi_quantized_kv_gb300 import _abi
    from gpu_util import dram_resident_cache, flush_l2
    L = _abi.lib()
    cache, q = dram_resident_cache()
    flush_l2()
    before = cache.decode(q).clone()
    assert cache.read_error() == 0
    flags = 0
    try:
        assert L.kivi_debug_set_wait_limit(1) == 0
        for _ in range(5):   # thousands of first looks per launch; one running out is enough
            flush_l2()
            cache.decode(q)
            flags |= cache.read_error()
            if flags & 1:
                break
    finally:
        assert L.kivi_debug_set_wait_limit(0) == 0
    assert flags & 1, flags
    flush_l2()
    after = cache.decode(q)
    torch.cuda.synchronize()
    assert row_rel_err(after.float().cpu().numpy(), before.float().cpu().numpy()) <= 1e-3
    assert cache.read_error() == 0
