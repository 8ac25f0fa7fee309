"""kivi_append_decode_attn (one call per decode step) against the oracle.

The fused step must leave the same cache bytes as the oracle's append and
return the oracle's attention over the cache including the new token, within
the parity tolerance.  The streams below step token by token through the
sink slots, the filling ring, group flushes (where the step runs the flush
launch first), a sliding window's slot ring wrapping, and GQA with more than
one head pass per kv head.
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


def fused_step(p: Pair, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor) -> float:
    """k, v: CPU float16 [B, H_kv, 1, d]; q: CPU float16 [B, H_q, d]."""
    out = p.gpu.append_decode(k.to(p.dev), v.to(p.dev), q.to(p.dev)).float().cpu().numpy()
    assert p.ref.append(k.numpy(), v.numpy()) == 0
    exp = p.ref.decode_attn(q.numpy(), threads=8)
    assert np.isfinite(out).all()
    return row_rel_err(out, exp)


CASES = [
    # sinks, ring filling and the first flushes, MHA, d 64
    dict(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=200),
    # GQA with two head passes per kv head (8 query heads per kv head), 2-bit
    dict(bits=2, group=32, residual=64, sinks=1, h_q=16, h_kv=2, head_dim=128, batch=2, max_tokens=300),
    # 8-bit, no sinks
    dict(bits=8, group=32, residual=32, sinks=0, h_q=8, h_kv=2, head_dim=128, batch=1, max_tokens=300),
    # sliding window over a wrapping ring of group slots
    dict(bits=4, group=16, residual=32, sinks=2, h_q=4, h_kv=2, head_dim=128, batch=2, max_tokens=0, window=48),
]


@pytest.mark.parametrize("shape", CASES)
def test_fused_step_matches_oracle_token_by_token(shape):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    steps = 130
    k, v = random_stream(cfg, steps, seed=11)
    worst = 0.0
    for t in range(steps):
        worst = max(worst, fused_step(p, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(),
                                      random_q(cfg, t)))
        if t % 9 == 0 or t == steps - 1:
            assert p.bytes_equal()
    assert worst <= TOL


def test_fused_step_after_bulk_prefix_and_mixed_calls():
    """A bulk-filled cache, then fused steps interleaved with plain appends
    and plain decodes: every path sees the same state."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=128, sinks=4, h_q=32, h_kv=8, head_dim=128, batch=3,
                     max_tokens=3000)
    p = Pair(cfg)
    k, v = random_stream(cfg, 2800, seed=5)
    p.append(k[:, :, :2700].contiguous(), v[:, :, :2700].contiguous())
    t = 2700
    for i in range(60):
        kt, vt = k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous()
        if i % 3 == 2:
            p.append(kt, vt)
            assert p.decode_err(random_q(cfg, 1000 + i)) <= TOL
        else:
            assert fused_step(p, kt, vt, random_q(cfg, 1000 + i)) <= TOL
        t += 1
    assert p.bytes_equal()


def test_fused_step_errors_leave_state_untouched():
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=1, max_tokens=3)
    c = KiviCache(cfg)
    k = torch.zeros((1, 4, 1, 64), dtype=torch.float16, device="cuda")
    q = torch.zeros((1, 4, 64), dtype=torch.float16, device="cuda")
    for _ in range(3):
        c.append_decode(k, k, q)
    assert c.tokens == 3
    with pytest.raises(_abi.KiviError) as e:
        c.append_decode(k, k, q)
    assert e.value.status == _abi.KIVI_ECAPACITY
    assert c.tokens == 3
    import ctypes
    L = _abi.lib()
    assert L.kivi_append_decode_attn(c._h, None, ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(q.data_ptr()), None) == _abi.KIVI_ENULL
    assert c.tokens == 3


@pytest.mark.parametrize("pinned", [True, False])
def test_fused_step_with_host_buffers_matches_device_buffers(pinned):
    """kivi_append_decode_attn_host leaves the same cache bytes and output as
    the device-buffer step: with pinned host K/V/q/out one launch gathers the
    inputs over the host mapping and the step writes the output to out_host;
    with pageable buffers the library copies them through the arena."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=120)
    a, b = KiviCache(cfg), KiviCache(cfg)
    k, v = random_stream(cfg, 100, seed=21)
    for t in range(100):
        kt, vt = k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous()
        q = random_q(cfg, 7 * t)
        out_d = a.append_decode(kt.cuda(), vt.cuda(), q.cuda())
        # host inputs held until the queued work has run
        if pinned:
            k_h, v_h, q_h = kt.pin_memory(), vt.pin_memory(), q.pin_memory()
            out_h = torch.empty_like(q).pin_memory()
        else:
            k_h, v_h, q_h, out_h = kt.clone(), vt.clone(), q.clone(), torch.empty_like(q)
        b.append_decode_host(k_h, v_h, q_h, out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(a.cache_region(), b.cache_region())


def test_fused_host_step_over_ragged_lengths_and_multiple_queries_per_head():
    """Pinned host buffers through the ragged launch (sequences of different
    lengths, GQA rep 4, one a group freeze): the same bytes and outputs as the
    device-buffer step."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    cfg = KiviConfig(bits=2, group=32, residual=64, sinks=3, h_q=16, h_kv=4, head_dim=64, batch=3, max_tokens=400)
    a, b = KiviCache(cfg), KiviCache(cfg)
    k, v = random_stream(cfg, 300, seed=5)
    counts = [300, 211, 95]
    for c in (a, b):
        c.append_ragged(k.cuda(), v.cuda(), counts)
    k2, v2 = random_stream(cfg, 40, seed=6)
    for t in range(40):
        kt, vt = k2[:, :, t:t + 1].contiguous(), v2[:, :, t:t + 1].contiguous()
        q = random_q(cfg, 11 * t)
        out_d = a.append_decode(kt.cuda(), vt.cuda(), q.cuda())
        k_h, v_h, q_h = kt.pin_memory(), vt.pin_memory(), q.pin_memory()
        out_h = torch.empty_like(q).pin_memory()
        b.append_decode_host(k_h, v_h, q_h, out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d.cpu()), t
    assert torch.equal(a.cache_region(), b.cache_region())


@pytest.mark.parametrize("extra", [dict(bits=3), dict(bits=4, rope_base=10000.0), dict(bits=2, outlier_permille=20)])
def test_fused_host_step_through_the_gather_launch(extra):
    """Caches without a host-io decode instantiation (a bit-stream width,
    pre-RoPE keys, outlier tables): pinned host buffers are gathered by one
    launch into the staging area and the output written to out_host; the same
    bytes and outputs as the device-buffer step."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    base = dict(group=32, residual=64, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=300)
    cfg = KiviConfig(**{**base, **extra})
    a, b = KiviCache(cfg), KiviCache(cfg)
    k, v = random_stream(cfg, 200, seed=31)
    for c in (a, b):
        c.append(k[:, :, :170].contiguous().cuda(), v[:, :, :170].contiguous().cuda())
    for t in range(170, 200):
        kt, vt = k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous()
        q = random_q(cfg, 5 * t)
        out_d = a.append_decode(kt.cuda(), vt.cuda(), q.cuda())
        k_h, v_h, q_h = kt.pin_memory(), vt.pin_memory(), q.pin_memory()
        out_h = torch.empty_like(q).pin_memory()
        b.append_decode_host(k_h, v_h, q_h, out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d.cpu()), t
    assert torch.equal(a.cache_region(), b.cache_region())
