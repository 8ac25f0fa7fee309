"""GPU parity: the CUDA cache against the CPU oracle, through the C ABI.

Packed bytes (codes, fp16 scales and zero points, fp32 sinks, fp16 ring) must
be identical; decode attention must be within 2e-3 (row-scaled max error, see
gpu_util).  Sizes span several groups, splits and a ragged tail; the edge
cases are T = 0, T < S, T = S + R (ring full, nothing frozen), the first
flush, bulk appends that cross many groups, windows, and every bit width.
"""
import numpy as np
import pytest
import torch

from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, KiviError
from gpu_util import TOL, Pair, random_q, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def cfg(**kw):
    base = dict(bits=4, group=32, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=1, max_tokens=256)
    base.update(kw)
    return KiviConfig(**base)


def test_tiny_workload_chunked():
    c = cfg()
    p = Pair(c)
    k, v = random_stream(c, 256, seed=1)
    t = 0
    for n in (1, 3, 33, 1, 64, 100, 54):
        p.append(k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
        p.bytes_equal()
        assert p.decode_err(random_q(c, t)) <= TOL
    assert t == 256


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("G,R,S,d", [(16, 16, 0, 64), (32, 64, 4, 128), (64, 128, 1, 128), (16, 48, 7, 64)])
def test_bits_groups_dims(bits, G, R, S, d):
    c = cfg(bits=bits, group=G, residual=R, sinks=S, head_dim=d, batch=2, h_q=8, h_kv=2, max_tokens=700)
    p = Pair(c)
    k, v = random_stream(c, 700, seed=bits * 7 + G)
    p.append(k[:, :, :517], v[:, :, :517])
    p.bytes_equal()
    assert p.decode_err(random_q(c, 1)) <= TOL
    p.append(k[:, :, 517:700], v[:, :, 517:700])
    p.bytes_equal()
    assert p.decode_err(random_q(c, 2)) <= TOL


@pytest.mark.parametrize("rep", [1, 2, 4, 8])
def test_gqa_ratios(rep):
    c = cfg(h_q=2 * rep, h_kv=2, batch=3, max_tokens=300, head_dim=128)
    p = Pair(c)
    k, v = random_stream(c, 300, seed=rep)
    p.append(k, v)
    p.bytes_equal()
    assert p.decode_err(random_q(c, rep)) <= TOL


def test_token_by_token_around_flush_boundaries():
    """Single-token appends (the decode-step pattern) across several flushes;
    bytes and attention checked at every step near a boundary."""
    c = cfg(group=16, residual=32, sinks=3, h_q=4, h_kv=2, batch=2, max_tokens=140)
    p = Pair(c)
    k, v = random_stream(c, 140, seed=5)
    for t in range(140):
        p.append(k[:, :, t:t + 1], v[:, :, t:t + 1])
        T = t + 1
        near = (T - 3) % 16 in (0, 1, 15) or T <= 4
        if near or T % 29 == 0:
            p.bytes_equal()
            assert p.decode_err(random_q(c, T)) <= TOL


def test_edge_token_counts():
    c = cfg(max_tokens=64)
    p = Pair(c)
    q = random_q(c, 0)
    # T = 0: nothing to attend to, the output is zero
    out = p.gpu.decode(q.cuda()).float().cpu().numpy()
    assert np.all(out == 0)
    k, v = random_stream(c, 64, seed=6)
    p.append(k[:, :, :2], v[:, :, :2])           # T < S: sinks only
    p.bytes_equal()
    assert p.decode_err(q) <= TOL
    p.append(k[:, :, 2:36], v[:, :, 2:36])       # T = S + R: ring full, no group
    assert p.gpu.layout()["n_groups"] == 0 and p.gpu.layout()["n_res"] == 32
    p.bytes_equal()
    assert p.decode_err(q) <= TOL
    p.append(k[:, :, 36:37], v[:, :, 36:37])     # first flush
    assert p.gpu.layout()["n_groups"] == 1 and p.gpu.layout()["n_res"] == 1
    p.bytes_equal()
    assert p.decode_err(q) <= TOL


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_forced_split_counts(splits):
    c = cfg(bits=2, head_dim=128, h_q=8, h_kv=2, batch=2, max_tokens=1200, residual=64)
    p = Pair(c)
    k, v = random_stream(c, 1111, seed=splits)
    p.append(k, v)
    p.gpu.set_num_splits(splits)
    assert p.decode_err(random_q(c, splits)) <= TOL


@pytest.mark.parametrize("W,chunk", [(64, 1), (100, 37), (256, 250), (64, 1000)])
def test_sliding_window(W, chunk):
    c = cfg(window=W, max_tokens=0, group=16, residual=32, sinks=4, h_q=4, h_kv=2, batch=2)
    p = Pair(c)
    k, v = random_stream(c, 1500, seed=W + chunk)
    t = 0
    while t < 1500:
        n = min(chunk, 1500 - t)
        p.append(k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
        if chunk > 1 or t % 97 == 0 or t < 80:
            p.bytes_equal()
            assert p.decode_err(random_q(c, t)) <= TOL


def test_bulk_equals_sequential_on_gpu():
    c = cfg(bits=8, group=32, residual=64, h_q=2, h_kv=2, batch=2, max_tokens=400)
    k, v = random_stream(c, 400, seed=8)
    a = KiviCache(c)
    b = KiviCache(c)
    a.append(k.cuda(), v.cuda())
    for t in range(0, 400, 7):
        n = min(7, 400 - t)
        b.append(k[:, :, t:t + n].cuda().contiguous(), v[:, :, t:t + n].cuda().contiguous())
    torch.cuda.synchronize()
    assert torch.equal(a.cache_region(), b.cache_region())


def test_errors_leave_state_untouched():
    c = cfg(max_tokens=40)
    p = Pair(c)
    k, v = random_stream(c, 41, seed=9)
    p.append(k[:, :, :40], v[:, :, :40])
    torch.cuda.synchronize()
    before = p.gpu.cache_region().clone()
    with pytest.raises(KiviError) as e:
        p.gpu.append(k[:, :, 40:41].cuda(), v[:, :, 40:41].cuda())
    assert e.value.status == 3  # KIVI_ECAPACITY
    kk = torch.zeros(1 * 4 * 1 * 64 + 8, dtype=torch.float16, device="cuda")
    mis = kk[1:1 + 4 * 64].view(1, 4, 1, 64)
    with pytest.raises(KiviError) as e:
        KiviCache(cfg(max_tokens=80)).append(mis, mis)
    assert e.value.status == 2  # KIVI_EALIGN
    torch.cuda.synchronize()
    assert torch.equal(before, p.gpu.cache_region())
    assert p.gpu.tokens == 40


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_matches_device_entry(pinned):
    """kivi_decode_attn_host: a pinned q is gathered by one launch over the
    host mapping and the output written to the pinned out; pageable buffers
    are copied through the arena."""
    c = cfg(batch=2, h_q=8, h_kv=2, max_tokens=300)
    p = Pair(c)
    k, v = random_stream(c, 300, seed=10)
    p.append(k, v)
    q = random_q(c, 3)
    dev_out = p.gpu.decode(q.cuda()).cpu()
    q_host = q.clone().pin_memory() if pinned else q.clone()
    out_host = torch.empty_like(q).pin_memory() if pinned else torch.empty_like(q)
    p.gpu.decode_host(q_host, out_host)
    torch.cuda.synchronize()
    assert torch.equal(dev_out, out_host)


def test_layout_matches_oracle():
    for c in (cfg(), cfg(bits=2, head_dim=128, window=300, max_tokens=0, group=64, residual=128)):
        gl = KiviCache(c).layout()
        ol = Pair(c).ref.layout
        for key, val in ol.items():
            assert gl[key] == val, key
