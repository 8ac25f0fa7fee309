"""Ragged batches: sequences of different lengths in one cache, through the C
ABI, against one single-sequence oracle cache per sequence.

Each sequence of a ragged batch must hold the bytes it would hold alone and
attend over its own tokens only.  The streams append a different number of
tokens to each sequence per round (some zero, some equal neighbours so that
runs span several sequences), then run the causal attention of each
sequence's new tokens, decode steps (plain and fused) on the ragged state,
and a uniform-count prefill on it; a windowed GQA case wraps the slot ring.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, oparams, random_stream, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Ragged:
    """A CUDA cache of B sequences and B single-sequence oracle caches."""

    def __init__(self, cfg):
        from kivi_quantized_kv_gb300 import KiviCache
        self.cfg = cfg
        self.gpu = KiviCache(cfg)
        self.ref = [oracle.Cache(oparams(cfg, batch=1)) for _ in range(cfg.batch)]
        self.streams = [random_stream(oparams(cfg, batch=1), 1200, seed=100 + b) for b in range(cfg.batch)]
        self.pos = [0] * cfg.batch

    def append(self, counts):
        c = self.cfg
        n_max = max(max(counts), 1)
        k = torch.zeros((c.batch, c.h_kv, n_max, c.head_dim), dtype=torch.float16)
        v = torch.zeros_like(k)
        for b, n in enumerate(counts):
            ks, vs = self.streams[b]
            k[b, :, :n] = ks[0, :, self.pos[b]:self.pos[b] + n]
            v[b, :, :n] = vs[0, :, self.pos[b]:self.pos[b] + n]
            if n:
                assert self.ref[b].append(k[b:b + 1, :, :n].numpy(), v[b:b + 1, :, :n].numpy()) == 0
            self.pos[b] += n
        self.gpu.append_ragged(k.cuda(), v.cuda(), counts)
        assert self.gpu.tokens_per_sequence() == self.pos

    def bytes_equal(self):
        torch.cuda.synchronize()
        region = self.gpu.cache_region().cpu().numpy()
        per_seq = self.gpu.layout()["unit_bytes"] * self.cfg.h_kv
        for b in range(self.cfg.batch):
            assert np.array_equal(region[b * per_seq:(b + 1) * per_seq], self.ref[b].arena()), b
        return True

    def prefill_err(self, counts, seed):
        c = self.cfg
        m = max(max(counts), 1)
        g = torch.Generator().manual_seed(seed)
        q = torch.randn((c.batch, m, c.h_q, c.head_dim), generator=g).half()
        out = self.gpu.prefill_ragged(q.cuda(), counts).float().cpu().numpy()
        worst = 0.0
        for b, n in enumerate(counts):
            if n == 0:
                assert not out[b].any()
                continue
            exp = self.ref[b].prefill_attn(q[b:b + 1, :n].numpy(), threads=8)
            worst = max(worst, row_rel_err(out[b:b + 1, :n], exp))
            assert not out[b, n:].any()   # rows past the count are not written
        return worst

    def decode_err(self, q):
        out = self.gpu.decode(q.cuda()).float().cpu().numpy()
        return max(row_rel_err(out[b:b + 1], self.ref[b].decode_attn(q[b:b + 1].numpy(), threads=8))
                   for b in range(self.cfg.batch))

    def fused_err(self, q):
        c = self.cfg
        k = torch.zeros((c.batch, c.h_kv, 1, c.head_dim), dtype=torch.float16)
        v = torch.zeros_like(k)
        for b in range(c.batch):
            ks, vs = self.streams[b]
            k[b, :, 0] = ks[0, :, self.pos[b]]
            v[b, :, 0] = vs[0, :, self.pos[b]]
            assert self.ref[b].append(k[b:b + 1].numpy(), v[b:b + 1].numpy()) == 0
            self.pos[b] += 1
        out = self.gpu.append_decode(k.cuda(), v.cuda(), q.cuda()).float().cpu().numpy()
        return max(row_rel_err(out[b:b + 1], self.ref[b].decode_attn(q[b:b + 1].numpy(), threads=8))
                   for b in range(c.batch))


def q_of(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((cfg.batch, cfg.h_q, cfg.head_dim), generator=g).half()


CASES = [
    (dict(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=4, max_tokens=600),
     [[5, 0, 17, 64], [30, 12, 0, 1], [100, 33, 50, 7], [1, 1, 1, 1], [0, 90, 90, 90]]),
    (dict(bits=2, group=32, residual=64, sinks=1, h_q=16, h_kv=2, head_dim=128, batch=3, max_tokens=600),
     [[40, 40, 3], [128, 0, 128], [33, 70, 33]]),
    (dict(bits=4, group=16, residual=32, sinks=2, h_q=8, h_kv=2, head_dim=128, batch=3, max_tokens=0, window=48),
     [[20, 20, 7], [70, 70, 70], [0, 150, 9], [33, 1, 64]]),
]


@pytest.mark.parametrize("shape,rounds", CASES)
def test_ragged_chunked_prefill_and_decode(shape, rounds):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    r = Ragged(cfg)
    for i, counts in enumerate(rounds):
        r.append(counts)
        assert r.prefill_err(counts, seed=i) <= TOL, (i, counts)
        assert r.decode_err(q_of(cfg, 50 + i)) <= TOL
    for i in range(20):   # fused steps on the ragged state
        assert r.fused_err(q_of(cfg, 90 + i)) <= TOL
    assert r.bytes_equal()
    # a uniform query count on ragged lengths
    m = min(r.pos)
    g = torch.Generator().manual_seed(7)
    q = torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=g).half()
    out = r.gpu.prefill(q.cuda()).float().cpu().numpy()
    for b in range(cfg.batch):
        assert row_rel_err(out[b:b + 1], r.ref[b].prefill_attn(q[b:b + 1].numpy(), threads=8)) <= TOL
    assert r.gpu.read_error() == 0


def test_ragged_argument_errors():
    import ctypes
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=2, max_tokens=40)
    c = KiviCache(cfg)
    L = _abi.lib()
    k = torch.zeros((2, 4, 8, 64), dtype=torch.float16, device="cuda")
    vp = ctypes.c_void_p

    def app(counts, n_max=8):
        arr = (ctypes.c_int64 * 2)(*counts)
        return L.kivi_append_ragged(c._h, vp(k.data_ptr()), vp(k.data_ptr()), arr, n_max, None)

    assert app([9, 0]) == _abi.KIVI_EINVAL
    assert app([-1, 0]) == _abi.KIVI_EINVAL
    assert app([1, 1], n_max=0) == _abi.KIVI_EINVAL
    assert app([8, 3]) == _abi.KIVI_OK
    assert c.tokens_per_sequence() == [8, 3] and c.tokens == -1
    for _ in range(4):
        assert app([8, 0]) == _abi.KIVI_OK
    assert app([1, 0]) == _abi.KIVI_ECAPACITY   # 41 > max_tokens
    assert c.tokens_per_sequence() == [40, 3]
    q = torch.zeros((2, 4, 4, 64), dtype=torch.float16, device="cuda")
    sc = torch.empty(c.prefill_scratch_bytes(4), dtype=torch.uint8, device="cuda")
    arr = (ctypes.c_int64 * 2)(4, 4)   # sequence 1 holds only 3 tokens
    assert L.kivi_prefill_attn_ragged(c._h, vp(q.data_ptr()), vp(q.data_ptr()), arr, 4, vp(sc.data_ptr()),
                                      sc.numel(), None) == _abi.KIVI_EINVAL
    out = torch.zeros_like(q)
    arr = (ctypes.c_int64 * 2)(4, 3)
    assert L.kivi_prefill_attn_ragged(c._h, vp(q.data_ptr()), vp(out.data_ptr()), arr, 4, vp(sc.data_ptr()),
                                      sc.numel(), None) == _abi.KIVI_OK
    assert L.kivi_prefill_bytes(c._h, 4) == -1 and L.kivi_prefill_bytes(c._h, 3) > 0
    torch.cuda.synchronize()


def test_more_runs_than_one_ragged_launch_holds():
    """70 sequences of 70 different lengths: more runs than one ragged launch
    takes (64), so the decode and the fused step are split over two."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=16, residual=32, sinks=2, h_q=2, h_kv=1, head_dim=64, batch=70, max_tokens=200)
    r = Ragged(cfg)
    r.append([b + 1 for b in range(70)])                  # lengths 1 .. 70
    r.append([(37 * b) % 61 for b in range(70)])          # ragged again, some zeros
    assert len(set(r.pos)) > 64
    for i in range(3):
        assert r.decode_err(q_of(cfg, 300 + i)) <= TOL
        assert r.fused_err(q_of(cfg, 400 + i)) <= TOL
    assert r.bytes_equal()
    assert r.gpu.read_error() == 0


def test_ragged_decode_at_the_mha7b_shape():
    """B 8, 32 heads, d 128, 4-bit, G 32, R 128, S 4 with lengths 4095 - 256 b
    (eight runs, one ragged launch): every sequence's decode and fused steps
    against its own oracle cache."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(bits=4, group=32, residual=128, sinks=4, h_q=32, h_kv=32, head_dim=128, batch=8,
                     max_tokens=4200)
    r = Ragged.__new__(Ragged)
    from kivi_quantized_kv_gb300 import KiviCache
    r.cfg = cfg
    r.gpu = KiviCache(cfg)
    r.ref = [oracle.Cache(oparams(cfg, batch=1)) for _ in range(cfg.batch)]
    r.streams = [random_stream(oparams(cfg, batch=1), 4200, seed=700 + b) for b in range(cfg.batch)]
    r.pos = [0] * cfg.batch
    r.append([4095 - 256 * b for b in range(8)])
    assert r.decode_err(q_of(cfg, 1)) <= TOL
    for i in range(40):   # crosses group freezes of several sequences at different steps
        assert r.fused_err(q_of(cfg, 10 + i)) <= TOL
    assert r.bytes_equal()
    assert r.gpu.read_error() == 0
