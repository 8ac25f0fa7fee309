"""Helpers for the GPU parity tests: drive the CUDA cache and the oracle with
the same inputs and compare them.

Tolerance (the spec's "max relative error <= 2e-3"): per (sequence, query
head) row, max_c |out - ref| / max_c |ref|, maximum over rows, where ref is
the oracle's fp64 attention over the same dequantized values.  Element-wise
relative error is ill-posed for channels near zero, hence the row scale.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kivi_quantized_kv_gb300 import KiviCache, KiviConfig

TOL = 2e-3


def oparams(cfg: KiviConfig, **over) -> oracle.Params:
    d = {f: getattr(cfg, f) for f in cfg.__dataclass_fields__}
    d.update(over)
    return oracle.Params(**d)


def row_rel_err(out: np.ndarray, ref: np.ndarray) -> float:
    out = out.reshape(-1, out.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1])
    scale = np.abs(ref).max(axis=1)
    scale = np.where(scale == 0, 1.0, scale)
    return float((np.abs(out - ref).max(axis=1) / scale).max())


class Pair:
    """A CUDA cache and an oracle cache fed the same token stream."""

    def __init__(self, cfg: KiviConfig, device="cuda"):
        self.cfg = cfg
        self.dev = torch.device(device)
        self.gpu = KiviCache(cfg, device=self.dev)
        self.ref = oracle.Cache(oparams(cfg))

    def append(self, k: torch.Tensor, v: torch.Tensor):
        """k, v: CPU float16 [B, H_kv, n, d]."""
        self.gpu.append(k.to(self.dev), v.to(self.dev))
        assert self.ref.append(k.numpy(), v.numpy()) == 0

    def bytes_equal(self) -> bool:
        torch.cuda.synchronize()
        got = self.gpu.cache_region().cpu().numpy()
        exp = self.ref.arena()
        if not np.array_equal(got, exp):
            bad = np.flatnonzero(got != exp)
            L = self.ref.layout
            u, off = divmod(int(bad[0]), L["unit_bytes"])
            raise AssertionError(f"{bad.size} bytes differ; first at unit {u} offset {off} "
                                 f"(groups start {L['groups']}, block {L['block_bytes']})")
        return True

    def decode_err(self, q: torch.Tensor) -> float:
        out = self.gpu.decode(q.to(self.dev)).float().cpu().numpy()
        exp = self.ref.decode_attn(q.numpy(), threads=8)
        assert np.isfinite(out).all()
        return row_rel_err(out, exp)


def random_stream(cfg: KiviConfig, T: int, seed: int, outliers: bool = True):
    g = torch.Generator().manual_seed(seed)
    shape = (cfg.batch, cfg.h_kv, T, cfg.head_dim)
    k = torch.randn(shape, generator=g)
    if outliers:
        k[..., 1] *= 25
        k[..., cfg.head_dim - 3] *= 12
    v = torch.randn(shape, generator=g) * torch.exp(0.5 * torch.randn((*shape[:3], 1), generator=g))
    return k.half(), v.half()


def random_q(cfg: KiviConfig, seed: int):
    g = torch.Generator().manual_seed(seed + 99991)
    return torch.randn((cfg.batch, cfg.h_q, cfg.head_dim), generator=g).half()


def dram_resident_cache(workload="gqa8b_b4"):
    """A cache of a full-size workload (about 155 MB for gqa8b_b4: larger
    than the 129 MB L2), filled from the seeded device-side stream, and its
    decode queries."""
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    from kivi_quantized_kv_gb300.synth import KVStream, WORKLOADS, queries
    w = WORKLOADS[workload]
    dev = torch.device("cuda")
    cache = KiviCache(KiviConfig.from_workload(w), device=dev)
    stream = KVStream(w, device=dev)
    t = 0
    while t < w.tokens:
        n = min(4096, w.tokens - t)
        k, v = stream.next(n)
        cache.append(k, v)
        t += n
    return cache, queries(w, device=dev)


_FLUSH = {}


def flush_l2():
    """Writes 512 MB on the current stream, so the next launch finds none of
    the cache in the 129 MB L2."""
    buf = _FLUSH.get("buf")
    if buf is None:
        buf = _FLUSH["buf"] = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
