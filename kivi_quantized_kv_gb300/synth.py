"""Seeded synthetic K/V/q workloads for the KIVI cache.

This module only draws inputs.  It holds none of the method's arithmetic (no
quantization, packing or attention), so both the CUDA path and the CPU oracle
can be fed from it.

Distributions (stand-ins for the real GPT-2 / OpenELM activations the pages
measure on, which are not available here):
  * keys: N(0, 1) with a fixed set of outlier channels per (layer, kv-head),
    scaled by a constant (tiny workload: x20) or by U(10, 30) per channel —
    the "few fixed channels with large magnitude" of the KV-cache quantization
    guide (pigeon), "How it works", step 1;
  * RoPE-shaped workloads apply the rotary embedding (theta = 10000,
    rotate-half pairing) to the pre-RoPE keys at their absolute positions;
  * values: N(0, 1) times a per-token log-normal scale exp(N(0, 0.5^2))
    ("values have no fixed outlier channels", same page, step 2); the tiny
    workload keeps plain N(0, 1) values;
  * queries: N(0, 1).
Generation is chunked and sequential: a ``KVStream`` draws token chunks in
order from one seeded ``torch.Generator``; the same chunks are given to every
consumer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_q: int
    h_kv: int
    head_dim: int
    tokens: int            # T: tokens in the cache when decode attention runs
    bits: int
    group: int
    residual: int
    sinks: int
    window: int = 0        # 0 = unbounded
    layers: int = 1
    outlier_channels: int = 4
    outlier_fixed: Optional[float] = None   # constant outlier scale, else U(lo, hi)
    outlier_range: tuple = (10.0, 30.0)
    rope: bool = False
    v_lognormal: bool = True
    seed: int = 0
    outlier_permille: int = 0   # dense-and-sparse: values per thousand kept exactly in the side tables
    rope_base: float = 0.0      # > 0: the cache takes pre-RoPE keys and rotates them at attention

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def max_tokens(self) -> int:
        return 0 if self.window > 0 else self.tokens


# The five workloads of the measurement plan.  Sizes are those of the
# published models the shapes are named after; data are synthetic.
WORKLOADS = {
    "tiny": Workload("tiny", batch=1, h_q=4, h_kv=4, head_dim=64, tokens=256, bits=4, group=32,
                     residual=32, sinks=4, outlier_fixed=20.0, v_lognormal=False),
    "mha7b": Workload("mha7b", batch=8, h_q=32, h_kv=32, head_dim=128, tokens=4096, bits=4,
                      group=32, residual=128, sinks=4),
    "gqa8b_b4": Workload("gqa8b_b4", batch=4, h_q=32, h_kv=8, head_dim=128, tokens=32768, bits=4,
                         group=32, residual=128, sinks=4, rope=True),
    "gqa8b_b2": Workload("gqa8b_b2", batch=4, h_q=32, h_kv=8, head_dim=128, tokens=32768, bits=2,
                         group=32, residual=128, sinks=4, rope=True),
    "swa_mistral": Workload("swa_mistral", batch=32, h_q=32, h_kv=8, head_dim=128, tokens=16384,
                            bits=8, group=64, residual=64, sinks=4, window=4096, rope=True),
    # the mha7b and gqa8b shapes at 3 bits (kvquant++'s recommended width),
    # packed as a bit stream
    "mha7b_b3": Workload("mha7b_b3", batch=8, h_q=32, h_kv=32, head_dim=128, tokens=4096, bits=3,
                         group=32, residual=128, sinks=4),
    "gqa8b_b3": Workload("gqa8b_b3", batch=4, h_q=32, h_kv=8, head_dim=128, tokens=32768, bits=3,
                         group=32, residual=128, sinks=4, rope=True),
    # dense-and-sparse: the mha7b shape with 1 % of each key and value block
    # kept exactly in the outlier tables (KVQuant's pairing of 3 bits and 1 %)
    "mha7b_o10": Workload("mha7b_o10", batch=8, h_q=32, h_kv=32, head_dim=128, tokens=4096, bits=4,
                          group=32, residual=128, sinks=4, outlier_permille=10),
    "mha7b_b3_o10": Workload("mha7b_b3_o10", batch=8, h_q=32, h_kv=32, head_dim=128, tokens=4096, bits=3,
                             group=32, residual=128, sinks=4, outlier_permille=10),
    # pre-RoPE keys: the gqa8b shape with its keys given to the cache before
    # the rotary embedding (the stream does not rotate them); the cache
    # rotates each key at its position inside the decode
    "gqa8b_b4_prerope": Workload("gqa8b_b4_prerope", batch=4, h_q=32, h_kv=8, head_dim=128, tokens=32768, bits=4,
                                 group=32, residual=128, sinks=4, rope=False, rope_base=10000.0),
    # head dim 64 at 3 bits: a bit-stream width whose key quarters may start
    # on a 16-bit boundary
    "mha_d64_b3": Workload("mha_d64_b3", batch=8, h_q=32, h_kv=32, head_dim=64, tokens=4096, bits=3,
                           group=32, residual=128, sinks=4),
}


def sweep_workload(batch: int, tokens: int, bits: int) -> Workload:
    """One cell of the 32-layer decode-step sweep (H 32/8, d 128, G 32, R 128, S 4)."""
    return Workload(f"sweep_B{batch}_T{tokens}_b{bits}", batch=batch, h_q=32, h_kv=8, head_dim=128,
                    tokens=tokens, bits=bits, group=32, residual=128, sinks=4, layers=32, rope=True)


SWEEP_BATCH = (1, 16, 128)
SWEEP_TOKENS = (1024, 16384, 131072)
SWEEP_BITS = (2, 4, 8)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


class KVStream:
    """Draws the K/V token stream of one layer, chunk by chunk, in order.

    ``next(n)`` returns (k, v), each [B, H_kv, n, d] float16 on ``device``,
    for absolute positions [pos, pos + n); ``pos`` then advances by n.
    """

    def __init__(self, w: Workload, layer: int = 0, device="cpu"):
        self.w = w
        self.device = torch.device(device)
        self.pos = 0
        seed = w.seed * 1000003 + layer
        self.g = _gen(seed, self.device)
        d = w.head_dim
        # fixed outlier channels and their scales, per kv head
        scale = torch.ones(w.h_kv, d, device=self.device)
        for h in range(w.h_kv):
            ch = torch.randperm(d, generator=self.g, device=self.device)[: w.outlier_channels]
            if w.outlier_fixed is not None:
                s = torch.full((w.outlier_channels,), float(w.outlier_fixed), device=self.device)
            else:
                lo, hi = w.outlier_range
                s = lo + (hi - lo) * torch.rand(w.outlier_channels, generator=self.g, device=self.device)
            scale[h, ch] = s
        self.k_scale = scale.view(1, w.h_kv, 1, d)
        if w.rope:
            half = d // 2
            self.inv_freq = 10000.0 ** (-torch.arange(half, device=self.device, dtype=torch.float64) * 2.0 / d)

    def _rope(self, k: torch.Tensor, pos0: int) -> torch.Tensor:
        n, d = k.shape[2], k.shape[3]
        half = d // 2
        pos = torch.arange(pos0, pos0 + n, device=self.device, dtype=torch.float64)
        ang = pos[:, None] * self.inv_freq[None, :]
        cos = torch.cos(ang).float()
        sin = torch.sin(ang).float()
        k1, k2 = k[..., :half], k[..., half:]
        return torch.cat([k1 * cos - k2 * sin, k2 * cos + k1 * sin], dim=-1)

    def next(self, n: int):
        w = self.w
        shape = (w.batch, w.h_kv, n, w.head_dim)
        k = torch.randn(shape, generator=self.g, device=self.device) * self.k_scale
        if w.rope:
            k = self._rope(k, self.pos)
        v = torch.randn(shape, generator=self.g, device=self.device)
        if w.v_lognormal:
            tok = torch.exp(0.5 * torch.randn((w.batch, w.h_kv, n, 1), generator=self.g, device=self.device))
            v = v * tok
        self.pos += n
        return k.half().contiguous(), v.half().contiguous()


def queries(w: Workload, step: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """Decode queries [B, H_q, d] float16 for one step of one layer."""
    g = _gen(w.seed * 7919 + layer * 104729 + step + 17, device)
    return torch.randn((w.batch, w.h_q, w.head_dim), generator=g, device=device).half().contiguous()


def fill_chunks(total: int, chunk: int):
    """Chunk sizes that sum to ``total``."""
    out = []
    left = total
    while left > 0:
        c = min(chunk, left)
        out.append(c)
        left -= c
    return out
