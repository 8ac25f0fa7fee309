"""KiviCache: a thin Python handle over the C ABI of libkivi.so.

PyTorch provides the device memory (the arena and the I/O tensors) and the
CUDA stream; every computation runs in the library's kernels.  The methods
only check shapes, dtypes and devices and marshal pointers.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, asdict

import torch

from . import _abi


@dataclass(frozen=True)
class KiviConfig:
    bits: int
    group: int
    residual: int
    sinks: int
    h_q: int
    h_kv: int
    head_dim: int
    batch: int
    max_tokens: int = 0
    window: int = 0
    outlier_permille: int = 0
    rope_base: float = 0.0

    def c(self) -> _abi.KiviParams:
        return _abi.KiviParams(self.bits, self.group, self.residual, self.sinks, self.h_q, self.h_kv,
                               self.head_dim, self.batch, self.max_tokens, self.window, self.outlier_permille, 0,
                               self.rope_base)

    @staticmethod
    def from_workload(w) -> "KiviConfig":
        return KiviConfig(bits=w.bits, group=w.group, residual=w.residual, sinks=w.sinks, h_q=w.h_q,
                          h_kv=w.h_kv, head_dim=w.head_dim, batch=w.batch, max_tokens=w.max_tokens,
                          window=w.window, outlier_permille=getattr(w, "outlier_permille", 0),
                          rope_base=getattr(w, "rope_base", 0.0))


def cache_bytes(cfg: KiviConfig) -> int:
    """Arena bytes for these parameters (0 if they are invalid)."""
    p = cfg.c()
    return int(_abi.lib().kivi_cache_bytes(ctypes.byref(p)))


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class KiviCache:
    """A quantized KV cache of one attention layer on one GPU."""

    def __init__(self, cfg: KiviConfig, device="cuda", stream=None, arena: torch.Tensor | None = None,
                 restore_tokens=None):
        """A new cache (the arena is zeroed), or with restore_tokens (one
        count per sequence) a handle over an `arena` that already holds a
        cache of this config (kivi_cache_restore)."""
        self.cfg = cfg
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise ValueError("KiviCache lives on a CUDA device")
        L = _abi.lib()
        p = cfg.c()
        nbytes = int(L.kivi_cache_bytes(ctypes.byref(p)))
        if nbytes == 0:
            raise _abi.KiviError(_abi.KIVI_EINVAL, f"kivi_cache_bytes({cfg})")
        if arena is None:
            arena = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.arena = arena
        self._scratch = None   # prefill scratch, grown on demand
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            if restore_tokens is None:
                _abi.check(L.kivi_cache_create(ctypes.byref(p), ctypes.c_void_p(arena.data_ptr()),
                                               arena.numel(), ctypes.c_void_p(_stream_ptr(stream)),
                                               ctypes.byref(h)), "kivi_cache_create")
            else:
                toks = (ctypes.c_int64 * cfg.batch)(*[int(t) for t in restore_tokens])
                _abi.check(L.kivi_cache_restore(ctypes.byref(p), ctypes.c_void_p(arena.data_ptr()),
                                                arena.numel(), toks, ctypes.c_void_p(_stream_ptr(stream)),
                                                ctypes.byref(h)), "kivi_cache_restore")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _abi.lib().kivi_cache_destroy(h)
            except Exception:
                pass
            self._h = None

    # ------------------------------------------------------------------ API
    def _check_io(self, t: torch.Tensor, shape, what: str):
        if t.dtype != torch.float16:
            raise TypeError(f"{what} must be float16, got {t.dtype}")
        if t.device != self.arena.device:
            raise ValueError(f"{what} must be on {self.arena.device}, got {t.device}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{what} must be contiguous")

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
        """k_new, v_new: [B, H_kv, n, d] float16 on the cache's device."""
        c = self.cfg
        n = k_new.shape[2] if k_new.dim() == 4 else -1
        shape = (c.batch, c.h_kv, n, c.head_dim)
        self._check_io(k_new, shape, "k_new")
        self._check_io(v_new, shape, "v_new")
        _abi.check(_abi.lib().kivi_append(self._h, ctypes.c_void_p(k_new.data_ptr()),
                                          ctypes.c_void_p(v_new.data_ptr()), n,
                                          ctypes.c_void_p(_stream_ptr(stream))), "kivi_append")

    def append_ragged(self, k_new: torch.Tensor, v_new: torch.Tensor, n_tokens, stream=None) -> None:
        """k_new, v_new: [B, H_kv, n_max, d] float16; sequence b takes the
        first n_tokens[b] tokens of its rows (kivi_append_ragged)."""
        c = self.cfg
        n_max = k_new.shape[2] if k_new.dim() == 4 else -1
        shape = (c.batch, c.h_kv, n_max, c.head_dim)
        self._check_io(k_new, shape, "k_new")
        self._check_io(v_new, shape, "v_new")
        counts = (ctypes.c_int64 * c.batch)(*[int(n) for n in n_tokens])
        _abi.check(_abi.lib().kivi_append_ragged(self._h, ctypes.c_void_p(k_new.data_ptr()),
                                                 ctypes.c_void_p(v_new.data_ptr()), counts, n_max,
                                                 ctypes.c_void_p(_stream_ptr(stream))), "kivi_append_ragged")

    def tokens_per_sequence(self) -> list:
        out = (ctypes.c_int64 * self.cfg.batch)()
        _abi.check(_abi.lib().kivi_cache_tokens(self._h, out), "kivi_cache_tokens")
        return list(out)

    def decode(self, q: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """q: [B, H_q, d] float16 -> out [B, H_q, d] float16."""
        c = self.cfg
        shape = (c.batch, c.h_q, c.head_dim)
        self._check_io(q, shape, "q")
        if out is None:
            out = torch.empty(shape, dtype=torch.float16, device=self.arena.device)
        self._check_io(out, shape, "out")
        _abi.check(_abi.lib().kivi_decode_attn(self._h, ctypes.c_void_p(q.data_ptr()),
                                               ctypes.c_void_p(out.data_ptr()),
                                               ctypes.c_void_p(_stream_ptr(stream))), "kivi_decode_attn")
        return out

    def append_decode(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """One decode step: append k_new, v_new ([B, H_kv, 1, d] float16) and
        return the attention of q ([B, H_q, d] float16) over the cache
        including them (kivi_append_decode_attn)."""
        c = self.cfg
        kv_shape = (c.batch, c.h_kv, 1, c.head_dim)
        self._check_io(k_new, kv_shape, "k_new")
        self._check_io(v_new, kv_shape, "v_new")
        shape = (c.batch, c.h_q, c.head_dim)
        self._check_io(q, shape, "q")
        if out is None:
            out = torch.empty(shape, dtype=torch.float16, device=self.arena.device)
        self._check_io(out, shape, "out")
        _abi.check(_abi.lib().kivi_append_decode_attn(
            self._h, ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(_stream_ptr(stream))), "kivi_append_decode_attn")
        return out

    def append_decode_host(self, k_host: torch.Tensor, v_host: torch.Tensor, q_host: torch.Tensor,
                           out_host: torch.Tensor, stream=None) -> torch.Tensor:
        """append_decode with host-resident tensors, queued on `stream`: pinned
        tensors are read and written by the step over the host mapping;
        pageable tensors are staged through the arena with copies."""
        c = self.cfg
        shapes = ((k_host, (c.batch, c.h_kv, 1, c.head_dim), "k_host"), (v_host, (c.batch, c.h_kv, 1, c.head_dim), "v_host"),
                  (q_host, (c.batch, c.h_q, c.head_dim), "q_host"), (out_host, (c.batch, c.h_q, c.head_dim), "out_host"))
        for t, shape, what in shapes:
            if t.device.type != "cpu" or t.dtype != torch.float16 or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"{what} must be a contiguous float16 CPU tensor of shape {shape}")
        _abi.check(_abi.lib().kivi_append_decode_attn_host(
            self._h, ctypes.c_void_p(k_host.data_ptr()), ctypes.c_void_p(v_host.data_ptr()),
            ctypes.c_void_p(q_host.data_ptr()), ctypes.c_void_p(out_host.data_ptr()),
            ctypes.c_void_p(_stream_ptr(stream))), "kivi_append_decode_attn_host")
        return out_host

    def decode_host(self, q_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> torch.Tensor:
        """Host-resident q and out, queued on `stream`: pinned tensors are read
        and written by the decode over the host mapping; pageable tensors are
        staged with copies."""
        c = self.cfg
        shape = (c.batch, c.h_q, c.head_dim)
        for t, what in ((q_host, "q_host"), (out_host, "out_host")):
            if t.device.type != "cpu" or t.dtype != torch.float16 or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"{what} must be a contiguous float16 CPU tensor of shape {shape}")
        _abi.check(_abi.lib().kivi_decode_attn_host(self._h, ctypes.c_void_p(q_host.data_ptr()),
                                                    ctypes.c_void_p(out_host.data_ptr()),
                                                    ctypes.c_void_p(_stream_ptr(stream))),
                   "kivi_decode_attn_host")
        return out_host

    def prefill(self, q: torch.Tensor, out: torch.Tensor | None = None, scratch: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
        """Causal attention of the M newest tokens (append the chunk first):
        q [B, M, H_q, d] float16 -> out [B, M, H_q, d] float16
        (kivi_prefill_attn).  `scratch` is a uint8 device tensor of at least
        prefill_scratch_bytes(M) bytes; by default the cache keeps one and
        grows it as needed."""
        c = self.cfg
        m = q.shape[1] if q.dim() == 4 else -1
        shape = (c.batch, m, c.h_q, c.head_dim)
        self._check_io(q, shape, "q")
        if out is None:
            out = torch.empty(shape, dtype=torch.float16, device=self.arena.device)
        self._check_io(out, shape, "out")
        need = self.prefill_scratch_bytes(m)
        if need == 0:
            raise _abi.KiviError(_abi.KIVI_EINVAL, "kivi_prefill_scratch_bytes")
        if scratch is None:
            if self._scratch is None or self._scratch.numel() < need:
                self._scratch = torch.empty(need, dtype=torch.uint8, device=self.arena.device)
            scratch = self._scratch
        _abi.check(_abi.lib().kivi_prefill_attn(self._h, ctypes.c_void_p(q.data_ptr()),
                                                ctypes.c_void_p(out.data_ptr()), m,
                                                ctypes.c_void_p(scratch.data_ptr()), scratch.numel(),
                                                ctypes.c_void_p(_stream_ptr(stream))), "kivi_prefill_attn")
        return out

    def prefill_ragged(self, q: torch.Tensor, n_queries, out: torch.Tensor | None = None,
                       scratch: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """q [B, m_max, H_q, d] float16; sequence b's n_queries[b] newest
        tokens attend (kivi_prefill_attn_ragged).  Rows past a sequence's
        count are left as they are in `out` (zeros when out is None)."""
        c = self.cfg
        m = q.shape[1] if q.dim() == 4 else -1
        shape = (c.batch, m, c.h_q, c.head_dim)
        self._check_io(q, shape, "q")
        if out is None:
            out = torch.zeros(shape, dtype=torch.float16, device=self.arena.device)
        self._check_io(out, shape, "out")
        need = self.prefill_scratch_bytes(m)
        if need == 0:
            raise _abi.KiviError(_abi.KIVI_EINVAL, "kivi_prefill_scratch_bytes")
        if scratch is None:
            if self._scratch is None or self._scratch.numel() < need:
                self._scratch = torch.empty(need, dtype=torch.uint8, device=self.arena.device)
            scratch = self._scratch
        counts = (ctypes.c_int64 * c.batch)(*[int(n) for n in n_queries])
        _abi.check(_abi.lib().kivi_prefill_attn_ragged(self._h, ctypes.c_void_p(q.data_ptr()),
                                                       ctypes.c_void_p(out.data_ptr()), counts, m,
                                                       ctypes.c_void_p(scratch.data_ptr()), scratch.numel(),
                                                       ctypes.c_void_p(_stream_ptr(stream))),
                   "kivi_prefill_attn_ragged")
        return out

    def prefill_scratch_bytes(self, n_queries: int) -> int:
        return int(_abi.lib().kivi_prefill_scratch_bytes(self._h, n_queries))

    def prefill_bytes(self, n_queries: int) -> int:
        return int(_abi.lib().kivi_prefill_bytes(self._h, n_queries))

    def read_error(self, stream=None) -> int:
        """Reads and clears the device error word (synchronises the stream)."""
        flags = ctypes.c_uint32(0)
        _abi.check(_abi.lib().kivi_read_error(self._h, ctypes.byref(flags), ctypes.c_void_p(_stream_ptr(stream))),
                   "kivi_read_error")
        return int(flags.value)

    def set_num_splits(self, n: int) -> None:
        _abi.check(_abi.lib().kivi_set_num_splits(self._h, n), "kivi_set_num_splits")

    def layout(self) -> dict:
        L = _abi.KiviLayout()
        _abi.check(_abi.lib().kivi_cache_layout(self._h, ctypes.byref(L)), "kivi_cache_layout")
        return {n: getattr(L, n) for n, _ in _abi.KiviLayout._fields_}

    def decode_bytes(self) -> int:
        return int(_abi.lib().kivi_decode_bytes(self._h))

    @property
    def tokens(self) -> int:
        return self.layout()["tokens"]

    def cache_region(self) -> torch.Tensor:
        """A view of the cache bytes (without the workspace)."""
        return self.arena[: self.layout()["cache_bytes"]]

    def config_dict(self) -> dict:
        return asdict(self.cfg)
