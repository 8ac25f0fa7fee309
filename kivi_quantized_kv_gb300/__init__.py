"""GB300-native KIVI quantized KV cache: packed 2/4/8-bit storage and split-K
decode attention over it, behind the C ABI of libkivi.so (include/kivi.h).

The Python layer only marshals arguments; build the library with
``python -c 'import __graft_entry__ as g; g.build()'``.
"""
from .cache import KiviCache, KiviConfig, cache_bytes  # noqa: F401
from ._abi import KiviError, lib  # noqa: F401

__all__ = ["KiviCache", "KiviConfig", "KiviError", "cache_bytes", "lib"]
