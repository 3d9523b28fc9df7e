"""Host block pool and KV-cache manager (``include/pa_kv_manager.h``) from Python.

``KVCacheManager`` wraps the C++ manager in ``libpa.so``: it hands out the physical
blocks of the paged KV pool, keeps each request's block table, shares full blocks between
requests with equal token prefixes (prefix caching) and reports copy-on-write block
pairs for forked requests.  Marshalling only: the policy lives in the C++ code.
"""
from __future__ import annotations

import ctypes
from typing import List, Sequence, Tuple

import numpy as np

from . import PAError, _lib

__all__ = ["KVCacheManager"]

_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
_lib.pa_kvm_create.argtypes = [_i32, _i32, _i32, ctypes.POINTER(_vp)]
_lib.pa_kvm_destroy.argtypes = [_vp]
_lib.pa_kvm_destroy.restype = None
_lib.pa_kvm_get_computed_blocks.argtypes = [_vp, _vp, _i32, _vp, _i32, ctypes.POINTER(_i32)]
_lib.pa_kvm_admit.argtypes = [_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)]
_lib.pa_kvm_allocate_slots.argtypes = [_vp, _i64, _i32, _vp, _i32, ctypes.POINTER(_i32)]
_lib.pa_kvm_cache_blocks.argtypes = [_vp, _i64, _vp, _i32]
_lib.pa_kvm_free.argtypes = [_vp, _i64]
_lib.pa_kvm_fork.argtypes = [_vp, _i64, _i64]
_lib.pa_kvm_block_table.argtypes = [_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)]
_lib.pa_kvm_slot_mapping.argtypes = [_vp, _i64, _i32, _i32, _vp]
_lib.pa_kvm_num_free_blocks.argtypes = [_vp]
_lib.pa_kvm_stats.argtypes = [_vp, _vp]
for _n in ("pa_kvm_create", "pa_kvm_get_computed_blocks", "pa_kvm_admit", "pa_kvm_allocate_slots",
           "pa_kvm_cache_blocks", "pa_kvm_free", "pa_kvm_fork", "pa_kvm_block_table",
           "pa_kvm_slot_mapping", "pa_kvm_num_free_blocks", "pa_kvm_stats"):
    getattr(_lib, _n).restype = _i32


def _check(code: int, what: str) -> None:
    if code != 0:
        raise PAError(code, what)


def _tok(tokens) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))


class KVCacheManager:
    """Block pool of ``num_blocks`` blocks of ``block_size`` tokens with prefix caching."""

    def __init__(self, num_blocks: int, block_size: int, prefix_cache: bool = True):
        h = _vp()
        _check(_lib.pa_kvm_create(num_blocks, block_size, 1 if prefix_cache else 0, ctypes.byref(h)),
               "pa_kvm_create")
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.pa_kvm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def get_computed_blocks(self, tokens: Sequence[int]) -> List[int]:
        t = _tok(tokens)
        out = np.empty(max(1, len(t) // self.block_size), dtype=np.int32)
        n = _i32()
        _check(_lib.pa_kvm_get_computed_blocks(self._h, t.ctypes.data, len(t), out.ctypes.data, len(out),
                                               ctypes.byref(n)), "pa_kvm_get_computed_blocks")
        return out[:n.value].tolist()

    def admit(self, req_id: int, tokens: Sequence[int]) -> int:
        """Register a request; returns how many of its prompt tokens are already cached."""
        t = _tok(tokens)
        n = _i32()
        _check(_lib.pa_kvm_admit(self._h, req_id, t.ctypes.data, len(t), ctypes.byref(n)), "pa_kvm_admit")
        return n.value

    def allocate_slots(self, req_id: int, num_tokens: int) -> List[Tuple[int, int]]:
        """Grow the request to ``num_tokens`` tokens; returns copy-on-write (src, dst) pairs."""
        pairs = np.empty(2, dtype=np.int64)
        n = _i32()
        _check(_lib.pa_kvm_allocate_slots(self._h, req_id, num_tokens, pairs.ctypes.data, 1,
                                          ctypes.byref(n)), "pa_kvm_allocate_slots")
        return [(int(pairs[0]), int(pairs[1]))] if n.value else []

    def cache_blocks(self, req_id: int, tokens: Sequence[int], num_computed_tokens: int) -> None:
        t = _tok(tokens)
        _check(_lib.pa_kvm_cache_blocks(self._h, req_id, t.ctypes.data, num_computed_tokens),
               "pa_kvm_cache_blocks")

    def free(self, req_id: int) -> None:
        _check(_lib.pa_kvm_free(self._h, req_id), "pa_kvm_free")

    def fork(self, parent: int, child: int) -> None:
        _check(_lib.pa_kvm_fork(self._h, parent, child), "pa_kvm_fork")

    def block_table(self, req_id: int) -> List[int]:
        cap = self.num_blocks
        out = np.empty(cap, dtype=np.int32)
        n = _i32()
        _check(_lib.pa_kvm_block_table(self._h, req_id, out.ctypes.data, cap, ctypes.byref(n)),
               "pa_kvm_block_table")
        return out[:n.value].tolist()

    def slot_mapping(self, req_id: int, first_pos: int, count: int) -> np.ndarray:
        out = np.empty(max(count, 1), dtype=np.int64)
        _check(_lib.pa_kvm_slot_mapping(self._h, req_id, first_pos, count, out.ctypes.data),
               "pa_kvm_slot_mapping")
        return out[:count]

    @property
    def num_free_blocks(self) -> int:
        return int(_lib.pa_kvm_num_free_blocks(self._h))

    def stats(self) -> dict:
        out = np.zeros(5, dtype=np.int64)
        _check(_lib.pa_kvm_stats(self._h, out.ctypes.data), "pa_kvm_stats")
        return dict(zip(("lookups", "blocks_looked_up", "blocks_hit", "blocks_cached", "evictions"),
                        out.tolist()))
