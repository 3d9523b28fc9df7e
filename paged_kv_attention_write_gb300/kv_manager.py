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

__all__ = ["KVCacheManager", "Scheduler"]

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


# ----------------------------------------------------------------------------- step scheduler

class _Batch(ctypes.Structure):
    _fields_ = [("kind", _i32), ("num_seqs", _i32), ("num_tokens", _i32), ("max_query_len", _i32),
                ("max_context_len", _i32), ("table_width", _i32), ("num_copy_pairs", _i32)]


class _Offsets(ctypes.Structure):
    _fields_ = [(n, _i64) for n in ("query_start_loc", "context_lens", "block_tables", "slot_mapping",
                                    "copy_pairs", "token_ids", "positions", "dev_bytes", "req_ids",
                                    "total_bytes")]


_lib.pa_sched_create.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_vp)]
_lib.pa_sched_packed_bytes.argtypes = [_vp]
_lib.pa_sched_packed_bytes.restype = _i64
_lib.pa_sched_step_packed.argtypes = [_vp, ctypes.POINTER(_Batch), _vp, _i64, ctypes.POINTER(_Offsets)]
_lib.pa_sched_step_packed.restype = _i32
_lib.pa_sched_destroy.argtypes = [_vp]
_lib.pa_sched_destroy.restype = None
_lib.pa_sched_add_request.argtypes = [_vp, _i64, _vp, _i32, _i32]
_lib.pa_sched_step.argtypes = [_vp, ctypes.POINTER(_Batch), _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                               _i32, _i32, _i32]
_lib.pa_sched_complete.argtypes = [_vp, _vp, _i32, _vp, _i32, ctypes.POINTER(_i32)]
_lib.pa_sched_capacity.argtypes = [_vp, _vp]
_lib.pa_sched_stats.argtypes = [_vp, _vp]
_lib.pa_sched_manager.argtypes = [_vp]
_lib.pa_sched_manager.restype = _vp
for _n in ("pa_sched_create", "pa_sched_add_request", "pa_sched_step", "pa_sched_complete",
           "pa_sched_capacity", "pa_sched_stats"):
    getattr(_lib, _n).restype = _i32

KIND_NAMES = {0: "idle", 1: "prefill", 2: "decode"}


class Scheduler:
    """Step scheduler (``include/pa_scheduler.h``): prefill or decode batches under a token
    budget, prompts cut into chunks, at most ``max_decode_steps`` decode steps in a row while
    prompts wait.  ``step()`` returns the batch as numpy arrays (views of reused buffers)."""

    def __init__(self, num_blocks: int, block_size: int, token_budget: int = 4096,
                 chunk_tokens: int = 512, max_decode_steps: int = 8, prefix_cache: bool = True):
        h = _vp()
        _check(_lib.pa_sched_create(num_blocks, block_size, token_budget, chunk_tokens, max_decode_steps,
                                    1 if prefix_cache else 0, ctypes.byref(h)), "pa_sched_create")
        self._h = h
        self.block_size = block_size
        self._cap = None
        self._fin = None
        self._last_n = 0

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.pa_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_request(self, req_id: int, prompt, max_new_tokens: int) -> None:
        t = _tok(prompt)
        _check(_lib.pa_sched_add_request(self._h, req_id, t.ctypes.data, len(t), max_new_tokens),
               "pa_sched_add_request")
        self._cap = None

    def _buffers(self):
        cap = np.zeros(4, dtype=np.int32)
        _check(_lib.pa_sched_capacity(self._h, cap.ctypes.data), "pa_sched_capacity")
        if self._cap is None or any(cap > self._cap):
            c = np.maximum(cap, self._cap) if self._cap is not None else cap
            self._cap = c
            S, T, W, P = (int(x) for x in c)
            self._b = {"req_ids": np.zeros(S, np.int64), "qsl": np.zeros(S + 1, np.int32),
                       "context_lens": np.zeros(S, np.int32), "tables": np.zeros(S * W, np.int32),
                       "token_ids": np.zeros(T, np.int32), "positions": np.zeros(T, np.int32),
                       "slots": np.zeros(T, np.int64), "pairs": np.zeros(2 * P, np.int64),
                       "finished": np.zeros(S, np.int64)}
        return self._b, self._cap

    def step(self) -> dict:
        b, cap = self._buffers()
        out = _Batch()
        _check(_lib.pa_sched_step(self._h, ctypes.byref(out), b["req_ids"].ctypes.data, b["qsl"].ctypes.data,
                                  b["context_lens"].ctypes.data, b["tables"].ctypes.data, int(cap[2]),
                                  b["token_ids"].ctypes.data, b["positions"].ctypes.data,
                                  b["slots"].ctypes.data, b["pairs"].ctypes.data,
                                  int(cap[0]), int(cap[1]), int(cap[3])), "pa_sched_step")
        S, T, W = out.num_seqs, out.num_tokens, out.table_width
        self._last_n = S
        return {"kind": KIND_NAMES[out.kind], "num_seqs": S, "num_tokens": T,
                "max_query_len": out.max_query_len, "max_context_len": out.max_context_len,
                "req_ids": b["req_ids"][:S], "query_start_loc": b["qsl"][:S + 1],
                "context_lens": b["context_lens"][:S], "block_tables": b["tables"][:S * W].reshape(S, W),
                "token_ids": b["token_ids"][:T], "positions": b["positions"][:T],
                "slot_mapping": b["slots"][:T], "copy_pairs": b["pairs"][:2 * out.num_copy_pairs].reshape(-1, 2)}

    def packed_bytes(self) -> int:
        """Buffer bytes ``step_packed`` may need with the requests queued so far."""
        return int(_lib.pa_sched_packed_bytes(self._h))

    def step_packed(self, buf_ptr: int, buf_bytes: int):
        """Plan the next step into one host buffer (``pa_sched_step_packed``); returns the
        batch sizes and the byte offsets of its arrays (ctypes structures)."""
        b, o = _Batch(), _Offsets()
        _check(_lib.pa_sched_step_packed(self._h, ctypes.byref(b), buf_ptr, buf_bytes, ctypes.byref(o)),
               "pa_sched_step_packed")
        self._last_n = b.num_seqs
        return b, o

    def complete(self, sampled) -> list:
        t = _tok(sampled)
        ns = len(t)
        if self._fin is None or len(self._fin) < max(1, ns):  # finished ids: at most one per sequence
            self._fin = np.zeros(max(16, 2 * ns), dtype=np.int64)
        n = _i32()
        _check(_lib.pa_sched_complete(self._h, t.ctypes.data if ns else None, ns, self._fin.ctypes.data,
                                      len(self._fin), ctypes.byref(n)), "pa_sched_complete")
        return self._fin[:n.value].tolist()

    def stats(self) -> dict:
        out = np.zeros(7, dtype=np.int64)
        _check(_lib.pa_sched_stats(self._h, out.ctypes.data), "pa_sched_stats")
        return dict(zip(("prefill_steps", "decode_steps", "prefill_tokens", "generated_tokens", "finished",
                         "preemptions", "in_flight"), out.tolist()))

    def manager_stats(self) -> dict:
        out = np.zeros(5, dtype=np.int64)
        _check(_lib.pa_kvm_stats(_lib.pa_sched_manager(self._h), out.ctypes.data), "pa_kvm_stats")
        return dict(zip(("lookups", "blocks_looked_up", "blocks_hit", "blocks_cached", "evictions"),
                        out.tolist()))
