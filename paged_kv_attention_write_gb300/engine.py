"""Step loop over the scheduler and the paged-attention kernels.

``PagedAttentionEngine`` runs one scheduler step at a time (``include/pa_scheduler.h``:
prefill or decode batches under a token budget, chunked prompts, prefix caching).  Per step
the C++ scheduler writes the whole batch description into one pinned host buffer
(``pa_sched_step_packed``), its device part goes over in one asynchronous copy
(``pa_engine_upload``), and one more call (``pa_engine_attend``) enqueues the step's
copy-on-write block copies, the fresh K/V written into the paged cache and decode or
chunked-prefill attention, reading the batch from that copy.  The model
side is supplied by the caller: ``qkv(step)`` returns the device tensors q ``[T][Hq][D]``, k and
v ``[T][Hkv][D]`` of the step's query tokens (``step`` holds their token ids and positions, on
the host and, through ``device_tokens``, on the device), ``sample(step, out)`` returns one next
token per sequence.  Marshalling only: every computation on the data runs in the library's
kernels.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np
import torch

import ctypes

from . import _DTYPES, _check, _lib, pa_decode_workspace_size
from .kv_manager import KIND_NAMES, Scheduler, _Batch, _Offsets


class _Cache(ctypes.Structure):
    _fields_ = [("key_cache", ctypes.c_void_p), ("value_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("scale", ctypes.c_float)]


_lib.pa_engine_upload.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Offsets), ctypes.c_void_p]
_lib.pa_engine_upload.restype = ctypes.c_int
_lib.pa_engine_attend.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Batch), ctypes.POINTER(_Offsets),
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p, ctypes.c_void_p]
_lib.pa_engine_attend.restype = ctypes.c_int

__all__ = ["PagedAttentionEngine"]

_PA_F32 = 0


class PagedAttentionEngine:
    def __init__(self, num_blocks: int, block_size: int, num_heads: int, num_kv_heads: int,
                 head_dim: int, dtype: torch.dtype = torch.bfloat16, device="cuda",
                 token_budget: int = 4096, chunk_tokens: int = 512, max_decode_steps: int = 8,
                 prefix_cache: bool = True, scale: Optional[float] = None):
        self.sched = Scheduler(num_blocks, block_size, token_budget, chunk_tokens, max_decode_steps,
                               prefix_cache)
        self.dev = torch.device(device)
        self.Hq, self.Hkv, self.D, self.bs = num_heads, num_kv_heads, head_dim, block_size
        self.NB = num_blocks
        self.scale = scale if scale is not None else 1.0 / head_dim ** 0.5
        self.dtype_code = _DTYPES[dtype]
        self.key_cache = torch.zeros((num_blocks, block_size, num_kv_heads, head_dim), dtype=dtype, device=self.dev)
        self.value_cache = torch.zeros_like(self.key_cache)
        self._cache = _Cache(self.key_cache.data_ptr(), self.value_cache.data_ptr(), num_blocks, block_size,
                             num_heads, num_kv_heads, head_dim, self.dtype_code, self.scale)
        # two pinned staging buffers used in turn, each with the event of its last copy out
        self._pinned = [None, None]
        self._pinned_np = [None, None]  # numpy views of the same memory
        self._events = [None, None]
        self._turn = 0
        self._dev_buf = None
        self._out = None
        self._ws = None
        self._need = None

    def add_request(self, req_id: int, prompt, max_new_tokens: int) -> None:
        self.sched.add_request(req_id, prompt, max_new_tokens)
        self._need = None  # the packed step may grow

    def _buffers(self):
        """The next pinned staging buffer (free once its previous copy has left it) and the
        device buffer, grown to the scheduler's packed size."""
        if self._need is None:
            self._need = self.sched.packed_bytes()
        need = self._need
        i = self._turn
        self._turn ^= 1
        if self._events[i] is not None:
            self._events[i].synchronize()
        if self._pinned[i] is None or self._pinned[i].numel() < need:
            self._pinned[i] = torch.empty(2 * need, dtype=torch.uint8, pin_memory=True)
            self._pinned_np[i] = self._pinned[i].numpy()
        if self._dev_buf is None or self._dev_buf.numel() < need:
            self._dev_buf = torch.empty(2 * need, dtype=torch.uint8, device=self.dev)
        return i

    def device_tokens(self, step: dict):
        """The step's token ids and positions as int32 device tensors (views of the copy)."""
        o, T = step["_offsets"], step["num_tokens"]
        buf = self._dev_buf
        tok = buf[o.token_ids:o.token_ids + 4 * T].view(torch.int32)
        pos = buf[o.positions:o.positions + 4 * T].view(torch.int32)
        return tok, pos

    def step(self, qkv: Callable, sample: Callable) -> Optional[dict]:
        """Run one scheduler step; returns the step (batch description and ``out``), or None
        when the scheduler is idle.  The step's host arrays are views of the staging buffer and
        ``out`` a view of the engine's output buffer: both stay valid until the next step."""
        i = self._buffers()
        host = self._pinned[i]
        b, o = self.sched.step_packed(host.data_ptr(), host.numel())
        if b.kind == 0:
            self.sched.complete([])  # close the idle step: requests added later can run
            return None
        S, T = b.num_seqs, b.num_tokens
        cur = torch.cuda.current_stream(self.dev)
        stream = cur.cuda_stream
        _check(_lib.pa_engine_upload(self._dev_buf.data_ptr(), host.data_ptr(), ctypes.byref(o), stream),
               "pa_engine_upload")
        if self._events[i] is None:
            self._events[i] = torch.cuda.Event()
        self._events[i].record(cur)
        hb = self._pinned_np[i]
        step = {"kind": KIND_NAMES[b.kind], "num_seqs": S, "num_tokens": T,
                "max_query_len": b.max_query_len, "max_context_len": b.max_context_len,
                "req_ids": np.frombuffer(hb, np.int64, S, o.req_ids),
                "query_start_loc": np.frombuffer(hb, np.int32, S + 1, o.query_start_loc),
                "context_lens": np.frombuffer(hb, np.int32, S, o.context_lens),
                "token_ids": np.frombuffer(hb, np.int32, T, o.token_ids),
                "positions": np.frombuffer(hb, np.int32, T, o.positions),
                "_offsets": o}
        q, k, v = qkv(step)
        if self._out is None or self._out.shape[0] < T:
            self._out = torch.empty((max(T, 2 * (0 if self._out is None else self._out.shape[0])), self.Hq, self.D),
                                    dtype=torch.float32, device=self.dev)
        out = self._out[:T]
        ws, ws_bytes = None, 0
        if b.kind == 2:  # decode: a workspace for the split of the contexts
            need = max(1, pa_decode_workspace_size(S, self.Hq, self.Hkv, self.D, b.max_context_len))
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(need * 2, dtype=torch.uint8, device=self.dev)
            ws, ws_bytes = self._ws.data_ptr(), self._ws.numel()
        _check(_lib.pa_engine_attend(ctypes.byref(self._cache), ctypes.byref(b), ctypes.byref(o),
                                     self._dev_buf.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     out.data_ptr(), _PA_F32, ws, ws_bytes, None, stream), "pa_engine_attend")
        step["out"] = out
        self.sched.complete(sample(step, out))
        return step

    def run(self, qkv: Callable, sample: Callable, max_steps: int = 10 ** 7) -> int:
        """Steps until idle; returns the number of steps."""
        n = 0
        while n < max_steps and self.step(qkv, sample) is not None:
            n += 1
        return n
