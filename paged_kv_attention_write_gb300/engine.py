"""Step loop over the scheduler and the paged-attention kernels.

``PagedAttentionEngine`` runs one scheduler step at a time (``include/pa_scheduler.h``:
prefill or decode batches under a token budget, chunked prompts, prefix caching): it moves
the step's batch description to the device in one copy, applies copy-on-write block copies,
writes the batch's fresh K/V into the paged cache and runs decode or chunked-prefill
attention.  The model side is supplied by the caller: ``qkv(step)`` returns the device
tensors q ``[T][Hq][D]``, k and v ``[T][Hkv][D]`` of the step's query tokens (``step`` holds
their token ids and positions), ``sample(step, out)`` returns one next token per sequence.
Marshalling only: every computation on the data runs in the library's kernels.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np
import torch

from . import pa_copy_blocks, pa_decode, pa_decode_workspace_size, pa_prefill_chunk, pa_reshape_and_cache
from .kv_manager import Scheduler

__all__ = ["PagedAttentionEngine"]


class PagedAttentionEngine:
    def __init__(self, num_blocks: int, block_size: int, num_heads: int, num_kv_heads: int,
                 head_dim: int, dtype: torch.dtype = torch.bfloat16, device="cuda",
                 token_budget: int = 4096, chunk_tokens: int = 512, max_decode_steps: int = 8,
                 prefix_cache: bool = True, scale: Optional[float] = None):
        self.sched = Scheduler(num_blocks, block_size, token_budget, chunk_tokens, max_decode_steps,
                               prefix_cache)
        self.dev = torch.device(device)
        self.Hq, self.Hkv, self.D, self.bs = num_heads, num_kv_heads, head_dim, block_size
        self.scale = scale if scale is not None else 1.0 / head_dim ** 0.5
        self.key_cache = torch.zeros((num_blocks, block_size, num_kv_heads, head_dim), dtype=dtype, device=self.dev)
        self.value_cache = torch.zeros_like(self.key_cache)
        self._pinned = None
        self._dev_buf = None
        self._copied = None   # event after the last copy out of the pinned buffer
        self._ws = None

    def add_request(self, req_id: int, prompt, max_new_tokens: int) -> None:
        self.sched.add_request(req_id, prompt, max_new_tokens)

    def _to_device(self, b: dict):
        """The step's int arrays in one pinned buffer, one host-to-device copy."""
        parts = [b["query_start_loc"], b["context_lens"], b["block_tables"].reshape(-1), b["slot_mapping"],
                 b["copy_pairs"].reshape(-1)]
        sizes = [p.nbytes for p in parts]
        need = sum((s + 15) // 16 * 16 for s in sizes)
        if self._copied is not None:   # the previous step's copy has left the pinned buffer
            self._copied.synchronize()
        if self._pinned is None or self._pinned.numel() < need:
            self._pinned = torch.empty(need * 2, dtype=torch.uint8, pin_memory=True)
            self._dev_buf = torch.empty(need * 2, dtype=torch.uint8, device=self.dev)
        host = self._pinned.numpy()
        offs, o = [], 0
        for p, s in zip(parts, sizes):
            host[o:o + s] = p.view(np.uint8).reshape(-1)
            offs.append(o)
            o += (s + 15) // 16 * 16
        self._dev_buf[:o].copy_(self._pinned[:o], non_blocking=True)
        if self._copied is None:
            self._copied = torch.cuda.Event()
        self._copied.record()
        out = []
        for p, off, s in zip(parts, offs, sizes):
            dt = {np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}[p.dtype]
            out.append(self._dev_buf[off:off + s].view(dt))
        return out

    def step(self, qkv: Callable, sample: Callable) -> Optional[dict]:
        """Run one scheduler step; returns the step (batch description and ``out``), or None
        when the scheduler is idle."""
        b = self.sched.step()
        if b["kind"] == "idle":
            return None
        S, W = b["num_seqs"], b["block_tables"].shape[1]
        qsl, cl, bt, slots, pairs = self._to_device(b)
        bt = bt.view(S, W)
        if b["copy_pairs"].size:
            pa_copy_blocks(self.key_cache, self.value_cache, pairs.view(-1, 2))
        q, k, v = qkv(b)
        pa_reshape_and_cache(k, v, self.key_cache, self.value_cache, slots)
        out = torch.empty((b["num_tokens"], self.Hq, self.D), dtype=torch.float32, device=self.dev)
        if b["kind"] == "decode":
            need = max(1, pa_decode_workspace_size(S, self.Hq, self.Hkv, self.D, b["max_context_len"]))
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(need * 2, dtype=torch.uint8, device=self.dev)
            pa_decode(out, q, self.key_cache, self.value_cache, bt, cl, b["max_context_len"], self.scale,
                      workspace=self._ws)
        else:
            pa_prefill_chunk(out, q, qsl, b["max_query_len"], self.key_cache, self.value_cache, bt, cl,
                             b["max_context_len"], self.scale)
        b["out"] = out
        self.sched.complete(sample(b, out))
        return b

    def run(self, qkv: Callable, sample: Callable, max_steps: int = 10 ** 7) -> int:
        """Steps until idle; returns the number of steps."""
        n = 0
        while n < max_steps and self.step(qkv, sample) is not None:
            n += 1
        return n
