"""Seeded synthetic inputs for paged attention over a block-tabled KV cache.

Shared by the tests, the benchmark and the smoke check: both the CUDA library
and the CPU oracle consume what this module returns, and it holds none of the
attention arithmetic.  It only draws random numbers (numpy PCG64, so the
stream is the same on every machine), shuffles block ids into block tables the
way a block pool hands them out, and writes slot numbers
``block_id * block_size + offset`` for the fresh tokens, as a scheduler does
(TensorSharp "Mistral 3" page, section 11, slot-mapping scatter).

Recipe (all host tensors; the caller moves them to the GPU):

* q, fresh k/v and every cached k/v element ~ N(0, 1), drawn in fp32 and
  rounded to the cache dtype;
* the block pool is ``[NB][bs][Hkv][D]`` per K and per V; each sequence gets
  ``ceil(context_len / bs)`` blocks taken in order from a seeded random
  permutation of the pool, with ``free_frac`` of the pool left as free blocks
  interleaved at random;
* every slot that holds no cached token (free blocks, block tails past the
  context, and the slots the step is about to write) is NaN, so a stray read
  or a missed write shows up in the output or in a bitwise pool comparison;
* block tables are int32 ``[S][max_blocks]`` padded with -1.

The named workloads follow the five configurations the library is measured
on (decode: one fresh token per sequence written, then attended).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

__all__ = [
    "PagedCase", "make_decode_case", "make_prefill_case", "tiny_decode", "decode_batch",
    "long_decode", "prefill_chunk", "stress_decode", "mixed_batch", "gqa_decode", "WORKLOADS",
]


@dataclass
class PagedCase:
    """One step's inputs.  Tensors are CPU tensors; see the module docstring."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    scale: float
    key_cache: torch.Tensor          # [NB][bs][Hkv][D]
    value_cache: torch.Tensor        # [NB][bs][Hkv][D]
    block_tables: torch.Tensor       # int32 [S][max_blocks]
    context_lens: torch.Tensor       # int32 [S], fresh tokens included
    cached_lens: np.ndarray          # tokens already in the pool before the step
    query: torch.Tensor              # [Tq][Hq][D]
    query_start_loc: torch.Tensor    # int32 [S+1]
    new_key: torch.Tensor            # [T][Hkv][D]
    new_value: torch.Tensor          # [T][Hkv][D]
    slot_mapping: torch.Tensor       # int64 [T]
    block_mapping: Optional[torch.Tensor] = None  # int64 [N][2] (src, dst), or None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.key_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def is_decode(self) -> bool:
        return int(self.query.shape[0]) == self.num_seqs and bool(
            (self.query_start_loc[1:] - self.query_start_loc[:-1] == 1).all())

    def kv_elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()


def _normal(rng: np.random.Generator, shape, dtype: torch.dtype, chunk: int = 1 << 24) -> torch.Tensor:
    """N(0,1) samples drawn in fp32 chunks and rounded to ``dtype``."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        flat[s:e] = torch.from_numpy(rng.standard_normal(e - s, dtype=np.float32))
    return out


def _fill_pool(rng, NB, bs, Hkv, D, dtype, bt, cached_lens):
    """Random pool whose only non-NaN slots are the cached tokens of the block tables."""
    kc = _normal(rng, (NB, bs, Hkv, D), dtype)
    vc = _normal(rng, (NB, bs, Hkv, D), dtype)
    valid = np.zeros((NB, bs), dtype=bool)
    for s, L in enumerate(cached_lens):
        nfull, rem = divmod(int(L), bs)
        ids = bt[s, :nfull]
        valid[ids, :] = True
        if rem:
            valid[bt[s, nfull], :rem] = True
    invalid = torch.from_numpy(~valid)
    kc[invalid] = float("nan")
    vc[invalid] = float("nan")
    return kc, vc


def _block_tables(rng, need_blocks, NB, max_blocks=None):
    """Hand out ``need_blocks[s]`` block ids per sequence from a shuffled pool of NB."""
    total = int(sum(need_blocks))
    assert total <= NB, "pool too small"
    perm = rng.permutation(NB)
    used = np.sort(rng.choice(NB, size=total, replace=False)) if total < NB else np.arange(NB)
    ids = perm[used]  # `total` distinct ids, shuffled, with the free ones interleaved
    mb = max_blocks or max(1, max(need_blocks) if len(need_blocks) else 1)
    bt = np.full((len(need_blocks), mb), -1, dtype=np.int32)
    o = 0
    for s, n in enumerate(need_blocks):
        bt[s, :n] = ids[o:o + n]
        o += n
    return bt


def _slots(bt, positions_per_seq, bs):
    out = []
    for s, pos in enumerate(positions_per_seq):
        for p in pos:
            out.append(int(bt[s, p // bs]) * bs + p % bs)
    return np.asarray(out, dtype=np.int64)


def make_decode_case(name: str, cached_lens, block_size: int, num_heads: int, num_kv_heads: int,
                     head_dim: int, dtype: torch.dtype, seed: int, num_blocks: Optional[int] = None,
                     free_frac: float = 0.0, share_frac: float = 0.0,
                     alias_frac: float = 0.0) -> PagedCase:
    """Decode step: one fresh token per sequence is written at position L, then attended.

    ``share_frac`` of the sequences receive the leading full blocks of a donor
    sequence through a block copy (``block_mapping``); ``alias_frac`` of them
    instead point their block tables at the donor's physical blocks
    (read-only sharing of a cached prefix).
    """
    rng = np.random.default_rng(seed)
    L = np.asarray(cached_lens, dtype=np.int64)
    S, bs, Hkv, D = len(L), block_size, num_kv_heads, head_dim
    need = [int(math.ceil((int(l) + 1) / bs)) for l in L]
    total = sum(need)
    NB = num_blocks or int(math.ceil(total / (1.0 - free_frac)))
    bt = _block_tables(rng, need, NB)

    block_mapping = None
    aliased = []
    if share_frac > 0 or alias_frac > 0:
        order = rng.permutation(S)
        n_share = int(round(share_frac * S))
        n_alias = int(round(alias_frac * S))
        recipients = order[:n_share + n_alias]
        donors_pool = order[n_share + n_alias:]
        pairs = []
        for i, r in enumerate(recipients):
            d = int(donors_pool[rng.integers(len(donors_pool))])
            k = int(min(L[r], L[d]) // bs)
            if i < n_share:
                pairs += [(int(bt[d, b]), int(bt[r, b])) for b in range(k)]
            else:  # alias: share the donor's physical blocks, free the recipient's own
                bt[r, :k] = bt[d, :k]
                aliased.append(int(r))
        if pairs:
            block_mapping = torch.tensor(pairs, dtype=torch.int64).view(-1, 2)

    kc, vc = _fill_pool(rng, NB, bs, Hkv, D, dtype, bt, L)
    query = _normal(rng, (S, num_heads, D), dtype)
    new_k = _normal(rng, (S, Hkv, D), dtype)
    new_v = _normal(rng, (S, Hkv, D), dtype)
    slots = _slots(bt, [[int(l)] for l in L], bs)
    return PagedCase(
        name=name, num_heads=num_heads, num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dtype,
        scale=float(np.float32(1.0 / math.sqrt(D))), key_cache=kc, value_cache=vc,
        block_tables=torch.from_numpy(bt), context_lens=torch.from_numpy((L + 1).astype(np.int32)),
        cached_lens=L, query=query,
        query_start_loc=torch.arange(S + 1, dtype=torch.int32),
        new_key=new_k, new_value=new_v, slot_mapping=torch.from_numpy(slots),
        block_mapping=block_mapping, meta={"seed": seed, "aliased": aliased, "free_frac": free_frac})


def make_prefill_case(name: str, prefix_lens, chunk_lens, block_size: int, num_heads: int,
                      num_kv_heads: int, head_dim: int, dtype: torch.dtype, seed: int,
                      free_frac: float = 0.0) -> PagedCase:
    """Chunked prefill: each sequence's chunk K/V go to their slots, then the chunk attends
    causally within itself and fully over its cached prefix."""
    rng = np.random.default_rng(seed)
    P = np.asarray(prefix_lens, dtype=np.int64)
    Q = np.asarray(chunk_lens, dtype=np.int64)
    S, bs, Hkv, D = len(P), block_size, num_kv_heads, head_dim
    C = P + Q
    need = [int(math.ceil(int(c) / bs)) for c in C]
    NB = int(math.ceil(sum(need) / (1.0 - free_frac)))
    bt = _block_tables(rng, need, NB)
    kc, vc = _fill_pool(rng, NB, bs, Hkv, D, dtype, bt, P)
    Tq = int(Q.sum())
    query = _normal(rng, (Tq, num_heads, D), dtype)
    new_k = _normal(rng, (Tq, Hkv, D), dtype)
    new_v = _normal(rng, (Tq, Hkv, D), dtype)
    slots = _slots(bt, [range(int(p), int(c)) for p, c in zip(P, C)], bs)
    qsl = np.concatenate([[0], np.cumsum(Q)]).astype(np.int32)
    return PagedCase(
        name=name, num_heads=num_heads, num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dtype,
        scale=float(np.float32(1.0 / math.sqrt(D))), key_cache=kc, value_cache=vc,
        block_tables=torch.from_numpy(bt), context_lens=torch.from_numpy(C.astype(np.int32)),
        cached_lens=P, query=query, query_start_loc=torch.from_numpy(qsl),
        new_key=new_k, new_value=new_v, slot_mapping=torch.from_numpy(slots),
        meta={"seed": seed, "prefix_lens": P.tolist(), "chunk_lens": Q.tolist()})


# --- the five named workloads ------------------------------------------------------------

def tiny_decode(seed: int = 1) -> PagedCase:
    """2 sequences with cached lengths 37 and 70, block 8, 4 q / 2 kv heads, D 64, fp32,
    a 24-block pool assigned by a seeded permutation."""
    return make_decode_case("tiny-decode S2 L37/70 bs8 Hq4 Hkv2 D64 fp32", [37, 70], 8, 4, 2, 64,
                            torch.float32, seed, num_blocks=24)


def decode_batch(seed: int = 2) -> PagedCase:
    """32 sequences, cached lengths uniform in [512, 4096], block 32, 32 q / 8 kv heads, D 128,
    bf16, pool sized to the tokens and shuffled."""
    rng = np.random.default_rng(1000 + seed)
    L = rng.integers(512, 4096, size=32, endpoint=True)
    return make_decode_case("decode-batch S32 L512-4096 bs32 Hq32 Hkv8 D128 bf16", L, 32, 32, 8,
                            128, torch.bfloat16, seed)


def long_decode(seed: int = 3) -> PagedCase:
    """8 sequences, cached lengths uniform in [16384, 32768], block 32, 32 q / 8 kv heads,
    D 128, bf16, shuffled pool (split-K over the context plus the log-sum-exp reduce)."""
    rng = np.random.default_rng(1000 + seed)
    L = rng.integers(16384, 32768, size=8, endpoint=True)
    return make_decode_case("long-decode S8 L16K-32K bs32 Hq32 Hkv8 D128 bf16", L, 32, 32, 8, 128,
                            torch.bfloat16, seed)


def prefill_chunk(seed: int = 4) -> PagedCase:
    """4 sequences, a 512-token chunk each on top of cached prefixes 0/1024/2048/3584,
    block 16, 32 q / 8 kv heads, D 128, bf16."""
    return make_prefill_case("prefill-chunk S4 Q512 prefix0/1K/2K/3.5K bs16 Hq32 Hkv8 D128 bf16",
                             [0, 1024, 2048, 3584], [512] * 4, 16, 32, 8, 128, torch.bfloat16, seed)


def gqa_decode(group: int = 8, seed: int = 7) -> PagedCase:
    """The long-context shape with `group` query heads per kv head (8 kv heads): 8 sequences,
    cached lengths uniform in [16384, 32768], block 32, D 128, bf16.  Eight query heads per kv
    head is the grouping of the larger GQA models."""
    rng = np.random.default_rng(1000 + seed)
    L = rng.integers(16384, 32768, size=8, endpoint=True)
    return make_decode_case(f"gqa-decode S8 L16K-32K bs32 Hq{8 * group} Hkv8 D128 bf16", L, 32, 8 * group, 8,
                            128, torch.bfloat16, seed)


def stress_decode(block_size: int = 16, dtype: torch.dtype = torch.bfloat16, seed: int = 5,
                  num_seqs: int = 256) -> PagedCase:
    """256 sequences, cached lengths log-uniform in [64, 8192], 32 q / 8 kv heads, D 128;
    10% of the sequences take a donor's leading blocks through a block copy; 20% of the
    pool is free blocks interleaved."""
    rng = np.random.default_rng(1000 + seed)
    L = np.floor(np.exp(rng.uniform(math.log(64), math.log(8192), size=num_seqs))).astype(np.int64)
    tag = {torch.bfloat16: "bf16", torch.float16: "fp16"}[dtype]
    return make_decode_case(f"stress S{num_seqs} L64-8192 bs{block_size} Hq32 Hkv8 D128 {tag}", L,
                            block_size, 32, 8, 128, dtype, seed * 100 + block_size,
                            free_frac=0.2, share_frac=0.1)


def mixed_batch(seed: int = 6) -> PagedCase:
    """One mixed step in the vLLM v1 manner (Pure-Rust engines page, scheduling section:
    prefill chunks and decode tokens share one batch under a token budget): 28 decode rows
    (one new token on cached lengths uniform in [512, 4096]) followed by the four 512-token
    chunks of the chunked-prefill workload; block 16, 32 q / 8 kv heads, D 128, bf16."""
    rng = np.random.default_rng(1000 + seed)
    dec = rng.integers(512, 4096, size=28, endpoint=True).tolist()
    prefix = dec + [0, 1024, 2048, 3584]
    chunk = [1] * 28 + [512] * 4
    return make_prefill_case("mixed S32 28 decode rows L512-4096 + 4 chunks Q512 bs16 Hq32 Hkv8 D128 bf16",
                             prefix, chunk, 16, 32, 8, 128, torch.bfloat16, seed)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "decode_batch": decode_batch,
    "long_decode": long_decode,
    "prefill_chunk": prefill_chunk,
    "stress_decode": stress_decode,
    "mixed_batch": mixed_batch,
    "gqa_decode": gqa_decode,
}
