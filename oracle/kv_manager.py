"""Reference KV-cache block manager: the allocation policy written out plainly.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only the tests and the
benchmark's reference leg use it.  It shares no code with the library's C++
manager and restates the same policy in the plainest form: a Python list as the
free queue, a dict keyed by the exact token prefix as the prefix cache (no hashing),
per-block reference counts.

What it follows: the Pure-Rust engines page (paged-attention block management: the
manager finds a request's longest prefix-cache hit, allocates blocks for new tokens,
caches newly full blocks and frees a finished request's blocks; the block pool is flat
with an LRU free list; prefix-cache section: full blocks are registered and a lookup
walks the chain of full blocks to the longest hit) and the TensorSharp "Mistral 3"
page, section 11 (slot = blockId * blockSize + offset).  Where the pages leave a step
open, the readings are the ones stated in ``include/pa_kv_manager.h``:

* free queue: all blocks in id order at first; allocation takes from the head; a freed
  request returns its blocks to the tail, last block first;
* a lookup covers at most ``len(tokens) - 1`` tokens (the last token is always computed);
* a full block is registered unless another block already holds the same prefix; a
  cached block keeps its content while free and leaves the cache when it is handed out
  again; a lookup that hits a free cached block takes it out of the free queue;
* fork shares blocks; writing new tokens into a shared partial last block first
  replaces it by a copy (returned as a (src, dst) pair for the block copy).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple


class ReferenceKVManager:
    def __init__(self, num_blocks: int, block_size: int, prefix_cache: bool = True):
        self.bs = block_size
        self.prefix_cache = prefix_cache
        self.free_queue: List[int] = list(range(num_blocks))
        self.ref = [0] * num_blocks
        self.prefix_of: Dict[int, Tuple[int, ...]] = {}   # cached block -> its full token prefix
        self.cache: Dict[Tuple[int, ...], int] = {}        # full token prefix -> cached block
        self.requests: Dict[int, dict] = {}
        self.lookups = self.looked = self.hits = self.evictions = 0

    # -- the cache --------------------------------------------------------------------
    def _lookup(self, tokens: Sequence[int]) -> List[int]:
        self.lookups += 1
        if not self.prefix_cache or len(tokens) <= 1:
            return []
        n_blocks = (len(tokens) - 1) // self.bs
        self.looked += n_blocks
        hits = []
        for i in range(n_blocks):
            key = tuple(tokens[:(i + 1) * self.bs])
            if key not in self.cache:
                break
            hits.append(self.cache[key])
        self.hits += len(hits)
        return hits

    def peek_hits(self, tokens: Sequence[int]) -> List[int]:
        """The blocks a lookup would hit, without counting a lookup."""
        if not self.prefix_cache or len(tokens) <= 1:
            return []
        tokens = list(tokens)
        hits = []
        for i in range((len(tokens) - 1) // self.bs):
            key = tuple(tokens[:(i + 1) * self.bs])
            if key not in self.cache:
                break
            hits.append(self.cache[key])
        return hits

    def _take_head(self) -> int:
        b = self.free_queue.pop(0)
        if b in self.prefix_of:  # a cached block handed out again leaves the cache
            del self.cache[self.prefix_of.pop(b)]
            self.evictions += 1
        self.ref[b] = 1
        return b

    # -- the operations ---------------------------------------------------------------
    def get_computed_blocks(self, tokens: Sequence[int]) -> List[int]:
        return self._lookup(list(tokens))

    def admit(self, req_id: int, tokens: Sequence[int]) -> int:
        assert req_id not in self.requests
        hits = self._lookup(list(tokens))
        for b in hits:
            if self.ref[b] == 0:
                self.free_queue.remove(b)
            self.ref[b] += 1
        self.requests[req_id] = {"blocks": list(hits), "num_tokens": len(hits) * self.bs,
                                 "num_cached": len(hits)}
        return len(hits) * self.bs

    def allocate_slots(self, req_id: int, num_tokens: int) -> List[Tuple[int, int]]:
        r = self.requests[req_id]
        bs = self.bs
        want = -(-num_tokens // bs)
        grow = max(0, want - len(r["blocks"]))
        cow = (num_tokens > r["num_tokens"] and r["num_tokens"] % bs != 0 and r["blocks"]
               and self.ref[r["blocks"][-1]] > 1)
        if grow + (1 if cow else 0) > len(self.free_queue):
            raise MemoryError("not enough free blocks")
        pairs = []
        if cow:
            old = r["blocks"][-1]
            new = self._take_head()
            self.ref[old] -= 1
            r["blocks"][-1] = new
            pairs.append((old, new))
        for _ in range(grow):
            r["blocks"].append(self._take_head())
        r["num_tokens"] = max(r["num_tokens"], num_tokens)
        return pairs

    def cache_blocks(self, req_id: int, tokens: Sequence[int], num_computed_tokens: int) -> None:
        r = self.requests[req_id]
        tokens = list(tokens)
        full = num_computed_tokens // self.bs
        assert full <= len(r["blocks"])
        if self.prefix_cache:
            for i in range(r["num_cached"], full):
                key = tuple(tokens[:(i + 1) * self.bs])
                b = r["blocks"][i]
                if b not in self.prefix_of and key not in self.cache:
                    self.cache[key] = b
                    self.prefix_of[b] = key
        r["num_cached"] = max(r["num_cached"], full)

    def free(self, req_id: int) -> None:
        r = self.requests.pop(req_id)
        for b in reversed(r["blocks"]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free_queue.append(b)

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.requests and parent != child
        r = self.requests[parent]
        for b in r["blocks"]:
            self.ref[b] += 1
        self.requests[child] = {"blocks": list(r["blocks"]), "num_tokens": r["num_tokens"],
                                "num_cached": r["num_cached"]}

    def block_table(self, req_id: int) -> List[int]:
        return list(self.requests[req_id]["blocks"])

    def slot_mapping(self, req_id: int, first_pos: int, count: int) -> List[int]:
        bl = self.requests[req_id]["blocks"]
        return [bl[p // self.bs] * self.bs + p % self.bs for p in range(first_pos, first_pos + count)]

    @property
    def num_free_blocks(self) -> int:
        return len(self.free_queue)

    def stats(self) -> dict:
        return {"lookups": self.lookups, "blocks_looked_up": self.looked, "blocks_hit": self.hits,
                "blocks_cached": len(self.cache), "evictions": self.evictions}
