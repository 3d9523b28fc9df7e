"""Reference step scheduler over the reference KV-cache manager.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It restates, in plain Python, the
batch policy the library's C++ scheduler implements, so that the two can be compared step
by step.  What it follows: the Pure-Rust engines page, scheduling section (mistral.rs):
every step is either a prefill batch or a decode batch, never both; with prompts that can be
admitted, a prefill may be inserted after decode steps and at most 8 decode steps run in a
row (DEFAULT_MAX_DECODE_STEPS_BEFORE_PREFILL); a prefill batch holds at most 4096 tokens
(DEFAULT_MAX_NUM_BATCHED_TOKENS) and a long prompt is cut into chunks of at most 512 tokens
(DEFAULT_MAX_PREFILL_CHUNK_TOKENS).  Readings where the page leaves a step open (also stated
in ``include/pa_scheduler.h``):

* the step decision: nothing running -> prefill (or idle); prefill work pending and 8
  decode steps in a row -> prefill; otherwise decode when something runs;
* a prefill batch first continues the prompts already being prefilled (in admission order),
  then admits waiting requests in arrival order while the token budget and the free blocks
  allow; each prompt contributes at most one chunk per step;
* a request's last prompt chunk yields its first generated token; each decode step computes
  the newest token of every running request and yields its next token;
* a request that has generated its maximum number of tokens is freed at once;
* when a decode step cannot get a block, the most recently admitted running request is
  preempted (its blocks freed, its tokens so far re-queued at the head of the waiting queue
  as its new prompt) until the allocation succeeds; likewise, when the next chunk of a prompt
  being prefilled cannot get its blocks, the most recently admitted prompt being prefilled
  is preempted until the chunk fits (or that prompt itself was preempted), so that prompts
  holding blocks can never block each other.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List

from .kv_manager import ReferenceKVManager


class ReferenceScheduler:
    def __init__(self, num_blocks: int, block_size: int, budget: int = 4096, chunk: int = 512,
                 max_decode_steps: int = 8, prefix_cache: bool = True):
        self.kv = ReferenceKVManager(num_blocks, block_size, prefix_cache)
        self.bs, self.budget, self.chunk, self.max_decode = block_size, budget, chunk, max_decode_steps
        self.req: Dict[int, dict] = {}
        self.waiting = deque()
        self.prefilling: List[int] = []
        self.running: List[int] = []
        self.decode_streak = 0
        self.last = None
        self.counters = {"prefill_steps": 0, "decode_steps": 0, "prefill_tokens": 0,
                         "generated_tokens": 0, "finished": 0, "preemptions": 0}

    def add_request(self, rid: int, prompt, max_new_tokens: int) -> None:
        assert rid not in self.req and len(prompt) > 0 and max_new_tokens > 0
        if -(-(len(prompt) + max_new_tokens) // self.bs) > len(self.kv.ref):
            raise ValueError("the request can never fit the pool")
        self.req[rid] = {"tokens": list(prompt), "prompt_len": len(prompt), "computed": 0,
                         "max_new": max_new_tokens, "generated": 0}
        self.waiting.append(rid)

    # -- the step decision --------------------------------------------------------------
    def _admissible(self, rid: int, left: int):
        """(hit tokens, chunk) if waiting request rid's first chunk fits the free blocks
        (those not taken by its own hits), else None.  Changes nothing."""
        r = self.req[rid]
        hits = self.kv.peek_hits(r["tokens"])
        got = len(hits) * self.bs
        n = min(self.chunk, len(r["tokens"]) - got, left)
        need = -(-(got + n) // self.bs) - len(hits)
        free_hits = sum(1 for b in hits if self.kv.ref[b] == 0)
        return (got, n) if need <= self.kv.num_free_blocks - free_hits else None

    def step(self) -> dict:
        pending = bool(self.prefilling) or bool(self.waiting)
        batch = None
        if pending and (not self.running or self.decode_streak >= self.max_decode):
            batch = self._prefill_batch()
            if not batch["seqs"]:
                batch = None               # nothing fits: decode (or idle) instead
        if batch is None:
            batch = self._decode_batch() if self.running else {"kind": "idle", "seqs": [], "pairs": []}
        self.last = batch
        return batch

    def _entry(self, rid, start, count):
        r = self.req[rid]
        return {"req": rid, "start": start, "count": count, "context": start + count,
                "tokens": r["tokens"][start:start + count],
                "table": self.kv.block_table(rid),
                "slots": self.kv.slot_mapping(rid, start, count)}

    def _prefill_batch(self) -> dict:
        left = self.budget
        seqs, pairs = [], []
        for rid in list(self.prefilling):   # prompts already being prefilled, in order
            if left == 0:
                break
            if rid not in self.prefilling:    # preempted below for an earlier prompt
                continue
            r = self.req[rid]
            n = min(self.chunk, r["prompt_len"] - r["computed"], left)
            while True:
                try:
                    pairs += self.kv.allocate_slots(rid, r["computed"] + n)
                    break
                except MemoryError:             # the most recently admitted prompt makes room
                    victim = self.prefilling.pop()
                    self._preempt(victim)
                    if victim == rid:
                        break
            if rid not in self.prefilling:
                continue
            seqs.append(self._entry(rid, r["computed"], n))
            left -= n
        while self.waiting and left > 0:    # then new prompts, in arrival order
            rid = self.waiting[0]
            fit = self._admissible(rid, left)
            if fit is None:
                break
            got, n = fit
            r = self.req[rid]
            assert self.kv.admit(rid, r["tokens"]) == got
            pairs += self.kv.allocate_slots(rid, got + n)
            self.waiting.popleft()
            r["computed"] = got
            r["prompt_len"] = len(r["tokens"])
            self.prefilling.append(rid)
            seqs.append(self._entry(rid, got, n))
            left -= n
        return {"kind": "prefill", "seqs": seqs, "pairs": pairs}

    def _decode_batch(self) -> dict:
        pairs = []
        i = 0
        while i < len(self.running):
            rid = self.running[i]
            try:
                pairs += self.kv.allocate_slots(rid, len(self.req[rid]["tokens"]))
                i += 1
            except MemoryError:
                self._preempt(self.running.pop())   # the most recently admitted request
        seqs = [self._entry(rid, len(self.req[rid]["tokens"]) - 1, 1) for rid in self.running]
        return {"kind": "decode", "seqs": seqs, "pairs": pairs}

    def _preempt(self, rid: int) -> None:
        r = self.req[rid]
        self.kv.free(rid)
        r["computed"] = 0
        r["prompt_len"] = len(r["tokens"])
        self.waiting.appendleft(rid)
        self.counters["preemptions"] += 1

    # -- completing a step --------------------------------------------------------------
    def complete(self, sampled) -> List[int]:
        """Apply a step: one sampled token per sequence of the last batch (ignored for a
        prefill chunk that is not the prompt's last).  Returns the requests finished."""
        b = self.last
        finished = []
        if b["kind"] == "prefill":
            self.counters["prefill_steps"] += 1
            self.decode_streak = 0
        elif b["kind"] == "decode":
            self.counters["decode_steps"] += 1
            self.decode_streak += 1
        for e, tok in zip(b["seqs"], sampled):
            rid = e["req"]
            r = self.req[rid]
            done = e["start"] + e["count"]
            r["computed"] = done
            self.kv.cache_blocks(rid, r["tokens"], done)
            if b["kind"] == "prefill":
                self.counters["prefill_tokens"] += e["count"]
                if done < r["prompt_len"]:
                    continue
                self.prefilling.remove(rid)
                self.running.append(rid)
            r["tokens"].append(int(tok))
            r["generated"] += 1
            self.counters["generated_tokens"] += 1
            if r["generated"] >= r["max_new"]:
                self.running.remove(rid)
                self.kv.free(rid)
                del self.req[rid]
                self.counters["finished"] += 1
                finished.append(rid)
        self.last = None
        return finished
