"""The host KV-cache manager driving the kernels end to end: requests that share a system
prompt reuse its cached blocks (their K/V are not written again), a forked request gets a
copy-on-write block through pa_copy_blocks, a finished request's cached blocks serve a
later one; every attention output equals dense attention over the request's whole token
history (the oracle), so any wrong sharing, copy or slot shows up.

K, V and q of a position are a function of the token prefix up to it (as in a model), so
equal prefixes give equal K/V and a prefix-cache hit is valid exactly when the prefixes
match."""
import zlib

import numpy as np
import pytest
import torch

from paged_steps import MAX_ABS, MEAN_ABS, assert_attention_close

pytestmark = pytest.mark.gpu

BS, NB, HKV, G, D = 16, 96, 2, 4, 128
HQ = HKV * G


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _rows(prefix, what, shape, dtype):
    h = zlib.crc32(np.asarray(prefix, dtype=np.int32).tobytes()) ^ zlib.crc32(what.encode())
    rng = np.random.default_rng(h)
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dtype)


class Session:
    def __init__(self, dtype):
        from paged_kv_attention_write_gb300.kv_manager import KVCacheManager
        self.dtype = dtype
        self.mgr = KVCacheManager(NB, BS)
        nan = float("nan")
        self.kc = torch.full((NB, BS, HKV, D), nan, dtype=dtype, device="cuda")
        self.vc = torch.full((NB, BS, HKV, D), nan, dtype=dtype, device="cuda")
        self.tokens = {}
        self.done = {}  # tokens whose K/V are in the cache

    def admit(self, rid, prompt):
        c = self.mgr.admit(rid, prompt)
        self.tokens[rid], self.done[rid] = list(prompt), c
        return c

    def fork(self, parent, child):
        self.mgr.fork(parent, child)
        self.tokens[child], self.done[child] = list(self.tokens[parent]), self.done[parent]

    def step(self, new_tokens, oracle):
        """new_tokens: rid -> tokens to append (empty: compute the rest of the prompt).
        Writes the K/V of every not-yet-computed position, runs attention for them and checks
        the outputs; returns the copy-on-write pairs applied."""
        import paged_kv_attention_write_gb300 as pa
        rids = list(new_tokens)
        pairs = []
        for r in rids:
            self.tokens[r] += list(new_tokens[r])
            pairs += self.mgr.allocate_slots(r, len(self.tokens[r]))
        if pairs:
            pa.pa_copy_blocks(self.kc, self.vc, torch.tensor(pairs, dtype=torch.int64, device="cuda"))
        ks, vs, qs, slots, qsl = [], [], [], [], [0]
        for r in rids:
            t, c = self.tokens[r], self.done[r]
            for p in range(c, len(t)):
                ks.append(_rows(t[:p + 1], "k", (HKV, D), self.dtype))
                vs.append(_rows(t[:p + 1], "v", (HKV, D), self.dtype))
                qs.append(_rows(t[:p + 1], "q", (HQ, D), self.dtype))
            slots.append(torch.from_numpy(self.mgr.slot_mapping(r, c, len(t) - c)))
            qsl.append(qsl[-1] + len(t) - c)
        dev = "cuda"
        pa.pa_reshape_and_cache(torch.stack(ks).to(dev), torch.stack(vs).to(dev), self.kc, self.vc,
                                torch.cat(slots).to(dev))
        q = torch.stack(qs).to(dev)
        tables = [self.mgr.block_table(r) for r in rids]
        width = max(len(b) for b in tables)
        bt = torch.tensor([b + [0] * (width - len(b)) for b in tables], dtype=torch.int32, device=dev)
        cl = torch.tensor([len(self.tokens[r]) for r in rids], dtype=torch.int32, device=dev)
        out = torch.empty((q.shape[0], HQ, D), dtype=torch.float32, device=dev)
        scale = 1.0 / D ** 0.5
        lq = [qsl[i + 1] - qsl[i] for i in range(len(rids))]
        if all(n == 1 for n in lq):
            ws = torch.empty(max(1, pa.pa_decode_workspace_size(len(rids), HQ, HKV, D, int(cl.max()))),
                             dtype=torch.uint8, device=dev)
            pa.pa_decode(out, q, self.kc, self.vc, bt, cl, int(cl.max()), scale, workspace=ws)
        else:
            pa.pa_prefill_chunk(out, q, torch.tensor(qsl, dtype=torch.int32, device=dev), max(lq),
                                self.kc, self.vc, bt, cl, int(cl.max()), scale)
        torch.cuda.synchronize()
        # oracle: dense attention over each request's whole history
        L = int(cl.max())
        kd = np.zeros((len(rids), HKV, L, D))
        vd = np.zeros((len(rids), HKV, L, D))
        for i, r in enumerate(rids):
            t = self.tokens[r]
            for p in range(len(t)):
                kd[i, :, p] = _rows(t[:p + 1], "k", (HKV, D), self.dtype).double().numpy()
                vd[i, :, p] = _rows(t[:p + 1], "v", (HKV, D), self.dtype).double().numpy()
        ref = oracle.dense_attention(q.cpu(), torch.tensor(qsl, dtype=torch.int32), kd, vd, cl.cpu(), scale)
        assert_attention_close(out.cpu(), ref, MAX_ABS, MEAN_ABS)
        for r in rids:
            self.done[r] = len(self.tokens[r])
            self.mgr.cache_blocks(r, self.tokens[r], self.done[r])
        return pairs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_manager_drives_kernels_with_prefix_sharing_fork_and_reuse(oracle_mod, dtype):
    rng = np.random.default_rng(3)
    sysp = rng.integers(0, 1000, size=40).tolist()           # shared system prompt (2 full blocks)
    r1 = sysp + rng.integers(0, 1000, size=30).tolist()
    r2 = sysp + rng.integers(0, 1000, size=25).tolist()
    r3 = sysp[:20] + rng.integers(0, 1000, size=37).tolist()
    s = Session(dtype)
    # request 1 alone: nothing cached yet
    assert s.admit(1, r1) == 0
    s.step({1: []}, oracle_mod)
    # requests 2 and 3 in one varlen prefill: 2 blocks and 1 block of the prompt are reused
    assert s.admit(2, r2) == 32 and s.admit(3, r3) == 16
    blocks_before = s.mgr.block_table(1)
    s.step({2: [], 3: []}, oracle_mod)
    assert s.mgr.block_table(2)[:2] == blocks_before[:2] and s.mgr.block_table(3)[:1] == blocks_before[:1]
    # three decode steps for all three
    for _ in range(3):
        s.step({r: [int(rng.integers(1000))] for r in (1, 2, 3)}, oracle_mod)
    # fork request 2 (its last block is partial): the first writer gets a copy-on-write block
    s.fork(2, 4)
    pairs = s.step({2: [7], 4: [8]}, oracle_mod)
    assert len(pairs) == 1 and pairs[0][0] != pairs[0][1]
    assert s.mgr.block_table(2)[-1] != s.mgr.block_table(4)[-1]
    # a prefill chunk and decode rows in one launch
    s.step({1: rng.integers(0, 1000, size=20).tolist(), 2: [9], 3: [10]}, oracle_mod)
    # request 1 finishes; request 5 repeats its history and reuses its (freed, cached) blocks
    hist = list(s.tokens[1])
    s.mgr.free(1)
    got = s.admit(5, hist + [11])
    assert got == (len(hist) // BS) * BS
    s.step({5: []}, oracle_mod)
    assert s.mgr.stats()["blocks_hit"] >= 3 + len(hist) // BS
