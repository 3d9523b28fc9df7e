"""The scheduler + kernels step loop (PagedAttentionEngine) on a small serving workload:
shared system prompts (prefix-cache hits), prompts chunked under the token budget, decode
streaks, a pool small enough to force preemptions and recomputation.  Every step's attention
output is checked against dense attention over each request's whole history (the oracle).
K, V and q of a token are a function of the token and its position, so a prefix-cache hit
(equal tokens at equal positions) is valid."""
import numpy as np
import pytest
import torch

from paged_steps import MAX_ABS, MEAN_ABS, assert_attention_close

pytestmark = pytest.mark.gpu

HQ, HKV, D, R = 8, 2, 128, 4096


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


@pytest.mark.parametrize("bs,blocks,budget,chunk", [(16, 20, 512, 128), (32, 200, 4096, 512)])
def test_engine_steps_match_dense_attention(oracle_mod, bs, blocks, budget, chunk):
    from paged_kv_attention_write_gb300.engine import PagedAttentionEngine
    dtype = torch.bfloat16
    g = torch.Generator().manual_seed(bs)
    ktab = torch.randn((R, HKV, D), generator=g).to(dtype)
    vtab = torch.randn((R, HKV, D), generator=g).to(dtype)
    qtab = torch.randn((R, HQ, D), generator=g).to(dtype)
    dk, dv, dq = ktab.cuda(), vtab.cuda(), qtab.cuda()

    def idx(tok, pos):
        return (np.asarray(tok, dtype=np.int64) * 7919 + np.asarray(pos, dtype=np.int64) * 104729) % R

    def qkv(step):
        i = torch.from_numpy(idx(step["token_ids"], step["positions"])).cuda()
        return dq[i].contiguous(), dk[i].contiguous(), dv[i].contiguous()

    rng = np.random.default_rng(bs)
    tokens = {}
    systems = [rng.integers(0, 500, size=int(n)).tolist() for n in (40, 70)]
    eng = PagedAttentionEngine(blocks, bs, HQ, HKV, D, dtype, token_budget=budget, chunk_tokens=chunk,
                               max_decode_steps=3)
    for rid in range(10):
        p = systems[rid % 2] + rng.integers(0, 500, size=int(rng.integers(5, 150))).tolist()
        tokens[rid] = list(p)
        eng.add_request(rid, p, int(rng.integers(2, 30)))
    checked = {"prefill": 0, "decode": 0}

    def sample(step, out):
        torch.cuda.synchronize()
        S = step["num_seqs"]
        qsl, cl = step["query_start_loc"].copy(), step["context_lens"].copy()
        L = int(cl.max())
        kd = np.zeros((S, HKV, L, D))
        vd = np.zeros((S, HKV, L, D))
        for i, rid in enumerate(step["req_ids"].tolist()):
            t = tokens[rid]
            j = idx(t[:cl[i]], np.arange(cl[i]))
            kd[i, :, :cl[i]] = ktab[torch.from_numpy(j)].double().numpy().transpose(1, 0, 2)
            vd[i, :, :cl[i]] = vtab[torch.from_numpy(j)].double().numpy().transpose(1, 0, 2)
        q = qtab[torch.from_numpy(idx(step["token_ids"], step["positions"]))]
        ref = oracle_mod.dense_attention(q, torch.from_numpy(qsl), kd, vd, torch.from_numpy(cl), eng.scale)
        assert_attention_close(out.cpu(), ref, MAX_ABS, MEAN_ABS)
        checked[step["kind"]] += 1
        nxt = rng.integers(0, 500, size=S).tolist()
        for rid, t in zip(step["req_ids"].tolist(), nxt):
            tokens[rid].append(int(t))   # kept only when the step ends the request's prompt or decodes
        return nxt

    # sample() appends a token for every sequence; a prefill chunk that does not end its prompt
    # must not keep it: undo those after each step
    while True:
        st = eng.step(qkv, lambda s, o: sample(s, o))
        if st is None:
            break
        if st["kind"] == "prefill":
            for i, rid in enumerate(st["req_ids"].tolist()):
                if rid in tokens and st["context_lens"][i] < len(tokens[rid]) - 1:
                    tokens[rid].pop()
    s = eng.sched.stats()
    assert s["finished"] == 10 and checked["prefill"] > 0 and checked["decode"] > 0
    if blocks == 20:  # staggered admissions: shared prompts are cached, the pool overflows
        assert s["preemptions"] > 0 and eng.sched.manager_stats()["blocks_hit"] > 0
