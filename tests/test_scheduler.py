"""Step scheduler: the reference policy pinned by hand-worked cases, and the C++ scheduler
(through its C ABI) equal to the reference batch by batch on seeded workloads with shared
prompts, chunked prefill, decode streaks and preemptions."""
import numpy as np
import pytest

from oracle.scheduler import ReferenceScheduler


@pytest.fixture(scope="module")
def cpp_cls(pa_lib_path):
    from paged_kv_attention_write_gb300.kv_manager import Scheduler
    return Scheduler


def _drain(s, rng, limit=100000):
    trace = []
    for _ in range(limit):
        b = s.step()
        if b["kind"] == "idle":
            return trace
        trace.append((b["kind"], [(e["req"], e["start"], e["count"]) for e in b["seqs"]]))
        s.complete([int(rng.integers(1000)) for _ in b["seqs"]])
    raise AssertionError("no idle step")


# ----------------------------------------------------------------------------- pins of the reference

def test_chunks_fill_the_token_budget_in_order():
    s = ReferenceScheduler(256, 16, budget=1024, chunk=512)
    s.add_request(0, list(range(1000)), 2)
    s.add_request(1, list(range(2000, 2300)), 2)
    s.add_request(2, list(range(3000, 3100)), 2)
    b = s.step()
    assert b["kind"] == "prefill"
    assert [(e["req"], e["start"], e["count"]) for e in b["seqs"]] == [(0, 0, 512), (1, 0, 300), (2, 0, 100)]
    s.complete([1, 2, 3])           # requests 1 and 2 finished their prompts
    assert s.running == [1, 2] and s.prefilling == [0]
    b = s.step()                    # something runs and the decode streak is 0: decode
    assert b["kind"] == "decode" and [(e["req"], e["start"]) for e in b["seqs"]] == [(1, 300), (2, 100)]


def test_at_most_eight_decode_steps_while_a_prompt_waits():
    s = ReferenceScheduler(512, 16, budget=600, chunk=512)
    s.add_request(0, list(range(40)), 50)
    s.add_request(1, list(range(100, 1100)), 5)     # its second chunk has to wait
    kinds = []
    rng = np.random.default_rng(0)
    for _ in range(12):
        b = s.step()
        kinds.append(b["kind"][0])
        s.complete([int(rng.integers(1000)) for _ in b["seqs"]])
    assert "".join(kinds) == "p" + "d" * 8 + "p" + "dd"


def test_preemption_recomputes_and_keeps_the_token_count():
    # 6 blocks of 8 tokens: two requests of 20 prompt tokens growing by 12 cannot both fit
    s = ReferenceScheduler(6, 8, budget=64, chunk=64)
    s.add_request(0, list(range(20)), 12)
    s.add_request(1, list(range(100, 120)), 12)
    rng = np.random.default_rng(1)
    trace = _drain(s, rng)
    assert s.counters["preemptions"] >= 1 and s.counters["finished"] == 2
    assert s.counters["generated_tokens"] >= 24
    # a preempted request comes back as a prefill of everything it had, then decodes on
    firsts = [t for t in trace if t[0] == "prefill"]
    assert len(firsts) >= 2


def test_prompt_cached_but_for_its_last_token():
    s = ReferenceScheduler(64, 16)
    p = list(range(48))
    s.add_request(0, p, 1)
    rng = np.random.default_rng(2)
    _drain(s, rng)                                   # request 0 caches its 3 full blocks
    s.add_request(1, p, 1)
    b = s.step()
    assert [(e["req"], e["start"], e["count"]) for e in b["seqs"]] == [(1, 32, 16)]  # 2 blocks hit


# ----------------------------------------------------------------------------- C++ scheduler == reference

def _workload(seed, n, prompt_max, gen_max):
    rng = np.random.default_rng(seed)
    systems = [rng.integers(0, 1000, size=int(rng.integers(8, min(200, prompt_max)))).tolist() for _ in range(3)]
    reqs = []
    for i in range(n):
        own = rng.integers(0, 1000, size=int(rng.integers(1, prompt_max))).tolist()
        prompt = (systems[int(rng.integers(3))] + own) if rng.random() < 0.7 else own
        reqs.append((i, prompt, int(rng.integers(1, gen_max))))
    return reqs


@pytest.mark.parametrize("seed,blocks,bs,budget,chunk,decode,prompt_max", [
    (1, 512, 16, 4096, 512, 8, 600),
    (2, 96, 16, 1024, 256, 8, 600),       # small pool: preemptions
    (3, 200, 8, 2048, 512, 4, 600),
    (4, 64, 32, 512, 128, 2, 600),        # very small pool
    (5, 18, 16, 512, 128, 3, 60),         # prompts being prefilled hold the whole pool
])
def test_cpp_scheduler_matches_reference(cpp_cls, seed, blocks, bs, budget, chunk, decode, prompt_max):
    reqs = _workload(seed, 40, prompt_max, 40)
    ref = ReferenceScheduler(blocks, bs, budget, chunk, decode)
    cpp = cpp_cls(blocks, bs, budget, chunk, decode)
    for rid, p, g in reqs[:25]:
        ref.add_request(rid, p, g)
        cpp.add_request(rid, p, g)
    rng = np.random.default_rng(seed + 100)
    steps = 0
    while True:
        if steps == 30:                 # more requests arrive mid-run
            for rid, p, g in reqs[25:]:
                ref.add_request(rid, p, g)
                cpp.add_request(rid, p, g)
        br, bc = ref.step(), cpp.step()
        assert br["kind"] == bc["kind"], steps
        if br["kind"] == "idle":
            break
        seqs = br["seqs"]
        assert [e["req"] for e in seqs] == bc["req_ids"].tolist()
        assert np.cumsum([0] + [e["count"] for e in seqs]).tolist() == bc["query_start_loc"].tolist()
        assert [e["context"] for e in seqs] == bc["context_lens"].tolist()
        for i, e in enumerate(seqs):
            assert bc["block_tables"][i, :len(e["table"])].tolist() == e["table"]
        assert sum((e["tokens"] for e in seqs), []) == bc["token_ids"].tolist()
        assert sum((list(range(e["start"], e["start"] + e["count"])) for e in seqs), []) == bc["positions"].tolist()
        assert sum((e["slots"] for e in seqs), []) == bc["slot_mapping"].tolist()
        sampled = [int(rng.integers(1000)) for _ in seqs]
        assert ref.complete(sampled) == cpp.complete(sampled)
        steps += 1
    st = cpp.stats()
    assert {k: v for k, v in st.items() if k != "in_flight"} == ref.counters
    assert st["in_flight"] == 0 and st["finished"] == len(reqs)
    assert cpp.manager_stats() == ref.kv.stats()
    if blocks <= 96:
        assert st["preemptions"] > 0


def test_prompts_being_prefilled_cannot_block_each_other():
    """18 blocks of 16 tokens: several long prompts admitted together would hold every block
    with none able to take its next chunk; preempting the newest one keeps the step moving."""
    rng = np.random.default_rng(16)
    systems = [rng.integers(0, 500, size=int(n)).tolist() for n in (40, 70)]
    s = ReferenceScheduler(18, 16, 512, 128, 3)
    for rid in range(10):
        s.add_request(rid, systems[rid % 2] + rng.integers(0, 500, size=int(rng.integers(5, 150))).tolist(),
                      int(rng.integers(2, 30)))
    _drain(s, np.random.default_rng(5))
    assert s.counters["finished"] == 10 and s.counters["preemptions"] > 0


def test_requests_that_cannot_fit_are_refused(cpp_cls):
    from paged_kv_attention_write_gb300 import PAError
    with pytest.raises(ValueError):
        ReferenceScheduler(4, 16).add_request(0, list(range(60)), 5)
    with pytest.raises(PAError):
        cpp_cls(4, 16).add_request(0, list(range(60)), 5)


def test_packed_step_writes_the_same_batch_as_the_array_step(cpp_cls):
    """pa_sched_step_packed: two schedulers fed the same requests and the same sampled tokens,
    one stepped through separate arrays and one through one packed buffer, give equal
    batches step by step (every array compared at the offsets the call reports, each on a
    16-byte boundary, the device span first)."""
    import ctypes
    rng = np.random.default_rng(7)
    a, b = cpp_cls(64, 16, 512, 128, 3), cpp_cls(64, 16, 512, 128, 3)
    system = rng.integers(0, 500, size=48).tolist()
    for rid in range(12):
        p = (system if rid % 3 == 0 else []) + rng.integers(0, 500, size=int(rng.integers(5, 200))).tolist()
        n = int(rng.integers(2, 20))
        a.add_request(rid, p, n)
        b.add_request(rid, p, n)
    steps = 0
    while True:
        x = a.step()
        buf = np.zeros(b.packed_bytes() // 8 + 2, dtype=np.int64)  # 16-byte aligned storage
        ptr = buf.ctypes.data
        assert ptr % 16 == 0
        bt, o = b.step_packed(ptr, buf.nbytes)
        assert x["kind"] == {0: "idle", 1: "prefill", 2: "decode"}[bt.kind]
        if bt.kind == 0:
            break
        raw = buf.view(np.uint8)
        S, T, W = bt.num_seqs, bt.num_tokens, bt.table_width
        assert (S, T, bt.max_query_len, bt.max_context_len) == (x["num_seqs"], x["num_tokens"], x["max_query_len"],
                                                                x["max_context_len"])
        for name, off, dt, n in (("query_start_loc", o.query_start_loc, np.int32, S + 1),
                                 ("context_lens", o.context_lens, np.int32, S),
                                 ("slot_mapping", o.slot_mapping, np.int64, T),
                                 ("token_ids", o.token_ids, np.int32, T), ("positions", o.positions, np.int32, T),
                                 ("req_ids", o.req_ids, np.int64, S)):
            assert off % 16 == 0
            got = np.frombuffer(raw, dt, n, off)
            assert np.array_equal(got, x[name]), name
        tables = np.frombuffer(raw, np.int32, S * W, o.block_tables).reshape(S, W)
        assert np.array_equal(tables, x["block_tables"])
        pairs = np.frombuffer(raw, np.int64, 2 * bt.num_copy_pairs, o.copy_pairs).reshape(-1, 2)
        assert np.array_equal(pairs, x["copy_pairs"])
        assert max(o.query_start_loc, o.context_lens, o.block_tables, o.slot_mapping, o.copy_pairs, o.token_ids,
                   o.positions) < o.dev_bytes <= o.req_ids < o.total_bytes <= buf.nbytes
        sampled = rng.integers(0, 500, size=S).tolist()
        a.complete(sampled)
        b.complete(sampled)
        steps += 1
    assert steps > 10


def test_packed_step_rejects_a_short_buffer(cpp_cls):
    from paged_kv_attention_write_gb300 import PAError
    s = cpp_cls(64, 16, 512, 128, 3)
    s.add_request(0, list(range(100)), 4)
    buf = np.zeros(4, dtype=np.int64)
    with pytest.raises(PAError):
        s.step_packed(buf.ctypes.data, buf.nbytes)
    buf = np.zeros(s.packed_bytes() // 8 + 2, dtype=np.int64)
    bt, _ = s.step_packed(buf.ctypes.data, buf.nbytes)   # nothing changed by the refused call
    assert bt.kind == 1 and bt.num_tokens == 100
