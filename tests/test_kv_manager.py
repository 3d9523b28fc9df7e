"""Host KV-cache manager: the reference policy pinned by hand-worked cases, and the C++
manager (through its C ABI) equal to the reference after every operation of seeded random
request streams (prefix sharing, chunked growth, decode steps, forks, frees, exhaustion)."""
import numpy as np
import pytest

from oracle.kv_manager import ReferenceKVManager


@pytest.fixture(scope="module")
def cpp_cls(pa_lib_path):
    from paged_kv_attention_write_gb300.kv_manager import KVCacheManager
    return KVCacheManager


# ----------------------------------------------------------------------------- pins of the reference

def test_free_queue_order_lru():
    """Allocation takes the head; a freed request goes to the tail last block first."""
    m = ReferenceKVManager(8, 8)
    m.admit(1, range(20)); m.allocate_slots(1, 20)
    m.admit(2, range(100, 110)); m.allocate_slots(2, 10)
    assert m.block_table(1) == [0, 1, 2] and m.block_table(2) == [3, 4]
    m.free(1)
    m.free(2)
    assert m.free_queue == [5, 6, 7, 2, 1, 0, 4, 3]
    m.admit(3, range(200, 230)); m.allocate_slots(3, 30)
    assert m.block_table(3) == [5, 6, 7, 2]


def test_prefix_hits_cover_full_blocks_and_leave_the_last_token():
    bs = 8
    m = ReferenceKVManager(16, bs)
    t = list(range(1000, 1028))                  # 3 full blocks + 4 tokens
    m.admit(1, t); m.allocate_slots(1, len(t)); m.cache_blocks(1, t, len(t))
    a = m.block_table(1)
    assert m.get_computed_blocks(t[:24] + [7]) == a[:3]   # 25 tokens: 3 full blocks hit
    assert m.get_computed_blocks(t[:24]) == a[:2]         # 24 tokens: the last block is recomputed
    assert m.get_computed_blocks(t[:16] + [5] * 9) == a[:2]  # diverges in block 2
    assert m.get_computed_blocks([5] + t[1:]) == []       # diverges in block 0
    assert m.get_computed_blocks(t[:7]) == []             # no full block


def test_cached_blocks_survive_free_until_handed_out():
    bs = 8
    m = ReferenceKVManager(4, bs)
    t = list(range(16))
    m.admit(1, t + [1]); m.allocate_slots(1, 17); m.cache_blocks(1, t + [1], 17)
    m.free(1)                                   # queue: [3, 2, 1, 0]; blocks 0, 1 stay cached
    assert m.free_queue == [3, 2, 1, 0] and m.get_computed_blocks(t + [2]) == [0, 1]
    m.admit(2, [9] * 17); m.allocate_slots(2, 17)  # takes 3, 2, 1: block 1 leaves the cache
    assert m.block_table(2) == [3, 2, 1]
    assert m.stats()["evictions"] == 1 and m.get_computed_blocks(t + [2]) == [0]


def test_hit_on_a_free_cached_block_takes_it_out_of_the_queue():
    m = ReferenceKVManager(6, 8)
    t = list(range(40, 57))
    m.admit(1, t); m.allocate_slots(1, 17); m.cache_blocks(1, t, 16)
    m.free(1)
    assert m.num_free_blocks == 6
    assert m.admit(2, t) == 16 and m.num_free_blocks == 4 and m.block_table(2) == [0, 1]


def test_fork_copy_on_write_of_the_shared_partial_block():
    m = ReferenceKVManager(8, 8)
    m.admit(1, range(12)); m.allocate_slots(1, 12)   # blocks [0, 1], block 1 partial
    m.fork(1, 2)
    assert m.allocate_slots(2, 13) == [(1, 2)] and m.block_table(2) == [0, 2]
    assert m.allocate_slots(1, 13) == [] and m.block_table(1) == [0, 1]
    assert m.ref[0] == 2 and m.ref[1] == 1 and m.ref[2] == 1


def test_slot_formula():
    m = ReferenceKVManager(8, 16)
    m.admit(7, range(5)); m.allocate_slots(7, 40)
    bl = m.block_table(7)
    assert m.slot_mapping(7, 14, 4) == [bl[0] * 16 + 14, bl[0] * 16 + 15, bl[1] * 16, bl[1] * 16 + 1]


def test_prefix_cache_off_never_hits():
    m = ReferenceKVManager(8, 8, prefix_cache=False)
    t = list(range(30))
    m.admit(1, t); m.allocate_slots(1, 30); m.cache_blocks(1, t, 30)
    assert m.get_computed_blocks(t) == [] and m.stats()["blocks_cached"] == 0


# ----------------------------------------------------------------------------- C++ manager == reference

def _run_stream(cpp_cls, seed, num_blocks, bs, prefix_cache=True, n_ops=600):
    rng = np.random.default_rng(seed)
    ref = ReferenceKVManager(num_blocks, bs, prefix_cache)
    cpp = cpp_cls(num_blocks, bs, prefix_cache)
    prefixes = [rng.integers(0, 50, size=int(rng.integers(bs, 5 * bs))).tolist() for _ in range(4)]
    live = {}  # req id -> [tokens, computed]
    next_id = 0

    def same(what):
        assert ref.num_free_blocks == cpp.num_free_blocks, what
        assert ref.stats() == cpp.stats(), what
        for rid in live:
            assert ref.block_table(rid) == cpp.block_table(rid), (what, rid)

    for op in range(n_ops):
        kind = rng.choice(["admit", "grow", "decode", "fork", "free", "lookup"],
                          p=[0.22, 0.2, 0.3, 0.05, 0.15, 0.08])
        if kind == "admit" or not live:
            p = prefixes[int(rng.integers(len(prefixes)))]
            cut = int(rng.integers(1, len(p) + 1))
            toks = p[:cut] + rng.integers(0, 50, size=int(rng.integers(0, 3 * bs))).tolist()
            rid = next_id
            next_id += 1
            a, b = ref.admit(rid, toks), cpp.admit(rid, toks)
            assert a == b
            live[rid] = [toks, a]
            same(f"admit {op}")
        elif kind in ("grow", "decode"):
            rid = list(live)[int(rng.integers(len(live)))]
            toks, done = live[rid]
            if kind == "grow" and done < len(toks):        # next prefill chunk of the prompt
                new = min(len(toks), done + int(rng.integers(1, 2 * bs)))
            else:                                         # one decode token
                toks = toks + [int(rng.integers(0, 50))]
                new = len(toks)
            try:
                pr = ref.allocate_slots(rid, new)
            except MemoryError:
                pr = None
            try:
                pc = cpp.allocate_slots(rid, new)
            except Exception as e:                        # PA_ERR_NO_BLOCKS
                assert getattr(e, "code", None) == -5
                pc = None
            assert pr == pc, op
            if pr is not None:
                live[rid] = [toks, new]
                ref.cache_blocks(rid, toks, new)
                cpp.cache_blocks(rid, toks, new)
                assert ref.slot_mapping(rid, 0, new) == cpp.slot_mapping(rid, 0, new).tolist()
            same(f"{kind} {op}")
        elif kind == "fork":
            rid = list(live)[int(rng.integers(len(live)))]
            child = next_id
            next_id += 1
            ref.fork(rid, child)
            cpp.fork(rid, child)
            live[child] = list(live[rid])
            same(f"fork {op}")
        elif kind == "free":
            rid = list(live)[int(rng.integers(len(live)))]
            ref.free(rid)
            cpp.free(rid)
            del live[rid]
            same(f"free {op}")
        else:
            p = prefixes[int(rng.integers(len(prefixes)))] + [int(rng.integers(0, 50))]
            assert ref.get_computed_blocks(p) == cpp.get_computed_blocks(p)
            same(f"lookup {op}")
    cpp.close()


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_cpp_manager_matches_reference(cpp_cls, bs, seed):
    _run_stream(cpp_cls, seed * 10 + bs, num_blocks=48, bs=bs)


def test_cpp_manager_matches_reference_under_exhaustion(cpp_cls):
    """A pool so small that allocations fail often: both refuse the same requests."""
    _run_stream(cpp_cls, 77, num_blocks=10, bs=8, n_ops=800)


def test_cpp_manager_matches_reference_without_prefix_cache(cpp_cls):
    _run_stream(cpp_cls, 5, num_blocks=40, bs=16, prefix_cache=False)


def test_cpp_manager_rejects_bad_calls(cpp_cls):
    from paged_kv_attention_write_gb300 import PAError
    m = cpp_cls(4, 8)
    with pytest.raises(PAError):
        m.free(99)
    m.admit(1, [1, 2, 3])
    with pytest.raises(PAError):
        m.admit(1, [1])                 # duplicate request
    with pytest.raises(PAError):
        m.allocate_slots(1, 100)        # 13 blocks of a 4-block pool: nothing changes
    assert m.num_free_blocks == 4 and m.block_table(1) == []
    with pytest.raises(PAError):
        m.slot_mapping(1, 0, 1)         # position not covered by the request's blocks
    with pytest.raises(PAError):
        cpp_cls(4, 12)                  # block size not 8, 16 or 32
