"""GPU parity: the CUDA library (called through its C ABI) against the fp64 oracle on
the same seeded inputs.  Cache writes and block copies bit-exact; attention within
max-abs 5e-3 / mean-abs 5e-4 in fp32 (tighter for fp32 inputs)."""
import math

import numpy as np
import pytest
import torch

import workloads
from paged_steps import (assert_attention_close, bits, check_case, gpu_step, oracle_step, oracle_step_pools)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


# ----------------------------------------------------------------------------- the five workloads

def test_tiny_decode(oracle_mod):
    case = workloads.tiny_decode()
    mx, _ = check_case(case, oracle_mod)
    assert mx < 1e-5  # fp32 inputs, fp32 accumulation


def test_decode_batch_full_size(oracle_mod):
    check_case(workloads.decode_batch(), oracle_mod)


def test_long_decode_full_size(oracle_mod):
    check_case(workloads.long_decode(), oracle_mod)


def test_prefill_chunk_full_size(oracle_mod):
    check_case(workloads.prefill_chunk(), oracle_mod)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_stress_full_size(oracle_mod, bs, dtype):
    case = workloads.stress_decode(block_size=bs, dtype=dtype)
    assert case.block_mapping is not None and case.block_mapping.shape[0] > 0
    check_case(case, oracle_mod)


# ----------------------------------------------------------------------------- decode shapes and edges

DECODE_LENS = [0, 1, 7, 8, 31, 32, 33, 511, 512, 513, 1100, 2049]


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16],
                         ids=["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_decode_shape_sweep(oracle_mod, dtype, D, G, bs):
    """Every built (dtype, head dim, group, block size) on ragged context lengths that
    cover single-token, exact-block, block+1 and multi-partition cases."""
    Hkv = 2
    case = workloads.make_decode_case("sweep", DECODE_LENS, bs, Hkv * G, Hkv, D, dtype,
                                      seed=D * 100 + G * 10 + bs, free_frac=0.1)
    mx, mn = check_case(case, oracle_mod)
    if dtype == torch.float32:
        assert mx < 1e-5


@pytest.mark.parametrize("Hkv", [1, 4, 8, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_eight_query_heads_per_kv_head(oracle_mod, Hkv, D):
    """Eight query heads per kv head run as two query slices of four heads per kv head: one
    kv head (four token slices), one group of four, two and four groups (one token slice),
    with a long sequence split over many CTAs."""
    case = workloads.make_decode_case("g8", DECODE_LENS + [9000], 16, 8 * Hkv, Hkv, D, torch.bfloat16,
                                      seed=800 + Hkv * 10 + D, free_frac=0.1)
    check_case(case, oracle_mod)


def test_decode_zero_context_gives_zero_row(oracle_mod):
    case = workloads.make_decode_case("zero", [40, 3, 700], 16, 8, 2, 128, torch.bfloat16, 9)
    case.context_lens[1] = 0       # sequence 1 attends nothing
    case.slot_mapping[1] = -1      # and writes nothing
    out, kc, vc, status = gpu_step(case)
    ref, okc, ovc = oracle_step(case, oracle_mod)
    assert status == 0
    assert torch.all(out[1] == 0)
    assert torch.equal(bits(kc), bits(okc))
    assert_attention_close(out, ref)


def test_decode_is_deterministic_and_placement_independent(oracle_mod):
    """Two runs are byte-identical; the same logical K/V under another block placement
    gives byte-identical output (the arithmetic order depends on logical positions only)."""
    a = workloads.make_decode_case("p", [900, 77, 1500, 2], 16, 16, 4, 128, torch.bfloat16, 21)
    o1, *_ = gpu_step(a)
    o2, *_ = gpu_step(a)
    assert torch.equal(bits(o1), bits(o2))
    # re-place every block of a at new physical ids
    NB = a.num_blocks
    perm = torch.from_numpy(np.random.default_rng(5).permutation(NB)).to(torch.int64)
    b = workloads.make_decode_case("p", [900, 77, 1500, 2], 16, 16, 4, 128, torch.bfloat16, 21)
    b.key_cache = torch.empty_like(a.key_cache)
    b.value_cache = torch.empty_like(a.value_cache)
    b.key_cache[perm] = a.key_cache
    b.value_cache[perm] = a.value_cache
    valid = a.block_tables >= 0
    b.block_tables = torch.where(valid, perm[a.block_tables.clamp(min=0).long()].to(torch.int32),
                                 a.block_tables)
    bs = a.block_size
    b.slot_mapping = perm[a.slot_mapping // bs] * bs + a.slot_mapping % bs
    o3, *_ = gpu_step(b)
    assert torch.equal(bits(o1), bits(o3))


def _decode_subset(case, t, seqs):
    """pa_decode of the sequences `seqs` of an already written case (shared pools)."""
    import paged_kv_attention_write_gb300 as pa
    idx = torch.tensor(seqs, dtype=torch.int64, device="cuda")
    q, bt, cl = t["q"][idx].contiguous(), t["bt"][idx].contiguous(), t["cl"][idx].contiguous()
    mcl = int(case.context_lens[seqs].max())
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device="cuda")
    n = pa.pa_decode_workspace_size(len(seqs), case.num_heads, case.num_kv_heads, case.head_dim, mcl)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(out, q, t["kc"], t["vc"], bt, cl, mcl, case.scale, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out.cpu()


def test_decode_result_independent_of_split(oracle_mod):
    """The same long sequence decoded alone and inside batches of different sizes: the
    balanced split cuts it into about 152, 40 and 10 pieces at different boundaries (the
    split follows every sequence's length), and its rows agree within 1e-5 each time; every
    batch also matches the oracle."""
    import paged_kv_attention_write_gb300 as pa
    rng = np.random.default_rng(17)
    lens = [30000] + [int(x) for x in rng.integers(6000, 14000, size=7)] + \
           [int(x) for x in rng.integers(100, 3000, size=56)]
    case = workloads.make_decode_case("split", lens, 32, 32, 8, 128, torch.bfloat16, 17)
    t = {"q": case.query.cuda(), "kc": case.key_cache.cuda(), "vc": case.value_cache.cuda(),
         "bt": case.block_tables.cuda(), "cl": case.context_lens.cuda()}
    pa.pa_reshape_and_cache(case.new_key.cuda(), case.new_value.cuda(), t["kc"], t["vc"],
                            case.slot_mapping.cuda())
    _, okc, ovc = oracle_step(case, oracle_mod)
    rows = []
    for seqs in ([0], list(range(8)), list(range(64))):
        out = _decode_subset(case, t, seqs)
        qsl = torch.arange(len(seqs) + 1, dtype=torch.int32)
        ref = oracle_mod.paged_attention(case.query[seqs], qsl, okc, ovc, case.block_tables[seqs],
                                         case.context_lens[seqs], case.scale)
        assert_attention_close(out, ref)
        rows.append(out[0])
    for r in rows[1:]:
        assert (r - rows[0]).abs().max().item() <= 1e-5


def test_decode_workspace_needs_no_initialisation_and_old_launches_never_count(oracle_mod):
    """One workspace, first filled with random bytes, shared by a 32-sequence call, a call on
    8 of its sequences and, after the workspace is put back to what the first call left in it
    (its partials and its launch tags), the first shape again with another query: the reduce
    must wait for this launch's pieces, never take the earlier launch's.  Every call against
    the oracle."""
    import paged_kv_attention_write_gb300 as pa
    rng = np.random.default_rng(23)
    lens = [9000] + [int(x) for x in rng.integers(2000, 5000, size=7)] + \
           [int(x) for x in rng.integers(100, 1500, size=24)]
    case = workloads.make_decode_case("reuse", lens, 32, 32, 8, 128, torch.bfloat16, 23)
    kc, vc = case.key_cache.cuda(), case.value_cache.cuda()
    pa.pa_reshape_and_cache(case.new_key.cuda(), case.new_value.cuda(), kc, vc, case.slot_mapping.cuda())
    _, okc, ovc = oracle_step(case, oracle_mod)
    S, Hq, D = case.query.shape
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, int(case.context_lens.max()))
    ws = torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(q, seqs):
        idx = torch.tensor(seqs, dtype=torch.int64)
        mcl = int(case.context_lens[idx].max())
        out = torch.full((len(seqs), Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        pa.pa_decode(out, q[idx].contiguous().cuda(), kc, vc, case.block_tables[idx].contiguous().cuda(),
                     case.context_lens[idx].contiguous().cuda(), mcl, case.scale, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        ref = oracle_mod.paged_attention(q[idx], torch.arange(len(seqs) + 1, dtype=torch.int32), okc, ovc,
                                         case.block_tables[idx], case.context_lens[idx], case.scale)
        assert_attention_close(out.cpu(), ref)
        return out.cpu()

    every = list(range(S))
    q2 = torch.from_numpy(rng.standard_normal(tuple(case.query.shape)).astype(np.float32)).to(case.query.dtype)
    first = run(case.query, every)
    left = ws.clone()
    run(case.query, list(range(0, S, 4)))
    ws.copy_(left)
    again = run(q2, every)
    assert (again - first).abs().max().item() > 0.1  # the new query's rows, not the old ones


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_decode_low_precision_output_is_rounded_fp32(oracle_mod, out_dtype):
    case = workloads.make_decode_case("o", [100, 1000, 3000], 32, 32, 8, 128, torch.bfloat16, 4)
    o32, *_ = gpu_step(case, torch.float32)
    olo, *_ = gpu_step(case, out_dtype)
    assert torch.equal(bits(olo), bits(o32.to(out_dtype)))


def test_decode_aliased_block_tables(oracle_mod):
    """Read-only sharing: several block tables point at the same physical prefix blocks."""
    case = workloads.make_decode_case("alias", list(range(100, 2100, 100)), 16, 32, 8, 128,
                                      torch.bfloat16, 13, free_frac=0.2, alias_frac=0.3)
    assert case.meta["aliased"]
    check_case(case, oracle_mod)


def test_decode_one_sequence_of_128k_tokens(oracle_mod):
    """The largest single context of the tests: 131,072 tokens (4,096 blocks of 32), one
    sequence split into one piece per CTA, so the reduce merges ~150 pieces in batches."""
    case = workloads.make_decode_case("128k", [131071], 32, 32, 8, 128, torch.bfloat16, 128)
    check_case(case, oracle_mod)


# ----------------------------------------------------------------------------- prefill shapes and edges

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_shape_sweep(oracle_mod, dtype, D, G):
    """Ragged chunks (1 row, sub-tile, multi-tile with tail) over prefixes that are empty,
    sub-block, and multi-tile."""
    Hkv = 2
    prefix = [0, 5, 64, 300, 0, 1000]
    chunk = [1, 17, 64, 130, 200, 3]
    for bs in (8, 16, 32):
        case = workloads.make_prefill_case("pf", prefix, chunk, bs, Hkv * G, Hkv, D, dtype,
                                           seed=bs + D + G, free_frac=0.1)
        check_case(case, oracle_mod)


def test_prefill_unit_order_many_ragged_units(oracle_mod):
    """60 sequences of random prefix and chunk lengths: the longest-first unit ranking
    sees many ties and empty units and must still give every unit exactly one CTA set."""
    rng = np.random.default_rng(21)
    prefix = rng.integers(0, 3000, size=60).tolist()
    chunk = rng.integers(1, 300, size=60).tolist()
    case = workloads.make_prefill_case("pf-rank", prefix, chunk, 16, 16, 4, 128, torch.bfloat16,
                                       seed=21)
    check_case(case, oracle_mod)


def test_prefill_unit_order_launch_order_fallback(oracle_mod):
    """More than 4096 units (2100 sequences x 2 query tiles at G=1) skip the ranking and
    run in launch order."""
    prefix = [(7 * i) % 90 for i in range(2100)]
    chunk = [1 + (i % 3) for i in range(2100)]
    chunk[5] = 129  # two 128-row tiles
    case = workloads.make_prefill_case("pf-many", prefix, chunk, 8, 2, 2, 64, torch.float16,
                                       seed=22)
    check_case(case, oracle_mod)


# ----------------------------------------------------------------------------- mixed decode + prefill batches

def test_mixed_batch_full_size(oracle_mod):
    """28 decode rows and four 512-token chunks in one pa_prefill_chunk launch."""
    check_case(workloads.mixed_batch(), oracle_mod)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("bs", [8, 32])
def test_mixed_batch_interleaved(oracle_mod, dtype, bs):
    """Decode rows between chunks (and a chunk on an empty prefix) in one launch."""
    prefix = [300, 0, 47, 1000, 5, 129, 600]
    chunk = [1, 200, 1, 64, 1, 1, 130]
    case = workloads.make_prefill_case("mixed-il", prefix, chunk, bs, 16, 4, 128, dtype, seed=bs,
                                       free_frac=0.1)
    check_case(case, oracle_mod)


def test_mixed_batch_decode_rows_match_alone_and_decode():
    """Each item's arithmetic is independent of the others: the decode rows of a mixed
    launch equal, bit for bit, the same rows run alone through pa_prefill_chunk, and
    agree with pa_decode within tolerance."""
    import paged_kv_attention_write_gb300 as pa
    dev = "cuda"
    mix = workloads.mixed_batch()
    out_mix, kc, vc, st = gpu_step(mix)
    assert st == 0
    nd = 28  # decode rows come first, one query token each
    q = mix.query[:nd].to(dev)
    qsl = torch.arange(nd + 1, dtype=torch.int32, device=dev)
    bt = mix.block_tables[:nd].contiguous().to(dev)
    cl = mix.context_lens[:nd].contiguous().to(dev)
    kc, vc = kc.to(dev), vc.to(dev)
    alone = torch.empty(tuple(q.shape), dtype=torch.float32, device=dev)
    pa.pa_prefill_chunk(alone, q, qsl, 1, kc, vc, bt, cl, int(cl.max()), mix.scale)
    ws = torch.empty(max(1, pa.pa_decode_workspace_size(nd, mix.num_heads, mix.num_kv_heads,
                                                        mix.head_dim, int(cl.max()))),
                     dtype=torch.uint8, device=dev)
    dec = torch.empty_like(alone)
    pa.pa_decode(dec, q, kc, vc, bt, cl, int(cl.max()), mix.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_mix[:nd], alone.cpu())
    assert (dec.cpu() - out_mix[:nd]).abs().max().item() < 5e-3


def test_prefill_long_prefix_large_chunks_sampled_rows(oracle_mod):
    """Two 2048-token chunks, one over a 16,384-token prefix (the unit of ~144 key tiles), one
    fresh: the whole launch on the GPU, and 48 rows per sequence -- the chunk's first and last
    rows, rows at 128-key tile edges, the rest random -- against the oracle, each sampled row
    as a one-row query over keys 0 .. its position (the causal definition)."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_prefill_case("long-prefix", [16384, 0], [2048, 2048], 16, 32, 8, 128,
                                       torch.bfloat16, 31)
    out, *_ , status = gpu_step(case)
    assert status == 0
    _, okc, ovc = oracle_step_pools(case, oracle_mod)
    rng = np.random.default_rng(31)
    qsl = case.query_start_loc.tolist()
    rows, bts, cls = [], [], []
    for s_ in range(case.num_seqs):
        Lq = qsl[s_ + 1] - qsl[s_]
        P = int(case.context_lens[s_]) - Lq
        pick = {0, 1, Lq - 1, Lq - 2} | {r for r in (127, 128, 255, 256, 1023, 1024) if r < Lq}
        pick |= set(int(x) for x in rng.integers(0, Lq, size=48 - len(pick)))
        for r in sorted(pick)[:48]:
            rows.append(qsl[s_] + r)
            bts.append(case.block_tables[s_])
            cls.append(P + r + 1)
    idx = torch.tensor(rows)
    ref = oracle_mod.paged_attention(case.query[idx], torch.arange(len(rows) + 1, dtype=torch.int32), okc, ovc,
                                     torch.stack(bts), torch.tensor(cls, dtype=torch.int32), case.scale)
    assert_attention_close(out[idx], ref)


def test_prefill_single_row_matches_decode(oracle_mod):
    """A chunk of one row is a decode step: both kernels agree within tolerance."""
    d = workloads.make_decode_case("pd", [63, 500, 1200], 16, 32, 8, 128, torch.bfloat16, 17)
    od, *_ = gpu_step(d)
    p = workloads.make_decode_case("pd", [63, 500, 1200], 16, 32, 8, 128, torch.bfloat16, 17)
    import paged_kv_attention_write_gb300 as pa
    dev = "cuda"
    kc, vc = p.key_cache.to(dev), p.value_cache.to(dev)
    pa.pa_reshape_and_cache(p.new_key.to(dev), p.new_value.to(dev), kc, vc, p.slot_mapping.to(dev))
    out = torch.empty(p.query.shape, dtype=torch.float32, device=dev)
    pa.pa_prefill_chunk(out, p.query.to(dev), p.query_start_loc.to(dev), 1, kc, vc,
                        p.block_tables.to(dev), p.context_lens.to(dev), p.max_context_len, p.scale)
    torch.cuda.synchronize()
    assert (out.cpu() - od).abs().max().item() < 5e-3


# ----------------------------------------------------------------------------- moving reference max

def _keys_growing_with_position(case, rate=1.0 / 8):
    """Scale every key (cached and fresh) by 1 + rate * position.  A row's scores then grow
    along its context by far more than the 2^8 that the lazily rescaled running max lets
    pass, so the reference moves inside rows, tile after tile, and the kernels rescale the
    output accumulated so far; with N(0,1) keys that path never runs."""
    kc, bt, bs = case.key_cache, case.block_tables, case.block_size
    for s in range(case.num_seqs):
        for j in range(int(case.cached_lens[s])):
            b, o = int(bt[s, j // bs]), j % bs
            kc[b, o] = (kc[b, o].double() * (1 + rate * j)).to(kc.dtype)
    if case.is_decode:
        pos = [int(n) for n in case.cached_lens]
    else:
        qsl = case.query_start_loc.tolist()
        pos = [int(case.cached_lens[s]) + i for s in range(case.num_seqs) for i in range(qsl[s + 1] - qsl[s])]
    for t, ps in enumerate(pos):
        case.new_key[t] = (case.new_key[t].double() * (1 + rate * ps)).to(case.new_key.dtype)
    return case


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_prefill_running_max_moves_across_tiles(oracle_mod, dtype):
    case = workloads.make_prefill_case("pf-grow", [0, 300, 1000], [200, 130, 64], 16, 8, 2, 128, dtype,
                                       seed=31)
    check_case(_keys_growing_with_position(case), oracle_mod)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "fp16", "fp32"])
def test_decode_running_max_moves_across_tiles(oracle_mod, dtype):
    case = workloads.make_decode_case("dec-grow", [100, 700, 2000], 16, 8, 2, 128, dtype, seed=32)
    check_case(_keys_growing_with_position(case), oracle_mod)


# ----------------------------------------------------------------------------- device-side range checks

def test_device_checks_report_instead_of_reading_out_of_range():
    """Bad block ids, slots, copy pairs and context lengths set status bits; nothing
    outside the buffers is read or written (the pools keep their bytes)."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_decode_case("bad", [40, 90], 16, 8, 2, 128, torch.bfloat16, 3)
    dev = "cuda"
    kc, vc = case.key_cache.to(dev), case.value_cache.to(dev)
    before = bits(kc).clone()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    NB = case.num_blocks
    # slot past the pool
    pa.pa_reshape_and_cache(case.new_key[:1].to(dev), case.new_value[:1].to(dev), kc, vc,
                            torch.tensor([NB * 16 + 3], dtype=torch.int64, device=dev), status=st)
    torch.cuda.synchronize()
    assert st.item() & 1 and torch.equal(bits(kc), before)
    # copy pair with a block id past the pool
    st.zero_()
    pa.pa_copy_blocks(kc, vc, torch.tensor([[0, NB + 2]], dtype=torch.int64, device=dev), status=st)
    torch.cuda.synchronize()
    assert st.item() & 2 and torch.equal(bits(kc), before)
    # block table entry past the pool, and a context longer than the table
    bt = case.block_tables.clone()
    bt[0, 1] = NB + 100
    cl = case.context_lens.clone()
    cl[1] = bt.shape[1] * 16 + 50
    out = torch.empty(case.query.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    st.zero_()
    pa.pa_decode(out, case.query.to(dev), kc, vc, bt.to(dev), cl.to(dev), int(cl.max()),
                 case.scale, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() & 2 and st.item() & 4
    st.zero_()
    qsl = torch.tensor([0, 1, 5], dtype=torch.int32, device=dev)  # runs past the 2 query rows
    pa.pa_prefill_chunk(out, case.query.to(dev), qsl, 4, kc, vc, bt.to(dev), cl.to(dev),
                        int(cl.max()), case.scale, status=st)
    torch.cuda.synchronize()
    assert st.item() & 8


def test_reshape_and_cache_skips_negative_slots(oracle_mod):
    case = workloads.make_decode_case("neg", [10, 20, 30, 40], 8, 4, 2, 64, torch.float16, 8)
    case.slot_mapping[2] = -1
    case.context_lens[2] = int(case.cached_lens[2])  # nothing fresh for sequence 2
    check_case(case, oracle_mod)
