"""Decode with eight query heads per kv head on a 16-bit cache and enough (sequence, kv head)
pairs to occupy the GPU: the query rows run through the tensor-core chunk kernel as
one-token chunks.  Against the oracle over cache types, head dims and block sizes (empty
contexts give zero rows), clamped contexts reported, results independent of the other
sequences of the batch (bit for bit), the fused cache write equal to its two calls, and a
captured call replaying like eager calls."""
import numpy as np
import pytest
import torch

import workloads
from paged_steps import assert_attention_close, bits, check_case, oracle_step

pytestmark = pytest.mark.gpu

PA_DEVERR_CONTEXT = 4


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _lens(seed, n=48):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 7, 8, 31, 32, 33, 127, 128, 129, 511, 2049, 5000]
    return fixed + [int(x) for x in rng.integers(1, 3000, size=n - len(fixed))]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_tensor_rows_against_oracle(oracle_mod, dtype, D, bs):
    case = workloads.make_decode_case("tr", _lens(D + bs), bs, 64, 8, D, dtype, seed=900 + D + bs,
                                      free_frac=0.1)
    check_case(case, oracle_mod)


def _device(case):
    dev = "cuda"
    return {"q": case.query.to(dev), "kc": case.key_cache.to(dev), "vc": case.value_cache.to(dev),
            "bt": case.block_tables.to(dev), "cl": case.context_lens.to(dev), "sl": case.slot_mapping.to(dev),
            "nk": case.new_key.to(dev), "nv": case.new_value.to(dev)}


def _decode(pa, case, t, seqs=None, cl=None, mcl=None, out_dtype=torch.float32):
    idx = torch.arange(case.num_seqs) if seqs is None else torch.tensor(seqs)
    idx = idx.to("cuda")
    q, bt = t["q"][idx].contiguous(), t["bt"][idx].contiguous()
    cl = (t["cl"] if cl is None else cl)[idx].contiguous()
    mcl = case.max_context_len if mcl is None else mcl
    S, Hq, D = q.shape
    out = torch.full((S, Hq, D), float("nan"), dtype=out_dtype, device="cuda")
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, mcl)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(out, q, t["kc"], t["vc"], bt, cl, mcl, case.scale, workspace=ws, status=status)
    torch.cuda.synchronize()
    return out.cpu(), int(status.item())


def test_tensor_rows_clamp_and_report_bad_contexts(oracle_mod):
    """A negative context gives a zero row and one longer than max_context_len is cut to it;
    both set PA_DEVERR_CONTEXT; every other row is unchanged."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_decode_case("bad", _lens(3), 16, 64, 8, 128, torch.bfloat16, 31)
    t = _device(case)
    pa.pa_reshape_and_cache(t["nk"], t["nv"], t["kc"], t["vc"], t["sl"])
    good, st = _decode(pa, case, t)
    assert st == 0
    cl = t["cl"].clone()
    mcl = case.max_context_len
    long_row = int(torch.argmax(case.context_lens))
    cl[2] = -5
    got, st = _decode(pa, case, t, cl=cl, mcl=mcl - 100)
    assert st & PA_DEVERR_CONTEXT
    assert torch.equal(got[2], torch.zeros_like(got[2]))
    # the longest row now sees only the first mcl - 100 keys: the oracle on that length
    _, okc, ovc = oracle_step(case, oracle_mod)
    clamped = case.context_lens.clone()
    clamped[long_row] = mcl - 100
    ref = oracle_mod.paged_attention(case.query[[long_row]], torch.arange(2, dtype=torch.int32), okc, ovc,
                                     case.block_tables[[long_row]], clamped[[long_row]], case.scale)
    assert_attention_close(got[[long_row]], ref)
    others = [s for s in range(case.num_seqs) if s not in (2, long_row)]
    assert torch.equal(bits(got[others]), bits(good[others]))


def test_tensor_rows_do_not_depend_on_the_rest_of_the_batch():
    """Each (sequence, kv head) is one item with a fixed key order, so a sequence's rows are
    the same bits in any batch that keeps this path (here 48, 24 and 12 sequences)."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_decode_case("ind", _lens(4), 32, 64, 8, 128, torch.bfloat16, 32)
    t = _device(case)
    pa.pa_reshape_and_cache(t["nk"], t["nv"], t["kc"], t["vc"], t["sl"])
    full, st = _decode(pa, case, t)
    assert st == 0
    for seqs in (list(range(0, 48, 2)), list(range(5, 48, 4))):
        part, st = _decode(pa, case, t, seqs=seqs, mcl=int(case.context_lens[seqs].max()))
        assert st == 0
        assert torch.equal(bits(part), bits(full[seqs]))
    again, _ = _decode(pa, case, t)
    assert torch.equal(bits(again), bits(full))


def test_tensor_rows_fused_write_equals_two_calls():
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_decode_case("fw", _lens(5), 16, 64, 8, 128, torch.float16, 33)
    a, b = _device(case), _device(case)
    S, Hq, D = case.query.shape
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, case.max_context_len)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o1 = torch.empty((S, Hq, D), dtype=torch.float32, device="cuda")
    o2 = torch.empty_like(o1)
    pa.pa_decode_write(o1, a["q"], a["nk"], a["nv"], a["sl"], a["kc"], a["vc"], a["bt"], a["cl"],
                       case.max_context_len, case.scale, workspace=ws)
    pa.pa_reshape_and_cache(b["nk"], b["nv"], b["kc"], b["vc"], b["sl"])
    pa.pa_decode(o2, b["q"], b["kc"], b["vc"], b["bt"], b["cl"], case.max_context_len, case.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(bits(o1), bits(o2))
    assert torch.equal(bits(a["kc"]), bits(b["kc"])) and torch.equal(bits(a["vc"]), bits(b["vc"]))


def test_tensor_rows_graph_replays_equal_eager_calls():
    import paged_kv_attention_write_gb300 as pa
    case = workloads.make_decode_case("gr", _lens(6), 32, 64, 8, 128, torch.bfloat16, 34)
    t = _device(case)
    pa.pa_reshape_and_cache(t["nk"], t["nv"], t["kc"], t["vc"], t["sl"])
    S, Hq, D = case.query.shape
    mcl = case.max_context_len
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, mcl)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    q = t["q"].clone()
    out = torch.empty((S, Hq, D), dtype=torch.float32, device="cuda")
    pa.pa_decode(out, q, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.pa_decode(out, q, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws)
    rng = np.random.default_rng(6)
    for _ in range(3):
        qv = torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float32)).to(q.dtype).cuda()
        q.copy_(qv)
        g.replay()
        ref = torch.empty_like(out)
        pa.pa_decode(ref, qv, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(bits(out), bits(ref))
