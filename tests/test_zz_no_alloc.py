"""pa_decode_noalloc: decode for callers that cannot allocate device memory (plugin
hosts that own all device memory, hot paths where cudaMalloc could synchronise the
device, bindings without an allocator).  Its scratch is a static array inside the
library, shared by every call.

The test calls the C entry point directly (ctypes) and checks its output against
pa_decode with a caller workspace and against the fp64 oracle, within the parity
tolerance, on two calls in a row with different problems, so that the first call's
leftover scratch cannot leak into the second.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads
from paged_steps import MAX_ABS, MEAN_ABS, assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _device_case(case, dev="cuda"):
    import paged_kv_attention_write_gb300 as pa
    kc, vc = case.key_cache.to(dev), case.value_cache.to(dev)
    pa.pa_reshape_and_cache(case.new_key.to(dev), case.new_value.to(dev), kc, vc,
                            case.slot_mapping.to(dev))
    return dict(q=case.query.to(dev), kc=kc, vc=vc, bt=case.block_tables.to(dev),
                cl=case.context_lens.to(dev))


def _noalloc_c_call(lib, out, t, case, status):
    """pa_decode_noalloc through the C ABI (raw pointers and sizes)."""
    S, Hq, D = case.query.shape
    NB, bs, Hkv, _ = case.key_cache.shape
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.pa_decode_noalloc
    fn.argtypes = [vp, i, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f, i, vp, vp]
    fn.restype = i
    return fn(out.data_ptr(), 0, t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
              t["bt"].data_ptr(), t["bt"].shape[1], t["cl"].data_ptr(), case.max_context_len,
              S, Hq, Hkv, D, bs, NB, case.scale, {torch.bfloat16: 2, torch.float16: 1,
                                                 torch.float32: 0}[case.dtype],
              status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _workspace_decode(case, t):
    import paged_kv_attention_write_gb300 as pa
    out = torch.empty(tuple(case.query.shape), dtype=torch.float32, device="cuda")
    n = pa.pa_decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                    case.head_dim, case.max_context_len)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    pa.pa_decode(out, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], case.max_context_len,
                 case.scale, workspace=ws)
    return out


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(oracle_mod):
    import paged_kv_attention_write_gb300 as pa
    lib = ctypes.CDLL(str(pa.library_path()))
    cases = [workloads.decode_batch(),
             workloads.make_decode_case("noalloc-2", [3000, 0, 17, 9000, 640], 16, 32, 8, 128,
                                        torch.bfloat16, 31, free_frac=0.2)]
    cases[1].context_lens[1] = 0   # a sequence with nothing to attend
    cases[1].slot_mapping[1] = -1
    for case in cases:
        t = _device_case(case)
        ref = _workspace_decode(case, t)
        out = torch.full(tuple(case.query.shape), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc_c_call(lib, out, t, case, status) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        d = (out - ref).abs()
        assert torch.isfinite(out).all()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS
        oracle_ref, _, _ = oracle_step(case, oracle_mod)
        assert_attention_close(out.cpu(), oracle_ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import paged_kv_attention_write_gb300 as pa
    lib = ctypes.CDLL(str(pa.library_path()))
    S = 4096  # far more partials than the static array holds
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.pa_decode_noalloc
    fn.argtypes = [vp, i, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f, i, vp, vp]
    fn.restype = i
    p = dummy.data_ptr()
    rc = fn(p, 0, p, p, p, p, 1, p, 32, S, 32, 8, 128, 32, 1, 0.088, 2, None, None)
    assert rc == -3  # PA_ERR_WORKSPACE, nothing launched
