"""Decode captured into a CUDA graph: every replay, with new queries (and new tokens for the
fused write) copied into the captured buffers, equals an eager call on the same inputs bit
for bit.  A captured launch carries one fixed set of arguments on every replay, so nothing in
the result may depend on a per-call value the replay does not renew."""
import numpy as np
import pytest
import torch

import workloads
from paged_steps import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _inputs(seed):
    case = workloads.decode_batch(seed)
    dev = "cuda"
    return case, {"kc": case.key_cache.to(dev), "vc": case.value_cache.to(dev), "bt": case.block_tables.to(dev),
                  "cl": case.context_lens.to(dev), "sl": case.slot_mapping.to(dev)}


def test_decode_graph_replays_equal_eager_calls():
    import paged_kv_attention_write_gb300 as pa
    case, t = _inputs(5)
    pa.pa_reshape_and_cache(case.new_key.cuda(), case.new_value.cuda(), t["kc"], t["vc"], t["sl"])
    S, Hq, D = case.query.shape
    mcl = case.max_context_len
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, mcl)
    ws, ws_eager = torch.empty(n, dtype=torch.uint8, device="cuda"), torch.empty(n, dtype=torch.uint8, device="cuda")
    q = case.query.cuda().clone()
    out = torch.empty((S, Hq, D), dtype=torch.float32, device="cuda")
    pa.pa_decode(out, q, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws)  # first call: eager
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.pa_decode(out, q, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws)
    rng = np.random.default_rng(5)
    for _ in range(4):
        qv = torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float32)).to(q.dtype).cuda()
        q.copy_(qv)
        g.replay()
        ref = torch.empty_like(out)
        pa.pa_decode(ref, qv, t["kc"], t["vc"], t["bt"], t["cl"], mcl, case.scale, workspace=ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(bits(out), bits(ref))


def test_decode_write_graph_replays_equal_eager_calls():
    import paged_kv_attention_write_gb300 as pa
    case, t = _inputs(6)
    case2, t2 = _inputs(6)  # the pools the eager calls write
    S, Hq, D = case.query.shape
    mcl = case.max_context_len
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, mcl)
    ws, ws_eager = torch.empty(n, dtype=torch.uint8, device="cuda"), torch.empty(n, dtype=torch.uint8, device="cuda")
    q, nk, nv = case.query.cuda().clone(), case.new_key.cuda().clone(), case.new_value.cuda().clone()
    out = torch.empty((S, Hq, D), dtype=torch.float32, device="cuda")
    args = lambda o, qq, kk, vv, tt, w: pa.pa_decode_write(o, qq, kk, vv, tt["sl"], tt["kc"], tt["vc"], tt["bt"],
                                                          tt["cl"], mcl, case.scale, workspace=w)
    args(out, q, nk, nv, t, ws)  # first call: eager
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        args(out, q, nk, nv, t, ws)
    rng = np.random.default_rng(6)
    for _ in range(4):
        new = [torch.from_numpy(rng.standard_normal(tuple(x.shape)).astype(np.float32)).to(x.dtype).cuda()
               for x in (q, nk, nv)]
        for dst, src in zip((q, nk, nv), new):
            dst.copy_(src)
        g.replay()
        ref = torch.empty_like(out)
        args(ref, *new, t2, ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(bits(out), bits(ref))
        assert torch.equal(bits(t["kc"]), bits(t2["kc"])) and torch.equal(bits(t["vc"]), bits(t2["vc"]))
