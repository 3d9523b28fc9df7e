"""Run one paged-attention step of a generated case on the GPU (through the C ABI)
and on the oracle, and compare.

GPU side: copy_blocks (if the case shares prefixes) -> reshape_and_cache of the
fresh tokens -> decode or prefill.  Oracle side: the same three steps on host
copies of the pools.  Tolerances for attention: max-abs 5e-3 and mean-abs
5e-4 against the fp64 oracle rounded to fp32; cache writes and copies must
match bit for bit.
"""
from __future__ import annotations

import os

import numpy as np
import torch

MAX_ABS = 5e-3
MEAN_ABS = 5e-4

# (test id, max-abs, mean-abs) of every attention comparison of the session; conftest
# writes them to the JSON file named by PA_PARITY_LOG at the end of the session, so the
# margin of each case against the tolerance can be followed from run to run.
RECORDS: list = []


def bits(t: torch.Tensor) -> torch.Tensor:
    """Integer view of a float tensor, so NaN sentinels compare bit for bit."""
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


def gpu_step(case, out_dtype=torch.float32, device="cuda", status=None):
    import paged_kv_attention_write_gb300 as pa
    kc = case.key_cache.to(device)
    vc = case.value_cache.to(device)
    bt = case.block_tables.to(device)
    cl = case.context_lens.to(device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=device)
    if case.block_mapping is not None:
        pa.pa_copy_blocks(kc, vc, case.block_mapping.to(device), status=status)
    pa.pa_reshape_and_cache(case.new_key.to(device), case.new_value.to(device), kc, vc,
                            case.slot_mapping.to(device), status=status)
    q = case.query.to(device)
    out = torch.full(tuple(q.shape), float("nan"), dtype=out_dtype, device=device)
    if case.is_decode:
        nbytes = pa.pa_decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                             case.head_dim,
                                             case.max_context_len)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        pa.pa_decode(out, q, kc, vc, bt, cl, case.max_context_len, case.scale, workspace=ws,
                     status=status)
    else:
        qsl = case.query_start_loc.to(device)
        mq = int((case.query_start_loc[1:] - case.query_start_loc[:-1]).max())
        pa.pa_prefill_chunk(out, q, qsl, mq, kc, vc, bt, cl, case.max_context_len, case.scale,
                            status=status)
    torch.cuda.synchronize()
    return out.cpu(), kc.cpu(), vc.cpu(), int(status.item())


def oracle_step(case, oracle):
    kc = case.key_cache.clone()
    vc = case.value_cache.clone()
    if case.block_mapping is not None:
        oracle.copy_blocks(kc, vc, case.block_mapping, case.block_size)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping,
                             case.block_size)
    ref = oracle.paged_attention(case.query, case.query_start_loc, kc, vc, case.block_tables,
                                 case.context_lens, case.scale)
    return ref, kc, vc


def oracle_step_pools(case, oracle):
    """The oracle's pools after the case's block copies and cache write (no attention)."""
    kc = case.key_cache.clone()
    vc = case.value_cache.clone()
    if case.block_mapping is not None:
        oracle.copy_blocks(kc, vc, case.block_mapping, case.block_size)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, case.block_size)
    return None, kc, vc


def attention_errors(got: torch.Tensor, ref: np.ndarray):
    g = got.float().numpy().astype(np.float64)
    r = ref.astype(np.float32).astype(np.float64)
    assert np.isfinite(g).all(), "non-finite attention output"
    d = np.abs(g - r)
    return float(d.max()), float(d.mean())


def record_errors(mx: float, mn: float, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.append({"test": test, "max_abs": mx, "mean_abs": mn, "max_abs_bound": max_abs,
                    "mean_abs_bound": mean_abs})


def assert_attention_close(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    mx, mn = attention_errors(got, ref)
    record_errors(mx, mn, max_abs, mean_abs)
    assert mx <= max_abs and mn <= mean_abs, f"max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    return mx, mn


def check_case(case, oracle, out_dtype=torch.float32, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    out, kc, vc, status = gpu_step(case, out_dtype)
    ref, okc, ovc = oracle_step(case, oracle)
    assert status == 0, f"device status {status}"
    assert torch.equal(bits(kc), bits(okc)), "key cache differs from the oracle's"
    assert torch.equal(bits(vc), bits(ovc)), "value cache differs from the oracle's"
    return assert_attention_close(out, ref, max_abs, mean_abs)
