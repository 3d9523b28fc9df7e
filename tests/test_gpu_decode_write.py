"""The fused cache write + decode (pa_decode_write) against the two calls it replaces,
pa_reshape_and_cache of each sequence's new token and pa_decode, on the same inputs: the
output and both pools bit for bit, across cache types, head dims, group sizes, block sizes,
kv-head groups of four (two token slices per stage), many short sequences (several segment
ends per CTA) and padding slots; and one case against the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads
from paged_steps import assert_attention_close, bits, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _both(case, pad=(), past=(), want_status=0):
    """[(out, key pool, value pool) of the two calls, the same of the fused call] for a decode
    case whose new tokens are not yet in the pools; the sequences in `pad` get slot -1 (nothing
    written), those in `past` a slot past the pool (reported, nothing written)."""
    import paged_kv_attention_write_gb300 as pa
    dev = "cuda"
    slots = case.slot_mapping.clone()
    for s in pad:
        slots[s] = -1
    for s in past:
        slots[s] = case.key_cache.shape[0] * case.block_size + 3 + s
    q, nk, nv = case.query.to(dev), case.new_key.to(dev), case.new_value.to(dev)
    bt, cl, sl = case.block_tables.to(dev), case.context_lens.to(dev), slots.to(dev)
    S, Hq, D = case.query.shape
    mcl = case.max_context_len
    n = pa.pa_decode_workspace_size(S, case.num_heads, case.num_kv_heads, D, mcl)
    res = []
    for fused in (False, True):
        kc, vc = case.key_cache.to(dev), case.value_cache.to(dev)
        out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=dev)
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if fused:
            pa.pa_decode_write(out, q, nk, nv, sl, kc, vc, bt, cl, mcl, case.scale, workspace=ws, status=status)
        else:
            pa.pa_reshape_and_cache(nk, nv, kc, vc, sl, status=status)
            pa.pa_decode(out, q, kc, vc, bt, cl, mcl, case.scale, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert status.item() == want_status
        res.append((out.cpu(), kc.cpu(), vc.cpu()))
    return res


def _same(res):
    (o1, k1, v1), (o2, k2, v2) = res
    assert torch.equal(bits(o1), bits(o2))
    assert torch.equal(bits(k1), bits(k2)) and torch.equal(bits(v1), bits(v2))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_decode_write_equals_write_then_decode(dtype, D, G):
    rng = np.random.default_rng(100 + D + G)
    lens = [int(x) for x in rng.integers(1, 3000, size=24)] + [0, 4095]
    case = workloads.make_decode_case("dw", lens, 16, 8 * G, 8, D, dtype, 7 + G)
    _same(_both(case))


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_decode_write_block_sizes_and_padding(bs):
    rng = np.random.default_rng(bs)
    lens = [int(x) for x in rng.integers(0, 5000, size=40)]
    case = workloads.make_decode_case("dwb", lens, bs, 32, 8, 128, torch.bfloat16, bs)
    _same(_both(case, pad=(1, 7, 30)))


def test_decode_write_four_kv_heads_two_token_slices():
    rng = np.random.default_rng(4)
    lens = [int(x) for x in rng.integers(1, 6000, size=20)]
    case = workloads.make_decode_case("dw4", lens, 16, 16, 4, 128, torch.bfloat16, 4)
    _same(_both(case))


def test_decode_write_many_short_sequences():
    """256 sequences of 1-200 tokens: most CTAs end several segments."""
    rng = np.random.default_rng(256)
    lens = [int(x) for x in rng.integers(0, 200, size=256)]
    case = workloads.make_decode_case("dws", lens, 16, 32, 8, 128, torch.float16, 256)
    _same(_both(case))


def test_decode_write_against_oracle(oracle_mod):
    case = workloads.decode_batch()
    res = _both(case)
    _same(res)
    ref, okc, ovc = oracle_step(case, oracle_mod)
    assert_attention_close(res[1][0], ref)
    assert torch.equal(bits(res[1][1]), bits(okc)) and torch.equal(bits(res[1][2]), bits(ovc))


def test_decode_write_reports_a_slot_past_the_pool():
    """A slot past the pool is reported (PA_DEVERR_SLOT) and not written by either path; the
    attention then reads what the cache holds there, the same in both."""
    rng = np.random.default_rng(9)
    lens = [int(x) for x in rng.integers(1, 2000, size=12)]
    case = workloads.make_decode_case("dwbad", lens, 16, 32, 8, 128, torch.bfloat16, 9)
    _same(_both(case, past=(2, 7), want_status=1))
