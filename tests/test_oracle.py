"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things other than itself: library conversions
over every bit pattern of the element formats, torch's
``scaled_dot_product_attention`` in fp64 (the library routine for dense
softmax attention), closed forms, and invariances the paged layout must have
(permuting physical block ids, changing the block size).  Each test names the
mistake it would catch.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads


# ----------------------------------------------------------------------------- helpers

def _pool_from_dense(kd, vd, lens, bs, rng, extra_blocks=3, aliases=None):
    """Test-side scatter of logical per-sequence K/V ``[S][Hkv][Lmax][D]`` into a pool
    ``[NB][bs][Hkv][D]`` with shuffled physical block ids (free blocks stay NaN)."""
    S, Hkv, Lmax, D = kd.shape
    need = [math.ceil(int(L) / bs) for L in lens]
    NB = sum(need) + extra_blocks
    perm = rng.permutation(NB)
    kc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=kd.dtype)
    vc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=kd.dtype)
    bt = torch.full((S, max(1, max(need))), -1, dtype=torch.int32)
    o = 0
    for s in range(S):
        for b in range(need[s]):
            bt[s, b] = int(perm[o])
            o += 1
        for j in range(int(lens[s])):
            blk = int(bt[s, j // bs])
            kc[blk, j % bs] = kd[s, :, j, :]
            vc[blk, j % bs] = vd[s, :, j, :]
    return kc, vc, bt


def _sdpa_reference(q, kd, vd, qsl, lens, scale, Hq):
    """torch SDPA in fp64 per sequence; GQA by repeat_interleave; bottom-right causal mask."""
    S, Hkv, _, D = kd.shape
    G = Hq // Hkv
    out = torch.zeros(q.shape, dtype=torch.float64)
    for s in range(S):
        a, b = int(qsl[s]), int(qsl[s + 1])
        C, Lq = int(lens[s]), b - a
        if Lq == 0 or C == 0:
            continue
        qs = q[a:b].to(torch.float64).permute(1, 0, 2).unsqueeze(0)  # [1, Hq, Lq, D]
        ks = kd[s, :, :C].to(torch.float64).repeat_interleave(G, dim=0).unsqueeze(0)
        vs = vd[s, :, :C].to(torch.float64).repeat_interleave(G, dim=0).unsqueeze(0)
        i = torch.arange(Lq).unsqueeze(1)
        j = torch.arange(C).unsqueeze(0)
        mask = j <= (C - Lq + i)
        o = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=scale)
        out[a:b] = o[0].permute(1, 0, 2)
    return out


def _random_problem(seed, S, lens, qlens, Hq, Hkv, D, dtype):
    g = torch.Generator().manual_seed(seed)
    Lmax = max(lens)
    kd = torch.randn(S, Hkv, Lmax, D, generator=g).to(dtype)
    vd = torch.randn(S, Hkv, Lmax, D, generator=g).to(dtype)
    qsl = torch.tensor([0] + list(np.cumsum(qlens)), dtype=torch.int32)
    q = torch.randn(int(qsl[-1]), Hq, D, generator=g).to(dtype)
    cl = torch.tensor(lens, dtype=torch.int32)
    return q, kd, vd, qsl, cl


# ----------------------------------------------------------------------------- element formats

def test_bf16_decoder_matches_torch_on_every_pattern(oracle_mod):
    """Catches a wrong shift / sign / NaN handling in the bf16 widening."""
    raw = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode_elements(raw, oracle_mod.BF16)
    ref = torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_f16_decoder_matches_numpy_on_every_pattern(oracle_mod):
    """Catches a wrong exponent bias, subnormal scale or inf/NaN case in the fp16 widening."""
    raw = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode_elements(raw, oracle_mod.F16)
    ref = raw.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_f32_decoder_is_exact(oracle_mod):
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.4e38, 1e-45, np.inf, -np.inf, 1 / 3], dtype=np.float32)
    got = oracle_mod.decode_elements(vals, oracle_mod.F32)
    np.testing.assert_array_equal(got, vals.astype(np.float64))


# ----------------------------------------------------------------------------- cache write / copy

@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_reshape_and_cache_is_a_flat_slot_scatter(oracle_mod, dtype):
    """The pool is [NB*bs] token rows of Hkv*D (section 11's flat layout): slot s is row s.
    Catches block/offset swapped, a head-major pool, writes for skipped (negative) slots."""
    NB, bs, Hkv, D, T = 7, 8, 2, 64, 13
    g = torch.Generator().manual_seed(0)
    kc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=dtype)
    vc = kc.clone()
    key = torch.randn(T, Hkv, D, generator=g).to(dtype)
    val = torch.randn(T, Hkv, D, generator=g).to(dtype)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[3] = -1
    slots[9] = -5
    oracle_mod.reshape_and_cache(key, val, kc, vc, slots, bs)
    ek = torch.full((NB * bs, Hkv, D), float("nan"), dtype=dtype)
    ev = ek.clone()
    keep = slots >= 0
    ek[slots[keep]] = key[keep]
    ev[slots[keep]] = val[keep]
    assert torch.equal(kc.view(NB * bs, Hkv, D).view(torch.int16 if dtype != torch.float32 else torch.int32),
                       ek.view(torch.int16 if dtype != torch.float32 else torch.int32))
    assert torch.equal(vc.view(NB * bs, Hkv, D).view(torch.int16 if dtype != torch.float32 else torch.int32),
                       ev.view(torch.int16 if dtype != torch.float32 else torch.int32))


def test_reshape_and_cache_rejects_out_of_range_slot(oracle_mod):
    kc = torch.zeros(2, 8, 1, 64)
    with pytest.raises(ValueError):
        oracle_mod.reshape_and_cache(torch.zeros(1, 1, 64), torch.zeros(1, 1, 64), kc, kc.clone(),
                                     torch.tensor([16], dtype=torch.int64), 8)


def test_copy_blocks_matches_sequential_index_copy(oracle_mod):
    """Catches copying the wrong direction, only K, or a partial block."""
    NB, bs, Hkv, D = 9, 16, 2, 64
    g = torch.Generator().manual_seed(1)
    kc = torch.randn(NB, bs, Hkv, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, bs, Hkv, D, generator=g).to(torch.bfloat16)
    pairs = torch.tensor([[0, 5], [2, 7], [0, 8]], dtype=torch.int64)
    ek, ev = kc.clone(), vc.clone()
    for src, dst in pairs.tolist():
        ek[dst] = ek[src]
        ev[dst] = ev[src]
    oracle_mod.copy_blocks(kc, vc, pairs, bs)
    assert torch.equal(kc.view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), ev.view(torch.int16))


# ----------------------------------------------------------------------------- attention pins

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_dense_oracle_matches_torch_sdpa_fp64(oracle_mod, dtype):
    """Dense softmax attention against the library routine, decode and chunked rows.
    Catches a dropped scale, a transposed operand, a wrong GQA head map, a softmax without
    the max shift blowing up, and an off-by-one in the causal alignment."""
    S, Hq, Hkv, D = 3, 8, 2, 64
    lens, qlens = [5, 40, 17], [1, 9, 17]
    q, kd, vd, qsl, cl = _random_problem(10, S, lens, qlens, Hq, Hkv, D, dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle_mod.dense_attention(q, qsl, kd.double().numpy(), vd.double().numpy(), cl, scale)
    ref = _sdpa_reference(q, kd, vd, qsl, cl, scale, Hq).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_square_chunk_matches_sdpa_is_causal(oracle_mod):
    """With no cached prefix (Lq == C) bottom-right and top-left causal coincide: pin the
    mask to the library's own is_causal."""
    Hq, Hkv, D, L = 4, 4, 64, 23
    q, kd, vd, qsl, cl = _random_problem(11, 1, [L], [L], Hq, Hkv, D, torch.float32)
    scale = 0.125
    got = oracle_mod.dense_attention(q, qsl, kd.double().numpy(), vd.double().numpy(), cl, scale)
    ref = F.scaled_dot_product_attention(q.double().permute(1, 0, 2), kd[0].double(), vd[0].double(),
                                         is_causal=True, scale=scale).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_paged_oracle_equals_dense_bit_for_bit(oracle_mod, bs):
    """The gather through the block table reproduces the dense cache exactly.
    Catches a wrong block/offset split, a wrong kv-head stride, a missed ragged tail."""
    S, Hq, Hkv, D = 4, 8, 2, 64
    lens, qlens = [1, 33, 64, 70], [1, 5, 1, 70]
    q, kd, vd, qsl, cl = _random_problem(12 + bs, S, lens, qlens, Hq, Hkv, D, torch.bfloat16)
    rng = np.random.default_rng(bs)
    kc, vc, bt = _pool_from_dense(kd, vd, lens, bs, rng)
    scale = float(np.float32(1 / math.sqrt(D)))
    paged = oracle_mod.paged_attention(q, qsl, kc, vc, bt, cl, scale)
    dense = oracle_mod.dense_attention(q, qsl, kd.double().numpy(), vd.double().numpy(), cl, scale)
    np.testing.assert_array_equal(paged, dense)


def test_block_id_permutation_and_block_size_invariance(oracle_mod):
    """Same logical K/V under three shuffles and three block sizes: bit-identical outputs.
    Catches any dependence on physical placement."""
    S, Hq, Hkv, D = 3, 4, 2, 64
    lens, qlens = [29, 70, 8], [1, 1, 1]
    q, kd, vd, qsl, cl = _random_problem(20, S, lens, qlens, Hq, Hkv, D, torch.float16)
    outs = []
    for bs in (8, 16, 32):
        for seed in (0, 1, 2):
            kc, vc, bt = _pool_from_dense(kd, vd, lens, bs, np.random.default_rng(seed), extra_blocks=seed)
            outs.append(oracle_mod.paged_attention(q, qsl, kc, vc, bt, cl, 0.125))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_brute_force_every_context_length_1_to_40(oracle_mod, bs):
    """Every context length 1..40 (every tail shape of every block size) against SDPA."""
    Hq, Hkv, D = 4, 2, 64
    lens = list(range(1, 41))
    S = len(lens)
    q, kd, vd, qsl, cl = _random_problem(30 + bs, S, lens, [1] * S, Hq, Hkv, D, torch.bfloat16)
    kc, vc, bt = _pool_from_dense(kd, vd, lens, bs, np.random.default_rng(bs))
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle_mod.paged_attention(q, qsl, kc, vc, bt, cl, scale)
    ref = _sdpa_reference(q, kd, vd, qsl, cl, scale, Hq).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_closed_forms(oracle_mod):
    """Single key -> that value exactly; q = 0 -> mean of the visible values; scores
    differing by ln 3 -> weights 1/4 and 3/4; a dominant score -> that value."""
    Hq = Hkv = 1
    D, bs = 64, 8
    # single key
    g = torch.Generator().manual_seed(3)
    kd = torch.randn(1, 1, 1, D, generator=g)
    vd = torch.randn(1, 1, 1, D, generator=g)
    q = torch.randn(1, 1, D, generator=g)
    kc, vc, bt = _pool_from_dense(kd, vd, [1], bs, np.random.default_rng(0))
    qsl, cl = torch.tensor([0, 1], dtype=torch.int32), torch.tensor([1], dtype=torch.int32)
    out = oracle_mod.paged_attention(q, qsl, kc, vc, bt, cl, 0.125)
    np.testing.assert_array_equal(out[0, 0], vd[0, 0, 0].double().numpy())
    # q = 0 -> uniform weights
    L = 19
    kd = torch.randn(1, 1, L, D, generator=g)
    vd = torch.randn(1, 1, L, D, generator=g)
    kc, vc, bt = _pool_from_dense(kd, vd, [L], bs, np.random.default_rng(1))
    out = oracle_mod.paged_attention(torch.zeros(1, 1, D), qsl, kc, vc, bt,
                                     torch.tensor([L], dtype=torch.int32), 0.125)
    np.testing.assert_allclose(out[0, 0], vd[0, 0].double().mean(0).numpy(), rtol=0, atol=1e-14)
    # two keys, scale * q.k = 0 and ln 3 (k along e0, q = e0): weights 1/4, 3/4
    kd = torch.zeros(1, 1, 2, D, dtype=torch.float64)
    kd[0, 0, 1, 0] = math.log(3.0)
    vd = torch.randn(1, 1, 2, D, generator=g).double()
    qv = torch.zeros(1, 1, D, dtype=torch.float32)
    qv[0, 0, 0] = 1.0
    out = oracle_mod.dense_attention(qv, qsl, kd.numpy(), vd.numpy(),
                                     torch.tensor([2], dtype=torch.int32), 1.0)
    np.testing.assert_allclose(out[0, 0], (0.25 * vd[0, 0, 0] + 0.75 * vd[0, 0, 1]).numpy(),
                               rtol=0, atol=1e-15)
    # dominant score: one key aligned with q at scale 1, the others orthogonal
    kd = torch.zeros(1, 1, 5, D)
    kd[0, 0, 3, 0] = 60.0
    vd = torch.randn(1, 1, 5, D, generator=g)
    qv = torch.zeros(1, 1, D)
    qv[0, 0, 0] = 1.0
    kc, vc, bt = _pool_from_dense(kd, vd, [5], bs, np.random.default_rng(2))
    out = oracle_mod.paged_attention(qv, qsl, kc, vc, bt, torch.tensor([5], dtype=torch.int32), 1.0)
    np.testing.assert_allclose(out[0, 0], vd[0, 0, 3].double().numpy(), rtol=0, atol=1e-20)


def test_empty_context_gives_zeros_and_empty_chunk_is_noop(oracle_mod):
    Hq, Hkv, D, bs = 2, 1, 64, 8
    kc = torch.full((2, bs, Hkv, D), float("nan"))
    bt = torch.full((2, 1), -1, dtype=torch.int32)
    q = torch.randn(1, Hq, D)
    out = oracle_mod.paged_attention(q, torch.tensor([0, 1, 1], dtype=torch.int32), kc, kc.clone(),
                                     bt, torch.tensor([0, 5], dtype=torch.int32), 0.125)
    assert np.all(out == 0.0)


def test_bad_block_id_is_an_error_not_a_read(oracle_mod):
    kc = torch.zeros(2, 8, 1, 64)
    bt = torch.tensor([[0, 2]], dtype=torch.int32)  # block 2 does not exist
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(torch.zeros(1, 1, 64), torch.tensor([0, 1], dtype=torch.int32), kc,
                                   kc.clone(), bt, torch.tensor([12], dtype=torch.int32), 0.125)


# ----------------------------------------------------------------------------- generator

def test_generator_sentinels_and_tables():
    """Inputs are seeded (same bytes twice), every non-cached slot is NaN, every cached
    slot is finite, block ids are distinct and in range, and the fresh-token slots are
    NaN before the step (so a missed write shows up)."""
    a = workloads.tiny_decode()
    b = workloads.tiny_decode()
    assert torch.equal(a.key_cache.view(torch.int32), b.key_cache.view(torch.int32))
    c = a
    NB, bs = c.num_blocks, c.block_size
    used = c.block_tables[c.block_tables >= 0]
    assert len(set(used.tolist())) == used.numel() and int(used.max()) < NB
    flat = c.key_cache.view(NB * bs, -1)
    finite = torch.isfinite(flat).all(1)
    assert int(finite.sum()) == int(c.cached_lens.sum())
    assert not finite[c.slot_mapping].any()
    assert (c.context_lens.numpy() == c.cached_lens + 1).all()


def test_stress_generator_share_and_alias():
    c = workloads.make_decode_case("t", [40, 70, 90, 33, 64, 100, 8, 50, 77, 45], 8, 4, 2, 64,
                                   torch.bfloat16, 7, free_frac=0.2, share_frac=0.2, alias_frac=0.2)
    assert c.block_mapping is not None
    src, dst = c.block_mapping[:, 0], c.block_mapping[:, 1]
    assert len(set(dst.tolist())) == dst.numel()
    assert not set(dst.tolist()) & set(src.tolist())
    assert len(c.meta["aliased"]) == 2
