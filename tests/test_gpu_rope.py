"""Fused rotary embedding on the GPU against the fp64 reference: keys rotated on the way into
the cache (values copied bit for bit, skipped slots and NaN sentinels untouched), and decode
with the raw query rotated and scaled at its position against dense attention over exactly
rotated keys and queries."""
import numpy as np
import pytest
import torch

from oracle import rope as ref_rope
from paged_steps import MAX_ABS, MEAN_ABS, assert_attention_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu(cuda_ok):
    yield


def _table(rope_dim):
    import paged_kv_attention_write_gb300 as pa
    return pa.pa_rope_yarn_freqs(rope_dim, 1e6, 8.0, 4096, 32.0, 1.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rope_dim", [128, 64])
def test_reshape_and_cache_rope_writes_rotated_keys(dtype, rope_dim):
    import paged_kv_attention_write_gb300 as pa
    rng = np.random.default_rng(rope_dim)
    T, Hkv, D, bs, NB = 37, 4, 128, 16, 32
    key = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32)).to(dtype)
    val = torch.from_numpy(rng.standard_normal((T, Hkv, D)).astype(np.float32)).to(dtype)
    pos = rng.integers(0, 200000, size=T).astype(np.int32)
    pos[[0, 1, 2, 4]] = [(1 << 24) - 1, (1 << 23) + 3, 1 << 20, 0]   # the range the angle bound covers
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[[3, 20]] = -1                                   # padding tokens are skipped
    kc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=dtype)
    vc = kc.clone()
    freqs = _table(rope_dim)
    dev = "cuda"
    kd, vd = kc.to(dev), vc.to(dev)
    r = pa.Rope(torch.from_numpy(freqs).to(dev), rope_dim)
    pa.pa_reshape_and_cache_rope(key.to(dev), val.to(dev), kd, vd, torch.from_numpy(slots).to(dev),
                                 torch.from_numpy(pos).to(dev), r)
    torch.cuda.synchronize()
    kd, vd = kd.cpu().view(NB * bs, Hkv, D), vd.cpu().view(NB * bs, Hkv, D)
    want = ref_rope.apply_rope(key.double().numpy(), pos, freqs, rope_dim)
    live = slots >= 0
    got_k = kd[torch.from_numpy(slots[live])]
    assert torch.equal(bits(vd[torch.from_numpy(slots[live])]), bits(val[torch.from_numpy(live)]))
    untouched = np.setdiff1d(np.arange(NB * bs), slots[live])
    assert torch.isnan(kd[torch.from_numpy(untouched)]).all() and torch.isnan(vd[torch.from_numpy(untouched)]).all()
    ref = torch.from_numpy(want[live])
    if dtype == torch.float32:
        assert (got_k.double() - ref).abs().max().item() < 2e-6 * (1 + ref.abs().max().item())
    else:
        rounded = ref.to(dtype)                             # the reference rounded to the cache format
        ulps = (bits(got_k).to(torch.int32) - bits(rounded).to(torch.int32)).abs()
        assert ulps.max().item() <= 1 and (ulps == 0).float().mean().item() > 0.99
    # pairs past rope_dim are plain copies
    if rope_dim < D:
        assert torch.equal(bits(got_k[..., rope_dim:]), bits(key[torch.from_numpy(live)][..., rope_dim:]))


@pytest.mark.parametrize("dtype,D,G,rope_dim,beta,orig", [
    (torch.bfloat16, 128, 4, 128, 0.1, 512),    # query scale steps at 512, 1024, ...
    (torch.float16, 64, 8, 32, 0.0, 0),         # partial rotation, no query scale
    (torch.float32, 128, 1, 128, 0.25, 1000),
])
def test_decode_rope_matches_reference(oracle_mod, dtype, D, G, rope_dim, beta, orig):
    import paged_kv_attention_write_gb300 as pa
    rng = np.random.default_rng(D + G)
    Hkv, bs = 2, 16
    Hq = Hkv * G
    L = [1, 17, 530, 1500, 3001]
    S = len(L)
    nblk = [-(-n // bs) for n in L]
    NB = sum(nblk) + 7
    perm = rng.permutation(NB)
    bt = np.zeros((S, max(nblk)), dtype=np.int32)
    o = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[o:o + n]
        o += n
    kraw = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in L]
    vraw = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in L]
    q = torch.from_numpy(rng.standard_normal((S, Hq, D)).astype(np.float32)).to(dtype)
    freqs = _table(rope_dim)
    dev = "cuda"
    kc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=dtype, device=dev)
    vc = kc.clone()
    r = pa.Rope(torch.from_numpy(freqs).to(dev), rope_dim, beta, orig)
    # every key goes through the rotating cache write, at its position
    for s, n in enumerate(L):
        p = np.arange(n)
        slots = bt[s, p // bs].astype(np.int64) * bs + p % bs
        pa.pa_reshape_and_cache_rope(torch.from_numpy(kraw[s]).to(dtype).to(dev),
                                     torch.from_numpy(vraw[s]).to(dtype).to(dev), kc, vc,
                                     torch.from_numpy(slots).to(dev), torch.from_numpy(p.astype(np.int32)).to(dev), r)
    cl = torch.tensor(L, dtype=torch.int32, device=dev)
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, pa.pa_decode_workspace_size(S, Hq, Hkv, D, max(L))), dtype=torch.uint8, device=dev)
    scale = 1.0 / D ** 0.5
    pa.pa_decode_rope(out, q.to(dev), kc, vc, torch.from_numpy(bt).to(dev), cl, max(L), scale, r, workspace=ws)
    torch.cuda.synchronize()
    # reference: exact rotation of the stored-format keys and of the query, query scale
    Lm = max(L)
    kd = np.zeros((S, Hkv, Lm, D))
    vd = np.zeros((S, Hkv, Lm, D))
    for s, n in enumerate(L):
        k_in = torch.from_numpy(kraw[s]).to(dtype).double().numpy()
        kd[s, :, :n] = ref_rope.apply_rope(k_in, np.arange(n), freqs, rope_dim).transpose(1, 0, 2)
        vd[s, :, :n] = torch.from_numpy(vraw[s]).to(dtype).double().numpy().transpose(1, 0, 2)
    qpos = np.array(L) - 1
    qr = ref_rope.apply_rope(q.double().numpy(), qpos, freqs, rope_dim) * ref_rope.q_scale(qpos, beta, orig)[:, None, None]
    ref = oracle_mod.dense_attention(torch.from_numpy(qr.astype(np.float32)), torch.arange(S + 1, dtype=torch.int32),
                                     kd, vd, torch.tensor(L, dtype=torch.int32), scale)
    assert_attention_close(out.cpu(), ref, MAX_ABS, MEAN_ABS)
