// prefill.cu -- chunked-prefill paged attention on the tensor cores.
//
// A chunk of Lq query tokens per sequence (the newest tokens, whose K/V the
// caller already wrote into the cache) attends the sequence's keys gathered
// through its block table: full attention over the cached prefix, causal
// inside the chunk, rows aligned bottom-right (row i at absolute position
// C - Lq + i).  mistral.rs page, scheduling section (long prompts chunked
// under a token budget, 512 tokens per chunk); TensorSharp "Mistral 3" page,
// section 11 (paged K/V gather, then fused attention).
//
// Grid (query tile, kv head, sequence).  A query tile is 64 rows of
// (token, head) pairs of ONE kv head's G query heads, so every K/V tile
// gathered into shared memory serves G heads.  Four warps own 16 rows each.
// Per 64-key tile: S = Q K^T and O += P V with mma.sync m16n8k16 (fp32
// accumulate), online softmax in registers in the log2 domain, cp.async
// double buffering of the gathered K/V rows (zero-filled past the context).
#include "common.cuh"

namespace pa {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kBM = 64;  // query rows per CTA (16 per warp)
constexpr int kBN = 64;  // keys per tile

template <class T>
struct MmaType;
template <>
struct MmaType<F16> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};
template <>
struct MmaType<BF16> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// 16-byte async copy; src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// Shared-memory tile of R rows x D 16-bit elements; the 16-byte chunk c of row
// `row` is stored at chunk c ^ (row % 8) so that ldmatrix's 8-row phases hit
// distinct banks.
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
    return base + (uint32_t)(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

struct PrefillParams {
    void *out;
    pa_dtype out_dtype;
    const void *query;
    const int32_t *query_start_loc;
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int max_blocks_per_seq, num_heads, num_kv_heads, block_size, num_blocks, max_context_len;
    int num_tokens;
    float qk_scale_log2;
    int32_t *status;
};

template <class OutT>
__device__ __forceinline__ void store2(void *out, int64_t idx, float a, float b) {
    store_out(static_cast<OutT *>(out) + idx, a, b);
}

template <class T, int D, int G>
__global__ void __launch_bounds__(kPfThreads)
prefill_kernel(const PrefillParams p) {
    constexpr int TT = kBM / G;        // query tokens per tile
    constexpr int CH = D / 8;          // 16-byte chunks per row
    constexpr int KS = D / 16;         // k-steps over the head dim
    constexpr int NTS = kBN / 8;       // n-tiles of S per warp
    constexpr int NTO = D / 8;         // n-tiles of O per warp
    using Elt = typename T::storage;
    using M = MmaType<T>;

    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sQ = (uint32_t)__cvta_generic_to_shared(smem);
    const uint32_t sK0 = sQ + kBM * D * 2;
    const uint32_t sV0 = sK0 + 2 * kBN * D * 2;

    pdl_wait_previous();
    pdl_launch_dependents();
    const int g = blockIdx.y, s = blockIdx.z;
    const int qt = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) tiles first
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int Hq = p.num_heads, Hkv = p.num_kv_heads, bs = p.block_size;

    const int q0 = p.query_start_loc[s];
    const int Lq = p.query_start_loc[s + 1] - q0;
    int C = p.context_lens[s];
    if (q0 < 0 || Lq < 0 || (int64_t)q0 + Lq > p.num_tokens) {  // never index past the query
        if (tid == 0 && blockIdx.x == 0 && g == 0) report(p.status, PA_DEVERR_QUERY);
        return;
    }
    if (qt * TT >= Lq) return;
    const int cap = min(p.max_blocks_per_seq * bs, p.max_context_len);
    if (C > cap || Lq > C) {
        if (tid == 0 && qt * TT == 0 && g == 0) report(p.status, C > cap ? PA_DEVERR_CONTEXT : PA_DEVERR_QUERY);
        if (C > cap) C = cap;
        if (Lq > C) return;
    }
    const int tok_begin = qt * TT;
    const int tok_end = min(Lq, tok_begin + TT);
    const int pos0 = C - Lq;                        // absolute position of chunk row 0
    const int kv_end = pos0 + tok_end;              // keys visible to the tile's last row
    const int n_tiles = (kv_end + kBN - 1) / kBN;

    const Elt *kc = static_cast<const Elt *>(p.key_cache);
    const Elt *vc = static_cast<const Elt *>(p.value_cache);
    const int32_t *bt = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
    const int64_t slot_stride = (int64_t)Hkv * D;

    // ---- Q tile: row r = (token tok_begin + r / G, head g*G + r % G)
    {
        const Elt *qbase = static_cast<const Elt *>(p.query);
        for (int i = tid; i < kBM * CH; i += kPfThreads) {
            const int row = i / CH, ch = i % CH;
            const int tok = tok_begin + row / G;
            const bool ok = tok < Lq;
            const Elt *src = qbase + ((int64_t)(q0 + (ok ? tok : 0)) * Hq + g * G + row % G) * D + ch * 8;
            cp_async16(swz<D>(sQ, row, ch), src, ok ? 16 : 0);
        }
    }
    // ---- K/V tile loader: 64 gathered key rows, zero past the context or on a bad block id
    auto load_kv = [&](int tile, int buf) {
        const int k0 = tile * kBN;
        const uint32_t sK = sK0 + buf * kBN * D * 2, sV = sV0 + buf * kBN * D * 2;
        for (int i = tid; i < kBN * CH; i += kPfThreads) {
            const int row = i / CH, ch = i % CH;
            const int j = k0 + row;
            int64_t off = 0;
            int bytes = 0;
            if (j < C) {
                const int blk = bt[j / bs];
                if (blk >= 0 && blk < p.num_blocks) {
                    off = ((int64_t)blk * bs + j % bs) * slot_stride + g * D + ch * 8;
                    bytes = 16;
                } else if (ch == 0) {
                    report(p.status, PA_DEVERR_BLOCK_ID);
                }
            }
            cp_async16(swz<D>(sK, row, ch), kc + off, bytes);
            cp_async16(swz<D>(sV, row, ch), vc + off, bytes);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // Rows this thread holds in the accumulator fragments.
    const int row_a = warp * 16 + lane / 4;
    const int pos_a = pos0 + tok_begin + row_a / G;
    const int pos_b = pos0 + tok_begin + (row_a + 8) / G;

    uint32_t qa[KS][4];
    float o[NTO][4];
#pragma unroll
    for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int tile = 0; tile < n_tiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < n_tiles) load_kv(tile + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (tile == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int m = lane / 8;
                const int row = warp * 16 + (m % 2) * 8 + lane % 8;
                ldmatrix_x4(qa[ks], swz<D>(sQ, row, ks * 2 + m / 2));
            }
        }
        const uint32_t sK = sK0 + buf * kBN * D * 2, sV = sV0 + buf * kBN * D * 2;
        // ---- S = Q K^T (16 rows x 64 keys per warp)
        float sc[NTS][4];
#pragma unroll
        for (int n = 0; n < NTS; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {
                uint32_t b[4];
                const int m = lane / 8;
                ldmatrix_x4(b, swz<D>(sK, n * 8 + lane % 8, ks * 2 + m));
                M::mma(sc[n], qa[ks], b[0], b[1]);
                M::mma(sc[n], qa[ks + 1], b[2], b[3]);
            }
        }
        // ---- mask, online softmax (log2 domain)
        const int k0 = tile * kBN;
        const bool need_mask = k0 + kBN - 1 > pos0 + tok_begin + warp * 16 / G || k0 + kBN > C;
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int j = k0 + n * 8 + (lane % 4) * 2 + c;
                float sa = sc[n][c] * p.qk_scale_log2;
                float sb = sc[n][2 + c] * p.qk_scale_log2;
                if (need_mask) {
                    if (j > pos_a || j >= C) sa = -INFINITY;
                    if (j > pos_b || j >= C) sb = -INFINITY;
                }
                sc[n][c] = sa;
                sc[n][2 + c] = sb;
                mx_a = fmaxf(mx_a, sa);
                mx_b = fmaxf(mx_b, sb);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, off));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
        const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
        const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
        m_a = mn_a;
        m_b = mn_b;
        float rs_a = 0.f, rs_b = 0.f;
        uint32_t pa[NTS][2];
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const float p0 = exp2f(sc[n][0] - base_a), p1 = exp2f(sc[n][1] - base_a);
            const float p2 = exp2f(sc[n][2] - base_b), p3 = exp2f(sc[n][3] - base_b);
            rs_a += p0 + p1;
            rs_b += p2 + p3;
            pa[n][0] = M::pack(p0, p1);
            pa[n][1] = M::pack(p2, p3);
        }
        l_a = l_a * al_a + rs_a;
        l_b = l_b * al_b + rs_b;
#pragma unroll
        for (int n = 0; n < NTO; ++n) {
            o[n][0] *= al_a;
            o[n][1] *= al_a;
            o[n][2] *= al_b;
            o[n][3] *= al_b;
        }
        // ---- O += P V
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t a[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
            for (int n = 0; n < NTO; n += 2) {
                uint32_t b[4];
                const int m = lane / 8;
                ldmatrix_x4_trans(b, swz<D>(sV, kk * 16 + (m % 2) * 8 + lane % 8, n + m / 2));
                M::mma(o[n], a, b[0], b[1]);
                M::mma(o[n + 1], a, b[2], b[3]);
            }
        }
        __syncthreads();  // this buffer is refilled two tiles later
    }
    cp_async_wait<0>();

    // ---- row sums across the quad, normalise, store
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_a += __shfl_xor_sync(kFullMask, l_a, off);
        l_b += __shfl_xor_sync(kFullMask, l_b, off);
    }
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    const int tok_a = tok_begin + row_a / G, tok_b = tok_begin + (row_a + 8) / G;
    const int64_t oa = ((int64_t)(q0 + tok_a) * Hq + g * G + row_a % G) * D;
    const int64_t ob = ((int64_t)(q0 + tok_b) * Hq + g * G + (row_a + 8) % G) * D;
#pragma unroll
    for (int n = 0; n < NTO; ++n) {
        const int d = n * 8 + (lane % 4) * 2;
        if (tok_a < Lq) {
            if (p.out_dtype == PA_F32) store2<float>(p.out, oa + d, o[n][0] * inv_a, o[n][1] * inv_a);
            else if (p.out_dtype == PA_F16) store2<__half>(p.out, oa + d, o[n][0] * inv_a, o[n][1] * inv_a);
            else store2<__nv_bfloat16>(p.out, oa + d, o[n][0] * inv_a, o[n][1] * inv_a);
        }
        if (tok_b < Lq) {
            if (p.out_dtype == PA_F32) store2<float>(p.out, ob + d, o[n][2] * inv_b, o[n][3] * inv_b);
            else if (p.out_dtype == PA_F16) store2<__half>(p.out, ob + d, o[n][2] * inv_b, o[n][3] * inv_b);
            else store2<__nv_bfloat16>(p.out, ob + d, o[n][2] * inv_b, o[n][3] * inv_b);
        }
    }
}

template <class T, int D, int G>
int launch_typed(const PrefillParams &prm, int max_query_len, int num_seqs, cudaStream_t st) {
    constexpr int TT = kBM / G;
    const int smem = (kBM + 4 * kBN) * D * 2;
    static bool configured = false;  // attribute set once per process (per instantiation)
    if (!configured) {
        if (cudaFuncSetAttribute(prefill_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem) != cudaSuccess)
            return PA_ERR_CUDA;
        configured = true;
    }
    dim3 grid((max_query_len + TT - 1) / TT, prm.num_kv_heads, num_seqs);
    return launch_pdl(prefill_kernel<T, D, G>, grid, dim3(kPfThreads), smem, st, prm) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

template <class T, int D>
int dispatch_g(const PrefillParams &prm, int G, int mq, int S, cudaStream_t st) {
    switch (G) {
        case 1: return launch_typed<T, D, 1>(prm, mq, S, st);
        case 2: return launch_typed<T, D, 2>(prm, mq, S, st);
        case 4: return launch_typed<T, D, 4>(prm, mq, S, st);
        case 8: return launch_typed<T, D, 8>(prm, mq, S, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

template <class T>
int dispatch_d(const PrefillParams &prm, int D, int G, int mq, int S, cudaStream_t st) {
    switch (D) {
        case 64: return dispatch_g<T, 64>(prm, G, mq, S, st);
        case 128: return dispatch_g<T, 128>(prm, G, mq, S, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_prefill(const PrefillArgs &a) {
    if (a.num_seqs == 0 || a.num_tokens == 0 || a.max_query_len == 0) return PA_OK;
    PrefillParams prm{};
    prm.out = a.out;
    prm.out_dtype = a.out_dtype;
    prm.query = a.query;
    prm.query_start_loc = a.query_start_loc;
    prm.key_cache = a.key_cache;
    prm.value_cache = a.value_cache;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.max_blocks_per_seq = a.max_blocks_per_seq;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.block_size = a.block_size;
    prm.num_blocks = a.num_blocks;
    prm.max_context_len = a.max_context_len;
    prm.num_tokens = a.num_tokens;
    prm.qk_scale_log2 = a.scale * kLog2e;
    prm.status = a.status;
    const int G = a.num_heads / a.num_kv_heads;
    switch (a.kv_dtype) {
        case PA_F16: return dispatch_d<F16>(prm, a.head_dim, G, a.max_query_len, a.num_seqs, a.stream);
        case PA_BF16: return dispatch_d<BF16>(prm, a.head_dim, G, a.max_query_len, a.num_seqs, a.stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace pa
