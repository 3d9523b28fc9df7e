// decode.cu -- paged decode attention: split-K over the context, then a
// log-sum-exp reduce of the partial results.
//
// One query token per sequence attends every cached key of its sequence,
// gathered through the block table (TensorSharp "Mistral 3" page, section 11:
// per-sequence paged attention over the paged K/V buffer; sections 3 / 4.1:
// causal GQA attention with Q scaled by 1/sqrt(headDim)).
//
// Pass 1, grid (partition, kv head, sequence): a CTA streams the keys and
// values of one kv head over one partition of the context once, and serves
// all G = Hq / Hkv query heads that read that kv head.  Each warp keeps an
// online softmax (running max m, running sum l, unnormalised output acc) in
// the log2 domain.  Lanes own 16-byte slices of the head dimension; the q.k
// partial dot products of a batch of tokens are reduce-scattered across the
// lanes of a token row, so every lane finishes with whole scores.
// Pass 2, grid (sequence, q head): merges the partitions' (m, l, acc).
#include "common.cuh"

namespace pa {
namespace {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kPartition = 512;  // tokens per split-K partition
constexpr int kWarpSpan = kPartition / kDecodeWarps;

template <class T, int D, int G, int NT>
struct DecodeShape {
    static constexpr int EPV = T::kPerVec;        // elements per 16-byte vector
    static constexpr int LPT = D / EPV;           // lanes covering one token row
    static constexpr int TPW = 32 / LPT;          // token rows per warp step
    static constexpr int NTG = NT / TPW;          // tokens per lane group per batch
    static constexpr int NV = NTG * G;            // partial dot products per lane
    static_assert(LPT >= 1 && LPT <= 32 && 32 % LPT == 0, "head row must span 1..32 lanes");
    static_assert(NT % TPW == 0, "batch must be whole warp steps");
    static_assert(kWarpSpan % NT == 0, "warp span must be whole batches");
};

// Reduce-scatter of v[0..N) across the lanes that differ in bits OFF, OFF/2, .., 1.
// After it, lane r (index within its row group) holds the full sums of original
// entries r*NV/LPT .. (+ max(NV/LPT, 1) - 1) in v[0..).
template <int NV, int N, int OFF>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane) {
    if constexpr (OFF >= 1) {
        if constexpr (N > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float keep = upper ? v[i + N / 2] : v[i];
                const float send = upper ? v[i] : v[i + N / 2];
                v[i] = keep + __shfl_xor_sync(kFullMask, send, OFF);
            }
            reduce_scatter<NV, N / 2, OFF / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFullMask, v[0], OFF);
            reduce_scatter<NV, 1, OFF / 2>(v, lane);
        }
    }
}

template <class OutT>
__device__ __forceinline__ void store_pair(void *out, int64_t idx, float a, float b) {
    store_out(static_cast<OutT *>(out) + idx, a, b);
}

__device__ __forceinline__ void store_pair_any(void *out, pa_dtype dt, int64_t idx, float a,
                                               float b) {
    if (dt == PA_F32)
        store_pair<float>(out, idx, a, b);
    else if (dt == PA_F16)
        store_pair<__half>(out, idx, a, b);
    else
        store_pair<__nv_bfloat16>(out, idx, a, b);
}

struct DecodeParams {
    void *out;
    pa_dtype out_dtype;
    const void *query;
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part_o;  // [S][Hq][NP][D]
    float *part_m;  // [S][Hq][NP]
    float *part_l;  // [S][Hq][NP]
    int max_blocks_per_seq, num_partitions, num_heads, num_kv_heads, block_size, num_blocks;
    float qk_scale_log2;  // scale * log2(e)
    int32_t *status;
};

// Effective context of sequence s after the range checks (identical in both passes).
__device__ __forceinline__ int effective_context(const DecodeParams &p, int s, bool report_errors) {
    int ctx = p.context_lens[s];
    const int cap = min(p.max_blocks_per_seq * p.block_size, p.num_partitions * kPartition);
    if (ctx < 0 || ctx > cap) {
        if (report_errors) report(p.status, PA_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : cap;
    }
    return ctx;
}

template <class T, int D, int G, int NT>
__global__ void __launch_bounds__(kDecodeThreads)
decode_partition_kernel(const DecodeParams p) {
    using Sh = DecodeShape<T, D, G, NT>;
    constexpr int EPV = Sh::EPV, LPT = Sh::LPT, TPW = Sh::TPW, NTG = Sh::NTG, NV = Sh::NV;

    __shared__ float sc[kDecodeWarps][NT * G];        // per-warp batch scores / weights
    __shared__ float red_m[kDecodeWarps][G], red_l[kDecodeWarps][G];
    __shared__ __align__(16) float red_o[kDecodeWarps][G][D];

    const int part = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int grp = lane / LPT, r = lane % LPT;
    const int Hkv = p.num_kv_heads, Hq = p.num_heads;

    const int ctx = effective_context(p, s, part == 0 && threadIdx.x == 0);
    const int nparts = (ctx + kPartition - 1) / kPartition;
    if (ctx == 0) {  // empty context: zero output row(s), written by one CTA
        if (part == 0)
            for (int i = threadIdx.x; i < G * D / 2; i += kDecodeThreads) {
                const int h = i / (D / 2), d = (i % (D / 2)) * 2;
                store_pair_any(p.out, p.out_dtype, ((int64_t)s * Hq + g * G + h) * D + d, 0.f, 0.f);
            }
        return;
    }
    if (part >= nparts) return;

    // q slices for the G heads of this kv head, pre-scaled into the log2 domain.
    float q[G][EPV];
    {
        const typename T::storage *qp = static_cast<const typename T::storage *>(p.query) +
                                        ((int64_t)s * Hq + g * G) * D + r * EPV;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            uint4 raw = *reinterpret_cast<const uint4 *>(qp + h * D);
            widen(T{}, raw, q[h]);
#pragma unroll
            for (int e = 0; e < EPV; ++e) q[h][e] *= p.qk_scale_log2;
        }
    }

    float acc[G][EPV], m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[h][e] = 0.f;
    }

    const int bs = p.block_size;
    const int64_t row_stride = (int64_t)Hkv * D;  // elements between consecutive slots
    const typename T::storage *kc = static_cast<const typename T::storage *>(p.key_cache);
    const typename T::storage *vc = static_cast<const typename T::storage *>(p.value_cache);
    const int32_t *bt = p.block_tables + (int64_t)s * p.max_blocks_per_seq;

    const int w_begin = part * kPartition + warp * kWarpSpan;
    const int w_end = min(ctx, w_begin + kWarpSpan);
    float *wsc = sc[warp];

    for (int j0 = w_begin; j0 < w_end; j0 += NT) {
        // ---- issue every K and V load of the batch
        uint4 kv_k[NTG], kv_v[NTG];
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
            const int j = j0 + i * TPW + grp;
            kv_k[i] = make_uint4(0, 0, 0, 0);
            kv_v[i] = make_uint4(0, 0, 0, 0);
            if (j < w_end) {
                const int blk = bt[j / bs];
                if (blk >= 0 && blk < p.num_blocks) {
                    const int64_t off = ((int64_t)blk * bs + j % bs) * row_stride + g * D + r * EPV;
                    kv_k[i] = ldg_stream(kc + off);
                    kv_v[i] = ldg_stream(vc + off);
                } else if (r == 0) {
                    report(p.status, PA_DEVERR_BLOCK_ID);
                }
            }
        }
        // ---- partial q.k over this lane's slice, then reduce-scatter over the row
        float part_dot[NV];
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
            float kf[EPV];
            widen(T{}, kv_k[i], kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < EPV; ++e) a = fmaf(q[h][e], kf[e], a);
                part_dot[i * G + h] = a;
            }
        }
        reduce_scatter<NV, NV, LPT / 2>(part_dot, lane);
        {
            constexpr int R = NV >= LPT ? NV / LPT : 1;
            const int idx0 = r * NV / LPT;
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const int idx = idx0 + u;
                const int t = (idx / G) * TPW + grp;
                wsc[t * G + idx % G] = (j0 + t < w_end) ? part_dot[u] : -INFINITY;
            }
        }
        __syncwarp();
        // ---- online softmax over the batch (log2 domain); lane owns head lane % G
        float mx = -INFINITY;
        for (int idx = lane; idx < NT * G; idx += 32) mx = fmaxf(mx, wsc[idx]);
#pragma unroll
        for (int o = G; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
        float alpha[G], my_m = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mn = fmaxf(m[h], __shfl_sync(kFullMask, mx, h));
            alpha[h] = exp2f(m[h] - mn);
            m[h] = mn;
            if (lane % G == h) my_m = mn;
        }
        float sum = 0.f;
        for (int idx = lane; idx < NT * G; idx += 32) {
            const float e = exp2f(wsc[idx] - my_m);
            wsc[idx] = e;
            sum += e;
        }
#pragma unroll
        for (int o = G; o < 32; o <<= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            l[h] = l[h] * alpha[h] + __shfl_sync(kFullMask, sum, h);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[h][e] *= alpha[h];
        }
        __syncwarp();
        // ---- acc += p * v over this lane group's tokens
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
            const int t = i * TPW + grp;
            float vf[EPV];
            widen(T{}, kv_v[i], vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pw = wsc[t * G + h];
#pragma unroll
                for (int e = 0; e < EPV; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
            }
        }
        __syncwarp();
    }

    // ---- merge the lane groups (same m and l, different tokens)
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[h][e] += __shfl_xor_sync(kFullMask, acc[h][e], o);

    // ---- merge the warps through shared memory
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < EPV; ++e) red_o[warp][h][r * EPV + e] = acc[h][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            red_m[warp][h] = m[h];
            red_l[warp][h] = l[h];
        }
    }
    __syncthreads();
    const bool single = nparts == 1;
    for (int i = threadIdx.x; i < G * D / 2; i += kDecodeThreads) {
        const int h = i / (D / 2), d = (i % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, red_m[w][h]);
        float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            const float f = exp2f(red_m[w][h] - M);  // 0 for a warp without tokens
            L = fmaf(red_l[w][h], f, L);
            o0 = fmaf(red_o[w][h][d], f, o0);
            o1 = fmaf(red_o[w][h][d + 1], f, o1);
        }
        const int hq = g * G + h;
        if (single) {
            const float inv = 1.f / L;
            store_pair_any(p.out, p.out_dtype, ((int64_t)s * Hq + hq) * D + d, o0 * inv, o1 * inv);
        } else {
            const int64_t pi = ((int64_t)s * Hq + hq) * p.num_partitions + part;
            *reinterpret_cast<float2 *>(p.part_o + pi * D + d) = make_float2(o0, o1);
            if (d == 0) {
                p.part_m[pi] = M;
                p.part_l[pi] = L;
            }
        }
    }
}

// Pass 2: out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p, for sequences split
// into more than one partition.  grid = (sequence, q head).
template <int D>
__global__ void __launch_bounds__(64) decode_reduce_kernel(const DecodeParams p) {
    const int s = blockIdx.x, hq = blockIdx.y;
    const int ctx = effective_context(p, s, false);
    const int nparts = (ctx + kPartition - 1) / kPartition;
    if (nparts <= 1) return;
    const int64_t base = ((int64_t)s * p.num_heads + hq) * p.num_partitions;
    float M = -INFINITY;
    for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.part_m[base + i]);
    float L = 0.f;
    for (int i = 0; i < nparts; ++i) L = fmaf(p.part_l[base + i], exp2f(p.part_m[base + i] - M), L);
    const float inv = 1.f / L;
    for (int d = threadIdx.x * 2; d < D; d += 128) {
        float o0 = 0.f, o1 = 0.f;
        for (int i = 0; i < nparts; ++i) {
            const float f = exp2f(p.part_m[base + i] - M);
            const float2 v = *reinterpret_cast<const float2 *>(p.part_o + (base + i) * D + d);
            o0 = fmaf(v.x, f, o0);
            o1 = fmaf(v.y, f, o1);
        }
        store_pair_any(p.out, p.out_dtype, ((int64_t)s * p.num_heads + hq) * D + d, o0 * inv,
                       o1 * inv);
    }
}

constexpr int kBatchTokens = 16;

template <class T, int D, int G>
int launch_typed(const DecodeParams &prm, int num_seqs, cudaStream_t stream) {
    dim3 grid(prm.num_partitions, prm.num_kv_heads, num_seqs);
    decode_partition_kernel<T, D, G, kBatchTokens><<<grid, kDecodeThreads, 0, stream>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (prm.num_partitions > 1) {
        decode_reduce_kernel<D><<<dim3(num_seqs, prm.num_heads), 64, 0, stream>>>(prm);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

template <class T, int D>
int dispatch_g(const DecodeParams &prm, int G, int num_seqs, cudaStream_t st) {
    switch (G) {
        case 1: return launch_typed<T, D, 1>(prm, num_seqs, st);
        case 2: return launch_typed<T, D, 2>(prm, num_seqs, st);
        case 4: return launch_typed<T, D, 4>(prm, num_seqs, st);
        case 8: return launch_typed<T, D, 8>(prm, num_seqs, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

template <class T>
int dispatch_d(const DecodeParams &prm, int D, int G, int num_seqs, cudaStream_t st) {
    switch (D) {
        case 64: return dispatch_g<T, 64>(prm, G, num_seqs, st);
        case 128: return dispatch_g<T, 128>(prm, G, num_seqs, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len) {
    const int np = (max_context_len + kPartition - 1) / kPartition;
    if (np <= 1) return 0;
    const size_t rows = (size_t)num_seqs * num_heads * np;
    return align_up(rows * head_dim * sizeof(float)) + 2 * align_up(rows * sizeof(float));
}

int launch_decode(const DecodeArgs &a) {
    if (a.num_seqs == 0) return PA_OK;
    DecodeParams prm{};
    prm.out = a.out;
    prm.out_dtype = a.out_dtype;
    prm.query = a.query;
    prm.key_cache = a.key_cache;
    prm.value_cache = a.value_cache;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.max_blocks_per_seq = a.max_blocks_per_seq;
    prm.num_partitions = a.max_context_len > 0 ? (a.max_context_len + kPartition - 1) / kPartition : 1;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.block_size = a.block_size;
    prm.num_blocks = a.num_blocks;
    prm.qk_scale_log2 = a.scale * kLog2e;
    prm.status = a.status;
    if (prm.num_partitions > 1) {
        const size_t rows = (size_t)a.num_seqs * a.num_heads * prm.num_partitions;
        char *ws = static_cast<char *>(a.workspace);
        prm.part_o = reinterpret_cast<float *>(ws);
        ws += align_up(rows * a.head_dim * sizeof(float));
        prm.part_m = reinterpret_cast<float *>(ws);
        ws += align_up(rows * sizeof(float));
        prm.part_l = reinterpret_cast<float *>(ws);
    }
    const int G = a.num_heads / a.num_kv_heads;
    switch (a.kv_dtype) {
        case PA_F32: return dispatch_d<F32>(prm, a.head_dim, G, a.num_seqs, a.stream);
        case PA_F16: return dispatch_d<F16>(prm, a.head_dim, G, a.num_seqs, a.stream);
        case PA_BF16: return dispatch_d<BF16>(prm, a.head_dim, G, a.num_seqs, a.stream);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
