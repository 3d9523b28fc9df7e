// decode_kernels.cuh -- paged decode attention on GB300: TMA-fed, balanced split-K,
// log-sum-exp reduce.  The kernels and their typed launchers; decode.cu holds the
// host side and the plain instantiations, decode_rope.cu the instantiations that
// rotate the query in the kernel.
//
// One query token per sequence attends every cached key of its sequence,
// gathered through the block table (TensorSharp "Mistral 3" page, section 11:
// per-sequence paged attention over the paged K/V buffer; sections 3 / 4.1:
// causal GQA attention with Q scaled by 1/sqrt(headDim)).
//
// Work decomposition.  A "unit" is TU consecutive tokens of one sequence for a
// group of HG kv heads (HG = min(Hkv, 8)); units never straddle sequences.  A
// "segment" is all units of one (head group, sequence).  All units of all
// segments, in order, are split into equal contiguous ranges over one CTA per
// SM (a balanced split-K: every CTA streams the same number of K/V bytes,
// whatever the mix of context lengths).  A CTA whose range covers a whole
// segment writes the output directly; otherwise it writes a partial
// (running max m, running sum l, unnormalised output acc) for its piece of the
// segment and the reduce kernel merges the pieces.
//
// Kernels (in stream order, each a programmatic dependent launch so that its
// launch and prologue overlap the previous kernel): split (the streaming
// kernel) and reduce (merges the pieces of every segment split over CTAs).
// The split needs the scan of the per-segment unit counts: with fewer than
// kSegSmem segments every CTA computes it in its prologue (CTA 0 publishes it
// for the reduce); beyond that a one-CTA plan kernel computes it first.  The
// scan's owner also clamps the context lengths (reporting bad ones) and zeroes
// the output of sequences with nothing to attend.
// The reduce does not wait for the end of the split grid before merging: each launch
// carries a 64-bit tag, the scan's owner and every CTA with partials store it (release)
// once their data is visible, and a reduce CTA -- small enough to be resident beside a
// split CTA -- waits (acquire, bounded in time) for the tags of its segment's pieces.
// It waits for the split grid only before it exits, so that the reduce grid still ends
// after every output the split kernel writes directly.  A launch made while its stream is
// captured into a CUDA graph merges after the end of the split grid instead: every replay
// of the graph carries the same tag, which the previous replay left in the workspace.
//
// Split kernel, per CTA: one producer warp issues 3-D TMA loads of whole
// [tokens][HG heads][D] boxes of K and V (one box per block piece, taken
// through the block table) into an NSTAGE-deep shared-memory ring guarded by
// full/empty mbarriers; eight consumer warps each own one kv head (and a
// token slice of the stage when HG * QS < 8) and G of the query heads that read it:
// all of them (QS = 1) while a kv head has at most four, else half (QS = 2 query slices,
// two warps reading the same K/V rows), so that a lane's state never exceeds four heads.
// Lanes own 16-byte slices of the head dimension; the q.k partial dot
// products of a batch of tokens are reduce-scattered across a token row's
// lanes so that every lane finishes with whole scores; the online softmax
// runs in the log2 domain; FMAs are packed fp32x2.
#pragma once

#include <type_traits>

#include "tma.cuh"

namespace pa {

struct DecodeParams {
    void *out;
    pa_dtype out_dtype;
    const void *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int32_t *seg_start;  // [K + 1] exclusive scan of units per segment (workspace)
    int32_t *cta_k0;     // [grid] first segment of each CTA's range (workspace)
    float *part_o;       // [(C + K) * HGq * D]
    float *part_m;       // [(C + K) * HGq]
    float *part_l;       // [(C + K) * HGq]
    // launch tags (workspace): [0] the segment table is written, [1 + c + k] the partial of CTA c
    // for segment k is written; each holds launch_tag once its data is visible
    unsigned long long *tags;
    unsigned long long launch_tag;
    int tagged;           // the reduce waits for tags (else for the end of the split grid: a
                          // launch captured into a CUDA graph replays with one fixed tag)
    int scan_in_split;    // the split kernel's CTA 0 writes the segment table (else the plan kernel)
    int max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, block_size, num_blocks;
    int max_context_len, head_dim;
    int heads_per_group;  // HG
    int num_groups;       // Hkv / HG
    int unit_tokens;      // TU
    int box_rows;         // tokens per TMA box (min(bs, TU))
    int grid;             // CTAs launched for the split kernel
    float qk_scale_log2;  // scale * log2(e)
    int32_t *status;
    // query RoPE (GPT-J pairs) and position-dependent scale, at position context_len - 1
    const float *rope_freqs;  // null: no rotation, no scale
    int rope_dim;
    float q_scale_beta;
    int q_scale_orig_ctx;
    // cache write fused in front of the attention (pa_decode_write): the new token of every
    // sequence, [S][Hkv][D] in the cache's type, stored at slot_mapping[s]
    const void *new_key, *new_value;
    const int64_t *slot_mapping;
    void *key_cache_w, *value_cache_w;
    int64_t num_slots;
};

// The launchers of the query-rotating instantiations (decode_rope.cu); the plain ones
// are instantiated in decode.cu.  Both take the parameters launch_decode prepared.
int dispatch_decode_rope(const DecodeParams &prm, pa_dtype kv_dtype, int D, int G, const CUtensorMap &km,
                         const CUtensorMap &vm, cudaStream_t st);
// ... and of the instantiations that write each sequence's new token first (decode_write.cu).
int dispatch_decode_write(const DecodeParams &prm, pa_dtype kv_dtype, int D, int G, const CUtensorMap &km,
                          const CUtensorMap &vm, cudaStream_t st);

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kPlanThreads = 1024;
constexpr int kSegSmem = 2048;  // segments whose scan the split kernel keeps in shared memory
constexpr float kRescaleLog2 = 8.f;  // lazy softmax: rescale when a score exceeds the reference by 2^8

template <class T, int D, int G, int QS = 1>
struct DecodeShape {
    static constexpr int EPV = T::kPerVec;            // elements per 16-byte vector
    static constexpr int LPT = D / EPV;               // lanes covering one token row
    static constexpr int TPW = 32 / LPT;              // token rows per warp step
    static constexpr int ROW_BYTES = D * T::kBytes;   // one (token, kv head) row
    // tokens per consumer warp per stage (8 when the per-lane state would spill)
    static constexpr int NT = (ROW_BYTES <= 256 && G <= 4) ? 16 : 8;
    static constexpr int NTG = NT / TPW;              // tokens per lane group per stage
    static constexpr int NV = NTG * G;                // partial dot products per lane
    static constexpr int R = NV >= LPT ? NV / LPT : 1;  // whole scores per lane
    static constexpr int TOKEN_BITS = NTG >= 16 ? 4 : NTG >= 8 ? 3 : NTG >= 4 ? 2 : NTG >= 2 ? 1 : 0;
    static_assert((1 << TOKEN_BITS) == NTG && NTG <= LPT, "token slots: a power of two, at most LPT");
    static constexpr int STAGE_ROWS = NT * kConsumerWarps / QS;  // (token, kv head) rows of a stage
    static constexpr int KV_BYTES = STAGE_ROWS * ROW_BYTES;  // K (and V) bytes per stage
    static constexpr int RED_BYTES = kConsumerWarps * G * (D + 2) * 4;
    static constexpr int SC_BYTES = kConsumerWarps * NT * G * 4;
    static constexpr int FIXED = RED_BYTES + SC_BYTES + kSegSmem * 4 + 1024;
    static constexpr int NSTAGE_FIT = (kSmemBudget - 1024 - FIXED) / (2 * KV_BYTES);
    static constexpr int NSTAGE = NSTAGE_FIT > 6 ? 6 : NSTAGE_FIT;
    static constexpr int SMEM = 1024 + NSTAGE * 2 * KV_BYTES + FIXED;
    static_assert(LPT >= 1 && LPT <= 32 && 32 % LPT == 0, "head row must span 1..32 lanes");
    static_assert(NT % TPW == 0 && EPV % 2 == 0, "stage must be whole warp steps");
    static_assert(NSTAGE >= 2, "at least double buffering");
    static_assert(SMEM <= kSmemBudget, "shared memory budget");
};


// ------------------------------------------------------------------------------ helpers

// Reduce-scatter of v[0..N) across the lanes that differ in bits OFF, OFF/2, .., 1
// of a token row group.  The first TOKEN_STEPS steps split token-slot bits: the
// caller loaded token slots in an order XOR-permuted by the lane's high bits, so
// every lane keeps the low half and sends the high half (no selects).  Remaining
// steps split head bits (keep the half selected by the lane bit) and, once a
// single value is left, plain all-reduce.  Lane r of the group ends with the
// full sums of logical entries r*NV/LPT .. (+ max(NV/LPT, 1) - 1).
template <int NV, int N, int OFF, int TOKEN_STEPS>
__device__ __forceinline__ void reduce_scatter_perm(float (&v)[NV], int lane) {
    if constexpr (OFF >= 1) {
        if constexpr (TOKEN_STEPS > 0) {
#pragma unroll
            for (int i = 0; i < N / 2; ++i) v[i] += __shfl_xor_sync(kFullMask, v[i + N / 2], OFF);
            reduce_scatter_perm<NV, N / 2, OFF / 2, TOKEN_STEPS - 1>(v, lane);
        } else if constexpr (N > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float keep = upper ? v[i + N / 2] : v[i];
                const float send = upper ? v[i] : v[i + N / 2];
                v[i] = keep + __shfl_xor_sync(kFullMask, send, OFF);
            }
            reduce_scatter_perm<NV, N / 2, OFF / 2, 0>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFullMask, v[0], OFF);
            reduce_scatter_perm<NV, 1, OFF / 2, 0>(v, lane);
        }
    }
}

// The G softmax weights of one token from the warp's score buffer (16-byte aligned rows).
template <int G>
__device__ __forceinline__ void load_weights(const float *w, float (&out)[G]) {
    if constexpr (G % 4 == 0) {
#pragma unroll
        for (int i = 0; i < G; i += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(w + i);
            out[i] = v.x;
            out[i + 1] = v.y;
            out[i + 2] = v.z;
            out[i + 3] = v.w;
        }
    } else if constexpr (G == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(w);
        out[0] = v.x;
        out[1] = v.y;
    } else {
        out[0] = w[0];
    }
}

__device__ __forceinline__ void store_pair_any(void *out, pa_dtype dt, int64_t idx, float a,
                                               float b) {
    if (dt == PA_F32)
        store_out(static_cast<float *>(out) + idx, a, b);
    else if (dt == PA_F16)
        store_out(static_cast<__half *>(out) + idx, a, b);
    else
        store_out(static_cast<__nv_bfloat16 *>(out) + idx, a, b);
}

// Packed 16-bit pair -> float2.
__device__ __forceinline__ float2 widen2(BF16, uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ float2 widen2(F16, uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2 *>(&u));
}

// 16-byte vector -> EPV/2 float2.
template <class T>
__device__ __forceinline__ void widen_vec(const uint4 &v, float2 *f);
template <>
__device__ __forceinline__ void widen_vec<F32>(const uint4 &v, float2 *f) {
    f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}
template <>
__device__ __forceinline__ void widen_vec<BF16>(const uint4 &v, float2 *f) {
    f[0] = widen2(BF16{}, v.x);
    f[1] = widen2(BF16{}, v.y);
    f[2] = widen2(BF16{}, v.z);
    f[3] = widen2(BF16{}, v.w);
}
template <>
__device__ __forceinline__ void widen_vec<F16>(const uint4 &v, float2 *f) {
    f[0] = widen2(F16{}, v.x);
    f[1] = widen2(F16{}, v.y);
    f[2] = widen2(F16{}, v.z);
    f[3] = widen2(F16{}, v.w);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// CTA that owns unit u when N units are split over C CTAs (CTA c owns
// [c*N/C, (c+1)*N/C)).
__device__ __forceinline__ int owner_cta(int u, int N, int C) {
    return (int)((((int64_t)u + 1) * C + N - 1) / N) - 1;
}

// ------------------------------------------------------------------------------ launch tags

__device__ __forceinline__ void store_release(unsigned long long *a, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long load_acquire(const unsigned long long *a) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
// Loads that see other CTAs' writes made visible by a release the caller has acquired.
__device__ __forceinline__ float load_relaxed(const float *a) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ float2 load_relaxed2(const float *a) {
    float2 v;
    asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ int load_relaxed_i(const int32_t *a) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Wait until *a holds this launch's tag; false (and a status bit) after kWaitLimitNs.
__device__ bool wait_tag(const unsigned long long *a, unsigned long long tag, int32_t *status) {
    if (load_acquire(a) == tag) return true;
    const unsigned long long t0 = global_ns();
    unsigned ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (ns < 256) ns *= 2;
        if (load_acquire(a) == tag) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            report(status, PA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------------------ plan kernel

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const DecodeParams p) {
    pdl_wait_previous();      // inputs written by earlier kernels are visible
    pdl_launch_dependents();  // the split kernel may launch now; it waits for our writes
    __shared__ int buf[kPlanThreads];
    __shared__ int carry;
    const int tid = threadIdx.x;
    const int S = p.num_seqs;
    const int K = p.num_groups * S;
    const int cap = min(p.max_blocks_per_seq * p.block_size, p.max_context_len);
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < K; base += kPlanThreads) {
        const int k = base + tid;
        int n = 0;
        if (k < K) {
            const int s = k % S;
            int ctx = p.context_lens[s];
            if (ctx < 0 || ctx > cap) {
                if (k < S) report(p.status, PA_DEVERR_CONTEXT);
                ctx = ctx < 0 ? 0 : cap;
            }
            n = (ctx + p.unit_tokens - 1) / p.unit_tokens;
        }
        // block-wide inclusive scan of n: warp shuffles, then the warp totals
        int v = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFullMask, v, o);
            if ((tid & 31) >= o) v += t;
        }
        if ((tid & 31) == 31) buf[tid >> 5] = v;
        __syncthreads();
        if (tid < 32) {
            int w = buf[tid];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFullMask, w, o);
                if (tid >= o) w += t;
            }
            buf[tid] = w;
        }
        __syncthreads();
        const int incl = v + ((tid >> 5) ? buf[(tid >> 5) - 1] : 0);
        if (k < K) p.seg_start[k] = carry + incl - n;
        __syncthreads();
        if (tid == kPlanThreads - 1) carry += incl;
        __syncthreads();
    }
    const int N = carry;
    if (tid == 0) p.seg_start[K] = N;
    __syncthreads();  // seg_start is visible to the whole block
    if (tid == 0) {   // and, once this fence is passed, to the reduce kernel
        __threadfence();
        store_release(p.tags, p.launch_tag);
    }
    // CTA c starts at unit c*N/C, inside the segment k with seg_start[k] <= c*N/C <
    // seg_start[k+1]: the CTAs starting in segment k are ceil(beg*C/N) .. ceil(end*C/N)-1.
    const int C = min(p.grid, N);
    const int HGq = p.heads_per_group * (p.num_heads / p.num_kv_heads);
    const int ob = p.out_dtype == PA_F32 ? 4 : 2;
    const int words = HGq * p.head_dim * ob / 4;
    for (int k = tid; k < K; k += kPlanThreads) {
        const int beg = p.seg_start[k], end = p.seg_start[k + 1];
        if (C > 0) {
            const int cf = (int)(((int64_t)beg * C + N - 1) / N);
            const int cl = (int)(((int64_t)end * C + N - 1) / N);
            for (int c = cf; c < cl; ++c) p.cta_k0[c] = k;
        }
        if (beg == end) {  // nothing to attend: a zero row that nobody else writes
            const int s = k % S, hg = k / S;
            uint32_t *row = reinterpret_cast<uint32_t *>(
                static_cast<char *>(p.out) + ((int64_t)s * p.num_heads + hg * HGq) * p.head_dim * ob);
            for (int i = 0; i < words; ++i) row[i] = 0u;
        }
    }
}

// ------------------------------------------------------------------------------ in-CTA plan

// sseg[0..K) = exclusive prefix of the units of every segment, sseg[K] = total,
// computed by all threads of the CTA (kDecodeThreads) in chunks.
__device__ void scan_units(const DecodeParams &p, int *sseg, int *wtot, int K, int cap,
                           bool report_errors) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, S = p.num_seqs;
    constexpr int NWARP = kDecodeThreads / 32;
    int carry = 0;
    for (int base = 0; base < K; base += kDecodeThreads) {
        const int k = base + tid;
        int n = 0;
        if (k < K) {
            int ctx = p.context_lens[k % S];
            if (ctx < 0 || ctx > cap) {
                if (report_errors && k < S) report(p.status, PA_DEVERR_CONTEXT);
                ctx = ctx < 0 ? 0 : cap;
            }
            n = (ctx + p.unit_tokens - 1) / p.unit_tokens;
        }
        int v = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFullMask, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) wtot[w] = v;
        __syncthreads();
        int before = carry, total = 0;
#pragma unroll
        for (int i = 0; i < NWARP; ++i) {
            before += i < w ? wtot[i] : 0;
            total += wtot[i];
        }
        if (k < K) sseg[k] = before + v - n;
        __syncthreads();
        carry += total;
    }
    if (tid == 0) sseg[K] = carry;
    __syncthreads();
}

// CTA 0 of the split kernel: the scan for the reduce kernel, and zero rows for
// sequences with nothing to attend (no CTA streams them).
__device__ void publish_scan(const DecodeParams &p, const int *sseg, int K, int HGq) {
    const int S = p.num_seqs;
    const int ob = p.out_dtype == PA_F32 ? 4 : 2;
    const int words = HGq * p.head_dim * ob / 4;
    for (int k = threadIdx.x; k <= K; k += kDecodeThreads) p.seg_start[k] = sseg[k];
    __syncthreads();
    if (threadIdx.x == 0) {  // the reduce kernel may read the table
        __threadfence();
        store_release(p.tags, p.launch_tag);
    }
    for (int k = threadIdx.x; k < K; k += kDecodeThreads) {
        if (sseg[k] != sseg[k + 1]) continue;
        const int s = k % S, hg = k / S;
        uint32_t *row = reinterpret_cast<uint32_t *>(
            static_cast<char *>(p.out) + ((int64_t)s * p.num_heads + hg * HGq) * p.head_dim * ob);
        for (int i = 0; i < words; ++i) row[i] = 0u;
    }
}

// ------------------------------------------------------------------------------ split kernel

template <class T, int D, int G, int QS, bool ROPE, bool WRITE>
__global__ void __launch_bounds__(kDecodeThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const DecodeParams p) {
    using Sh = DecodeShape<T, D, G, QS>;
    constexpr int GQ = G * QS;  // query heads per kv head (this warp holds G of them)
    constexpr int EPV = Sh::EPV, LPT = Sh::LPT, TPW = Sh::TPW, NT = Sh::NT, NTG = Sh::NTG;
    constexpr int NV = Sh::NV, NSTAGE = Sh::NSTAGE, KVB = Sh::KV_BYTES, ROWB = Sh::ROW_BYTES;
    constexpr int NW = kConsumerWarps;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stage_base = smem_u32(smem);                    // NSTAGE x [K | V]
    float *red_o = reinterpret_cast<float *>(smem + NSTAGE * 2 * KVB);  // [NW][G][D]
    float *red_m = red_o + NW * G * D;                             // [NW][G]
    float *red_l = red_m + NW * G;                                 // [NW][G]
    float *scores = red_l + NW * G;                                // [NW][NT * G]
    uint64_t *bars = reinterpret_cast<uint64_t *>(scores + NW * NT * G);  // full[NSTAGE], empty[NSTAGE]
    int *abort_flag = reinterpret_cast<int *>(bars + 2 * NSTAGE);

    int *wtot = abort_flag + 4;                                    // [kDecodeThreads / 32]
    int *sseg = wtot + 12;                                         // [kSegSmem]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NSTAGE;
    // Prologue that needs nothing from earlier kernels, overlapping them.
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, NW);
        }
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_wait_previous();      // context lengths, block tables, caches (and the plan) are ready
    pdl_launch_dependents();  // the reduce kernel may launch; it waits for our completion

    const int S = p.num_seqs;
    const int K = p.num_groups * S;
    const int c = blockIdx.x;
    const int cap = min(p.max_blocks_per_seq * p.block_size, p.max_context_len);
    const int HG = p.heads_per_group, HGq = HG * GQ, TU = p.unit_tokens;
    const bool fused = K < kSegSmem;
    const int *segs = fused ? sseg : p.seg_start;
    if (fused) {
        scan_units(p, sseg, wtot, K, cap, c == 0);
        if (c == 0) publish_scan(p, sseg, K, HGq);
    }
    const int N = segs[K];
    const int C = min(p.grid, N);
    if (c >= C) return;  // whole CTA: nothing to stream
    const int u0 = (int)((int64_t)c * N / C), u1 = (int)((int64_t)(c + 1) * N / C);
    int k0;
    if (fused) {  // largest k with sseg[k] <= u0
        int lo = 0, hi = K;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sseg[mid] <= u0) lo = mid; else hi = mid;
        }
        k0 = lo;
    } else {
        k0 = p.cta_k0[c];
    }
    __syncthreads();  // barrier initialisation visible to every thread
    volatile int *abort_v = abort_flag;
    auto context_of = [&](int s) {
        const int ctx = p.context_lens[s];
        return ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    };

    // ============================================================ producer
    if (warp == NW) {
        if (lane != 0) return;
        const uint64_t policy = policy_evict_first();
        const int bs = p.block_size, rows = p.box_rows, nbox = TU / rows;
        const uint32_t box_bytes = (uint32_t)rows * HG * ROWB;
        int k = k0, seg_beg = segs[k], seg_end = segs[k + 1];
        int s = k % S, hg = k / S, ctx = context_of(s);
        for (int u = u0, i = 0; u < u1; ++u, ++i) {
            while (u >= seg_end) {
                ++k;
                seg_beg = seg_end;
                seg_end = segs[k + 1];
                s = k % S;
                hg = k / S;
                ctx = context_of(s);
            }
            const int stage = i % NSTAGE;
            const uint32_t parity = ((i / NSTAGE) & 1) ^ 1;
            if (*abort_v || !mbar_wait(empty0 + 8 * stage, parity, p.status)) {
                *abort_v = 1;
                break;
            }
            const int t0 = (u - seg_beg) * TU;
            const int32_t *bt = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
            const uint32_t full = full0 + 8 * stage;
            const uint32_t kdst = stage_base + stage * 2 * KVB;
#pragma unroll 1
            for (int b = 0; b < nbox; ++b) {
                const int tb = t0 + b * rows;
                if (tb >= ctx) break;
                const int id = bt[tb / bs];
                if (id < 0 || id >= p.num_blocks) {  // never dereferenced; the stage keeps stale data
                    report(p.status, PA_DEVERR_BLOCK_ID);
                    continue;
                }
                const int row = id * bs + tb % bs;
                mbar_expect_tx(full, 2 * box_bytes);
                tma_load_3d(kdst + b * box_bytes, &kmap, 0, hg * HG, row, full, policy);
                tma_load_3d(kdst + KVB + b * box_bytes, &vmap, 0, hg * HG, row, full, policy);
            }
            mbar_arrive(full);
        }
        return;
    }

    // ============================================================ consumers
    const int h = warp % HG;          // kv head within the group
    const int qs = (warp / HG) % QS;  // query slice: heads h * GQ + qs * G .. + G - 1 of the group
    const int sb = warp / (HG * QS);  // token slice of the stage
    const int grp = lane / LPT, r = lane % LPT;
    float *wsc = scores + warp * NT * G;
    // After the reduce-scatter, lane r holds whole scores of one token of its slice,
    // tl_own, for heads hb .. hb + R - 1 (several lanes hold the same values when
    // NV < LPT; only the owner counts them).
    constexpr int R = Sh::R;
    constexpr int DUP = NV >= LPT ? 1 : LPT / NV;
    const int perm = r / (LPT / NTG);                 // XOR permutation of token slots
    const int tl_own = perm * TPW + grp;
    const int hb = (r * NV / LPT) % G;
    const bool owner = (r % DUP) == 0;

    float2 q2[G][EPV / 2];
    float2 acc[G][EPV / 2];
    float m[G];         // reference max per head (log2 domain), same in every lane
    float mref[R];      // m[] of this lane's own heads
    float l_lane[R];    // this lane's share of the softmax denominators
    auto reset = [&]() {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            m[hh] = -INFINITY;
#pragma unroll
            for (int e = 0; e < EPV / 2; ++e) acc[hh][e] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            mref[u] = -INFINITY;
            l_lane[u] = 0.f;
        }
    };
    // This lane's 16-byte slices of the warp's G query rows of (sequence s, head group hg).
    auto q_global = [&](int s, int hg, uint4 (&raw)[G]) {
        const typename T::storage *qp = static_cast<const typename T::storage *>(p.query) +
                                        ((int64_t)s * p.num_heads + hg * HGq + h * GQ + qs * G) * D + r * EPV;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) raw[hh] = *reinterpret_cast<const uint4 *>(qp + hh * D);
    };
    // Query prefetch for the next segment of the range: with eight kv heads per group (the
    // flush then needs no shared memory) each warp copies its rows into its own slice of
    // red_o with cp.async while it streams the segment's last unit, so that the switch
    // waits for no global load.
    const bool q_prefetch = G <= 4 && HG * QS == NW;
    const uint32_t q_slot = smem_u32(red_o) + (uint32_t)(warp * G * D * (int)sizeof(typename T::storage));
    auto q_prefetch_issue = [&](int s, int hg) {
        if (grp == 0) {
            const typename T::storage *qp = static_cast<const typename T::storage *>(p.query) +
                                            ((int64_t)s * p.num_heads + hg * HGq + h * GQ + qs * G) * D + r * EPV;
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 q_slot + (uint32_t)((hh * D + r * EPV) * (int)sizeof(typename T::storage))),
                             "l"(qp + hh * D)
                             : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto q_prefetched = [&](uint4 (&raw)[G]) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
            raw[hh] = lds128(q_slot + (uint32_t)((hh * D + r * EPV) * (int)sizeof(typename T::storage)));
        __syncwarp();  // every lane has read the slice before the next prefetch overwrites it
    };
    auto load_q = [&](const uint4 (&qraw)[G], int ctx) {
        if constexpr (!ROPE) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const uint4 raw = qraw[hh];
                widen_vec<T>(raw, q2[hh]);
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e) {
                    q2[hh][e].x *= p.qk_scale_log2;
                    q2[hh][e].y *= p.qk_scale_log2;
                }
            }
        } else {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const uint4 raw = qraw[hh];
                widen_vec<T>(raw, q2[hh]);
            }
            // RoPE at the newest token's position (GPT-J pairs: this lane's float2 entries
            // are the pairs (2i, 2i+1), i = r * EPV / 2 + e), then the position scale
            const int pos = max(ctx - 1, 0);
#pragma unroll
            for (int e = 0; e < EPV / 2; ++e) {
                const int pair = r * (EPV / 2) + e;
                if (2 * pair < p.rope_dim) {
                    const float2 cs = rope_cos_sin(pos, p.rope_freqs[pair]);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float x = q2[hh][e].x, y = q2[hh][e].y;
                        q2[hh][e] = make_float2(x * cs.x - y * cs.y, x * cs.y + y * cs.x);
                    }
                }
            }
            float qs = p.qk_scale_log2;
            if (p.q_scale_orig_ctx > 0)
                qs *= fmaf(p.q_scale_beta, log1pf((float)(pos / p.q_scale_orig_ctx)), 1.f);
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e) {
                    q2[hh][e].x *= qs;
                    q2[hh][e].y *= qs;
                }
        }
    };

    // One stage: NT tokens of kv head h starting at logical token `tok0`.
    auto consume = [&](uint32_t kbase, uint32_t vbase, int tok0, int ctx, auto masked_tag) {
        constexpr bool MASKED = decltype(masked_tag)::value;
        const uint32_t row0 = (uint32_t)((sb * NT * HG + h) * ROWB + r * 16);
        const uint32_t tok_stride = (uint32_t)(HG * ROWB);  // bytes between token rows
        // ---- partial q.k; slot i of this lane holds token slot (i ^ perm)
        float part[NV];
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
            const int t = (i ^ perm) * TPW + grp;
            const uint4 kv = lds128(kbase + row0 + t * tok_stride);
            float2 kf[EPV / 2];
            widen_vec<T>(kv, kf);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float2 a = __fmul2_rn(q2[hh][0], kf[0]);
#pragma unroll
                for (int e = 1; e < EPV / 2; ++e) a = __ffma2_rn(q2[hh][e], kf[e], a);
                part[i * G + hh] = a.x + a.y;
            }
        }
        reduce_scatter_perm<NV, NV, LPT / 2, Sh::TOKEN_BITS>(part, lane);
        float sc[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            sc[u] = part[u];
            if constexpr (MASKED) sc[u] = (tok0 + tl_own < ctx) ? sc[u] : -INFINITY;
        }
        // ---- lazy reference update: only when a score exceeds its reference by 2^8
        bool grow = false;
#pragma unroll
        for (int u = 0; u < R; ++u) grow |= sc[u] > mref[u] + kRescaleLog2;
        if (__any_sync(kFullMask, grow)) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float mx = -INFINITY;
#pragma unroll
                for (int u = 0; u < R; ++u) mx = (hb + u == hh) ? fmaxf(mx, sc[u]) : mx;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
                const float mn = fmaxf(m[hh], mx);
                const float alpha = fast_exp2(m[hh] - mn);  // 0 while m is -inf
                m[hh] = mn;
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e) acc[hh][e] = __fmul2_rn(acc[hh][e], a2);
#pragma unroll
                for (int u = 0; u < R; ++u)
                    if (hb + u == hh) {
                        l_lane[u] *= alpha;
                        mref[u] = mn;
                    }
            }
        }
        // ---- weights of this lane's scores, shared through the warp's score buffer
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const float e = fast_exp2(sc[u] - mref[u]);
            if (owner) l_lane[u] += e;
            wsc[tl_own * G + hb + u] = e;
        }
        __syncwarp();
        // ---- acc += p * v over this lane group's tokens
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
            const int tl = i * TPW + grp;
            const uint4 vv = lds128(vbase + row0 + tl * tok_stride);
            float2 vf[EPV / 2];
            widen_vec<T>(vv, vf);
            if constexpr (MASKED) {
                if (tok0 + tl >= ctx) {
#pragma unroll
                    for (int e = 0; e < EPV / 2; ++e) vf[e] = make_float2(0.f, 0.f);
                }
            }
            float pw[G];
            load_weights<G>(wsc + tl * G, pw);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float2 p2 = make_float2(pw[hh], pw[hh]);
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e) acc[hh][e] = __ffma2_rn(p2, vf[e], acc[hh][e]);
            }
        }
        __syncwarp();
    };

    // The segments whose partial this CTA writes (its first and its last at most); their launch
    // tags are published once the CTA has streamed its whole range.
    int part0 = -1, part1 = -1;

    // Write this CTA's piece of segment k: merge lane groups and token slices,
    // then the output (whole segment here) or a partial for the reduce kernel.
    auto flush = [&](int k, bool whole) {
        if (!whole) (part0 < 0 ? part0 : part1) = k;
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1)
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e) {
                    acc[hh][e].x += __shfl_xor_sync(kFullMask, acc[hh][e].x, o);
                    acc[hh][e].y += __shfl_xor_sync(kFullMask, acc[hh][e].y, o);
                }
        float lsum[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float v = 0.f;
#pragma unroll
            for (int u = 0; u < R; ++u) v += (hb + u == hh) ? l_lane[u] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(kFullMask, v, o);
            lsum[hh] = v;
        }
        const int s = k % S, hg = k / S, nsub = NW / (HG * QS);
        if (G <= 4 && nsub == 1) {  // every warp holds whole rows of its heads: write from registers
            if (grp == 0) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const int hl = h * GQ + qs * G + hh;
                    if (whole) {
                        const float inv = 1.f / lsum[hh];
                        const int64_t o0 = ((int64_t)s * p.num_heads + hg * HGq + hl) * D + r * EPV;
#pragma unroll
                        for (int e = 0; e < EPV / 2; ++e)
                            store_pair_any(p.out, p.out_dtype, o0 + 2 * e, acc[hh][e].x * inv, acc[hh][e].y * inv);
                    } else {
                        const int64_t pi = (int64_t)(c + k) * HGq + hl;
#pragma unroll
                        for (int e = 0; e < EPV / 2; ++e)
                            *reinterpret_cast<float2 *>(p.part_o + pi * D + r * EPV + 2 * e) = acc[hh][e];
                        if (r == 0) {
                            p.part_m[pi] = m[hh];
                            p.part_l[pi] = lsum[hh];
                        }
                    }
                }
            }
            reset();
            return;
        }
        if (grp == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < EPV / 2; ++e)
                    *reinterpret_cast<float2 *>(red_o + (warp * G + hh) * D + r * EPV + 2 * e) = acc[hh][e];
        }
        if (lane == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                red_m[warp * G + hh] = m[hh];
                red_l[warp * G + hh] = lsum[hh];
            }
        }
        named_barrier(1, NW * 32);
        for (int idx = threadIdx.x; idx < HGq * (D / 2); idx += NW * 32) {
            const int hl = idx / (D / 2), d = (idx % (D / 2)) * 2;
            const int hk = hl / GQ, hq = hl % GQ / G, hh = hl % G;
            float M = -INFINITY;  // warp of token slice j: j * HG * QS + hq * HG + hk
            for (int j = 0; j < nsub; ++j) M = fmaxf(M, red_m[((j * QS + hq) * HG + hk) * G + hh]);
            float L = 0.f, o0 = 0.f, o1 = 0.f;
            for (int j = 0; j < nsub; ++j) {
                const int w = (j * QS + hq) * HG + hk;
                const float f = fast_exp2(red_m[w * G + hh] - M);  // 0 for a slice without tokens
                L = fmaf(red_l[w * G + hh], f, L);
                o0 = fmaf(red_o[(w * G + hh) * D + d], f, o0);
                o1 = fmaf(red_o[(w * G + hh) * D + d + 1], f, o1);
            }
            if (whole) {
                const float inv = 1.f / L;
                store_pair_any(p.out, p.out_dtype, ((int64_t)s * p.num_heads + hg * HGq + hl) * D + d,
                               o0 * inv, o1 * inv);
            } else {
                const int64_t pi = (int64_t)(c + k) * HGq + hl;
                *reinterpret_cast<float2 *>(p.part_o + pi * D + d) = make_float2(o0, o1);
                if (d == 0) {
                    p.part_m[pi] = M;
                    p.part_l[pi] = L;
                }
            }
        }
        named_barrier(1, NW * 32);
        reset();
    };

    // Fused cache write: the CTA that streams a segment's last unit stores the sequence's new
    // token (position context_len - 1) into its cache slot and patches the token's rows into
    // that unit's shared-memory stage, so that its own scores never depend on the store having
    // landed; only the warp whose token slice holds the token does it, one 16-byte slice per
    // lane.  A negative slot writes nothing (the stage keeps what the cache holds), like
    // pa_reshape_and_cache.
    [[maybe_unused]] uint4 new_k{}, new_v{};
    [[maybe_unused]] int patch_tn = -1;  // stage row of the new token in the segment's last unit
    auto new_token = [&](int s, int hg, int ctx, int seg_beg, int seg_end) {
        if constexpr (WRITE) {
            patch_tn = -1;
            if (seg_end > u1 || ctx <= 0 || p.context_lens[s] != ctx) return;  // not ours, or clamped
            const int tn = (ctx - 1) - (seg_end - 1 - seg_beg) * TU;
            if (tn / NT != sb) return;
            const int64_t slot = p.slot_mapping[s];
            if (slot < 0) return;
            if (slot >= p.num_slots) {
                if (lane == 0) report(p.status, PA_DEVERR_SLOT);
                return;
            }
            patch_tn = tn;
            if (grp == 0) {
                const int64_t head = (int64_t)hg * HG + h;
                const int64_t src = ((int64_t)s * p.num_kv_heads + head) * D + r * EPV;
                const int64_t dst = (slot * p.num_kv_heads + head) * D + r * EPV;
                using ST = typename T::storage;
                new_k = ldg_stream(reinterpret_cast<const uint4 *>(static_cast<const ST *>(p.new_key) + src));
                new_v = ldg_stream(reinterpret_cast<const uint4 *>(static_cast<const ST *>(p.new_value) + src));
                if (qs == 0) {  // both query slices patch their stage; one stores to the cache
                    *reinterpret_cast<uint4 *>(static_cast<ST *>(p.key_cache_w) + dst) = new_k;
                    *reinterpret_cast<uint4 *>(static_cast<ST *>(p.value_cache_w) + dst) = new_v;
                }
            }
        }
    };

    reset();
    int k = k0, seg_beg = segs[k], seg_end = segs[k + 1];
    int s = k % S, hg = k / S, ctx = context_of(s);
    {
        uint4 raw[G];
        q_global(s, hg, raw);
        load_q(raw, ctx);
    }
    new_token(s, hg, ctx, seg_beg, seg_end);
    bool pf_pending = false;
    int pf_ctx = 0;
    for (int u = u0, i = 0; u < u1; ++u, ++i) {
        if (u >= seg_end) {
            while (u >= seg_end) {
                ++k;
                seg_beg = seg_end;
                seg_end = segs[k + 1];
            }
            s = k % S;
            hg = k / S;
            uint4 raw[G];
            if (pf_pending) {
                q_prefetched(raw);
                ctx = pf_ctx;
                pf_pending = false;
            } else {
                ctx = context_of(s);
                q_global(s, hg, raw);
            }
            load_q(raw, ctx);
            new_token(s, hg, ctx, seg_beg, seg_end);
        }
        if (q_prefetch && u + 1 == seg_end && u + 1 < u1) {  // the next unit starts a segment
            int kn = k + 1;
            while (segs[kn + 1] <= u + 1) ++kn;  // skip segments with nothing to attend
            q_prefetch_issue(kn % S, kn / S);
            pf_ctx = context_of(kn % S);
            pf_pending = true;
        }
        const int stage = i % NSTAGE;
        const uint32_t parity = (i / NSTAGE) & 1;
        const bool ok = !*abort_v && mbar_wait(full0 + 8 * stage, parity, p.status);
        if (!ok) *abort_v = 1;
        [[maybe_unused]] bool patched = false;
        if (ok) {
            const uint32_t kbase = stage_base + stage * 2 * KVB, vbase = kbase + KVB;
            if constexpr (WRITE) {
                if (patch_tn >= 0 && u == seg_end - 1) {  // the new token's rows into the stage
                    if (grp == 0) {
                        const uint32_t off = (uint32_t)((patch_tn * HG + h) * ROWB + r * 16);
                        sts128(kbase + off, new_k);
                        sts128(vbase + off, new_v);
                    }
                    __syncwarp();
                    patched = true;
                }
            }
            const int tok0 = (u - seg_beg) * TU + sb * NT;
            if (tok0 + NT <= ctx)
                consume(kbase, vbase, tok0, ctx, std::false_type{});
            else if (tok0 < ctx)
                consume(kbase, vbase, tok0, ctx, std::true_type{});
        }
        if constexpr (WRITE) {
            // the stage is written by TMA (the async proxy) again after this warp releases it
            if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        if (u == seg_end - 1 || u == u1 - 1) flush(k, seg_beg >= u0 && seg_end <= u1);
    }
    // Every consumer warp's partial stores are done; one thread makes them visible at GPU
    // scope and publishes this launch's tag for each of the CTA's partials.
    named_barrier(1, NW * 32);
    if (warp == 0 && lane == 0 && part0 >= 0) {
        __threadfence();
        store_release(p.tags + 1 + c + part0, p.launch_tag);
        if (part1 >= 0) store_release(p.tags + 1 + c + part1, p.launch_tag);
    }
}

// ------------------------------------------------------------------------------ reduce kernel

constexpr int kMaxPieces = 1024;  // CTAs of the split kernel (one per SM)
constexpr int kReduceBatch = 16;  // pieces whose loads are in flight together

// For every segment split over several CTAs: out = sum_c 2^(m_c - M) acc_c /
// sum_c 2^(m_c - M) l_c.  grid = (segment, group of blockDim.y query heads of the
// group); one thread per pair of outputs of one head.  The launcher packs up to
// kReduceHeads heads per CTA while that still leaves about a wave of CTAs; the CTAs are
// small so that they fit beside the split kernel's and can wait there.  A CTA waits for
// the launch tags of its segment's pieces, not for the split grid to end, then issues the
// loads of a batch of pieces before using any (one round trip for a segment of up to
// kReduceBatch pieces) and merges the batch online (running max).
constexpr int kReduceHeads = 2;
template <int D>
__global__ void __launch_bounds__(D / 2 * kReduceHeads) decode_reduce_kernel(const DecodeParams p, int HGq) {
    // The partials are awaited piece by piece (their launch tags) rather than through the end
    // of the split grid, so that a segment merges as soon as its own CTAs have written it;
    // the wait for the split grid comes last, so that this grid still ends after it.
    __shared__ int ready;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    const int k = blockIdx.x, hl = blockIdx.y * blockDim.y + threadIdx.y, d = threadIdx.x * 2;
    const int S = p.num_seqs, K = p.num_groups * S;
    if (p.tagged && p.scan_in_split) {
        if (tid == 0) ready = wait_tag(p.tags, p.launch_tag, p.status);
    } else {
        pdl_wait_previous();  // the split grid has ended (or, tagged, the plan kernel before it)
        if (tid == 0) ready = 1;
    }
    __syncthreads();
    int c_lo = 0, n = 0;
    if (ready) {
        const int N = load_relaxed_i(p.seg_start + K);
        const int beg = load_relaxed_i(p.seg_start + k), end = load_relaxed_i(p.seg_start + k + 1);
        if (beg != end) {  // else a zero row, written by the split or plan kernel
            const int C = min(p.grid, N);
            c_lo = owner_cta(beg, N, C);
            const int c_hi = owner_cta(end - 1, N, C);
            n = c_hi > c_lo ? c_hi - c_lo + 1 : 0;  // one piece: written by the split kernel
        }
    }
    if (n > 0) {  // the same in every thread of the CTA
        __syncthreads();  // every thread has read `ready`
        if (tid < 32 && p.tagged) {  // lane j waits for the pieces j, j + 32, ...
            bool all = true;
            for (int j = tid; j < n; j += 32) all = wait_tag(p.tags + 1 + c_lo + k + j, p.launch_tag, p.status) && all;
            all = __all_sync(kFullMask, all);
            if (tid == 0) ready = all;
        }
        __syncthreads();
        if (ready && hl < HGq) {
            const int64_t base = (int64_t)(c_lo + k) * HGq + hl;  // piece j is base + j * HGq
            float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f;
            for (int j0 = 0; j0 < n; j0 += kReduceBatch) {
                float mj[kReduceBatch], lj[kReduceBatch];
                float2 oj[kReduceBatch];
#pragma unroll
                for (int i = 0; i < kReduceBatch; ++i) {
                    const int64_t pi = base + (int64_t)(j0 + i) * HGq;
                    const bool ok = j0 + i < n;
                    mj[i] = ok ? load_relaxed(p.part_m + pi) : -INFINITY;
                    lj[i] = ok ? load_relaxed(p.part_l + pi) : 0.f;
                    oj[i] = ok ? load_relaxed2(p.part_o + pi * D + d) : make_float2(0.f, 0.f);
                }
                float bm = M;
#pragma unroll
                for (int i = 0; i < kReduceBatch; ++i) bm = fmaxf(bm, mj[i]);
                const float a = fast_exp2(M - bm);  // 0 on the first batch
                L *= a;
                o0 *= a;
                o1 *= a;
#pragma unroll
                for (int i = 0; i < kReduceBatch; ++i) {
                    const float f = fast_exp2(mj[i] - bm);  // 0 for padding entries
                    L = fmaf(lj[i], f, L);
                    o0 = fmaf(oj[i].x, f, o0);
                    o1 = fmaf(oj[i].y, f, o1);
                }
                M = bm;
            }
            const float inv = 1.f / L;
            const int s = k % S, hg = k / S;
            store_pair_any(p.out, p.out_dtype, ((int64_t)s * p.num_heads + hg * HGq + hl) * D + d, o0 * inv,
                           o1 * inv);
        }
    }
    pdl_wait_previous();  // this grid ends after the split kernel (whose whole segments it does not await)
}

template <class T, int D, int G, int QS, bool ROPE, bool WRITE>
int launch_typed(DecodeParams prm, const CUtensorMap &km, const CUtensorMap &vm, cudaStream_t st) {
    using Sh = DecodeShape<T, D, G, QS>;
    static std::atomic<int> smem_ready[kMaxDevices];  // per device: shared-memory limit raised
    prm.unit_tokens = Sh::NT * (kConsumerWarps / (prm.heads_per_group * QS));
    prm.box_rows = prm.block_size < prm.unit_tokens ? prm.block_size : prm.unit_tokens;
    const bool fused = prm.num_groups * prm.num_seqs < kSegSmem;  // scan inside the split kernel
    prm.scan_in_split = fused ? 1 : 0;
    // reduce: heads per CTA, as many as keep about 128 CTAs (one wave)
    const int K = prm.num_groups * prm.num_seqs, HGq = prm.heads_per_group * G * QS;
    int rh = kReduceHeads;
    while (rh > 1 && (int64_t)K * ((HGq + rh - 1) / rh) < 128) rh >>= 1;
    if ((!fused &&
         launch_pdl(decode_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, prm) != cudaSuccess) ||
        launch_pdl_smem(decode_split_kernel<T, D, G, QS, ROPE, WRITE>, smem_ready, dim3(prm.grid), dim3(kDecodeThreads),
                        Sh::SMEM, st, km, vm, prm) != cudaSuccess ||
        launch_pdl(decode_reduce_kernel<D>, dim3(K, (HGq + rh - 1) / rh), dim3(D / 2, rh), 0, st, prm, HGq) !=
            cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

template <class T, int D, bool ROPE, bool WRITE>
int dispatch_g(const DecodeParams &prm, int G, const CUtensorMap &km, const CUtensorMap &vm,
               cudaStream_t st) {
    switch (G) {
        case 1: return launch_typed<T, D, 1, 1, ROPE, WRITE>(prm, km, vm, st);
        case 2: return launch_typed<T, D, 2, 1, ROPE, WRITE>(prm, km, vm, st);
        case 4: return launch_typed<T, D, 4, 1, ROPE, WRITE>(prm, km, vm, st);
        case 8: return launch_typed<T, D, 4, 2, ROPE, WRITE>(prm, km, vm, st);  // two query slices
        default: return PA_ERR_UNSUPPORTED;
    }
}

template <class T, bool ROPE, bool WRITE>
int dispatch_d(const DecodeParams &prm, int D, int G, const CUtensorMap &km, const CUtensorMap &vm,
               cudaStream_t st) {
    switch (D) {
        case 64: return dispatch_g<T, 64, ROPE, WRITE>(prm, G, km, vm, st);
        case 128: return dispatch_g<T, 128, ROPE, WRITE>(prm, G, km, vm, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

// Typed dispatch of one decode call on the cache format, head dim and group size.
template <bool ROPE, bool WRITE = false>
int dispatch_kv(const DecodeParams &prm, pa_dtype kv_dtype, int D, int G, const CUtensorMap &km,
                const CUtensorMap &vm, cudaStream_t st) {
    switch (kv_dtype) {
        case PA_F32: return dispatch_d<F32, ROPE, WRITE>(prm, D, G, km, vm, st);
        case PA_F16: return dispatch_d<F16, ROPE, WRITE>(prm, D, G, km, vm, st);
        case PA_BF16: return dispatch_d<BF16, ROPE, WRITE>(prm, D, G, km, vm, st);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace pa
