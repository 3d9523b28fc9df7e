// prefill.cu -- chunked-prefill paged attention on the 5th-generation tensor
// cores (tcgen05: operands in shared memory via TMA, accumulators in TMEM).
//
// A chunk of Lq query tokens per sequence (the newest tokens, whose K/V the
// caller already wrote into the cache) attends the sequence's keys gathered
// through its block table: full attention over the cached prefix, causal
// inside the chunk, rows aligned bottom-right (row i at absolute position
// C - Lq + i).  mistral.rs page, scheduling section (long prompts chunked
// under a token budget, 512 tokens per chunk); TensorSharp "Mistral 3" page,
// section 11 (paged K/V gather, then fused attention).
//
// A work unit is one query tile of one sequence; a tile is 128 rows of
// (token, head) pairs of ONE kv head's G query heads (128/G tokens), so each
// gathered K/V tile serves G heads.  An item is a unit for one kv head.
// Persistent grid: one CTA per SM walks its items back to back, so the fixed
// cost of a CTA (barrier setup, TMEM allocation, pipeline fill, epilogue) is
// paid once per SM and the next item's loads and S products overlap the
// previous item's last P.V and epilogue.  Units differ in cost by their number
// of key tiles (a tile deep in a long prefix sees many more keys than the first
// tile of a fresh prompt), so every CTA first ranks all units longest-first
// from the query and context lengths (a stable counting sort in shared memory,
// identical in every CTA) and the CTAs deal the ranked items out round by
// round, alternating direction.
// Per 128-key tile j:
//   S_j = Q K_j^T   tcgen05.mma M128 N128 K=D, fp32 in TMEM (three buffers, so
//                   the S products run up to three tiles ahead)
//   P_j             the softmax warps read S from TMEM (a row spread over
//                   four lanes): mask, online softmax in the log2 domain with
//                   lazy rescaling (the reference max moves only when a score
//                   exceeds it by 2^8), P_j rounded to bf16/fp16 and written
//                   back to TMEM over the S row
//   O  += P_j V_j   tcgen05.mma M128 N=D K128 with A = P from TMEM, fp32 in
//                   TMEM; V is the MN-major shared-memory operand
// Warp roles: warps 0 and 2 issue the TMA loads (the Q tile; per key tile one
// 5-D box per block through the block table, issued by the lanes in parallel,
// into separate K and V rings: a K stage frees when its S finishes, a V stage
// when its P.V does), warp 1 issues the S products and warp 3 the P.V products
// (a thread waits for each MMA to be accepted, so one issuer cannot keep the
// tensor core busy), warps 4-11 run the softmax and the epilogue, two warps per
// TMEM lane quarter, each on a 16-row slab through the 16-lane TMEM shapes (a row's
// keys spread over four lanes).  All shared-memory operands use the 128-byte swizzle.
// Every mbarrier wait is bounded in time.
#include <algorithm>
#include <type_traits>

#include "tma.cuh"

namespace pa {
namespace {

constexpr int kPfThreads = 12 * 32;
constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 128;  // keys per tile
constexpr float kRescaleLog2 = 8.f;

// ---------------------------------------------------------------- tcgen05 helpers
// Shared-memory matrix descriptor (sm_100 format): start address, leading and
// stride byte offsets (>> 4), version 1, 128-byte swizzle.  K-major operands:
// SBO = 1024 (between 8-row groups), the start advances 32 bytes per 16-element
// k step inside the swizzle span.  MN-major operands: LBO = bytes between
// 64-element atoms along MN, SBO = 1024 (between 8-row groups along K).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation, A K-major.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, bool bf16, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

// Same, with A (M x 16 elements) read from TMEM: row i in lane i, two 16-bit
// elements per 32-bit column, 8 columns per k step.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t db,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(db), "r"(idesc), "r"(accumulate));
}

// The mbarrier completes one arrival when every MMA issued so far has finished.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 lanes x N groups of 8 consecutive 32-bit columns -> 4N registers per thread: thread t
// holds rows t/4 and t/4 + 8 of the 16, columns 8j + 2(t%4) and the next one of group j, as
// registers 4j, 4j+1 (first row) and 4j+2, 4j+3 (second row).
template <int N>
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&r)[4 * N]);
template <>
__device__ __forceinline__ void tmem_ld_16x256b<8>(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// The 16-lane shapes in the other direction: 16x256b as loaded above, and 16x128b, where
// thread t holds column 4j + t%4 of rows t/4 and t/4 + 8 of group j (registers 2j, 2j+1).
__device__ __forceinline__ void tmem_st_16x256b_x8(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_16x128b_x16(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Generic-proxy shared-memory writes become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// max(a, b, c) in one instruction (returns the other operands when one is NaN)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

template <class T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<BF16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<F16>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// A packed pair widened to fp32 exactly as it enters the P.V product, so that the
// row sum (denominator) adds the same rounded weights as the numerator.
template <class T>
__device__ __forceinline__ float2 unpack2(uint32_t u);
template <>
__device__ __forceinline__ float2 unpack2<BF16>(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<F16>(uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2 *>(&u));
}

struct PrefillParams {
    void *out;
    pa_dtype out_dtype;
    const int32_t *query_start_loc;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int max_blocks_per_seq, num_heads, num_kv_heads, block_size, num_blocks, max_context_len;
    int num_tokens, num_seqs;
    int q_tiles;    // query tiles per sequence (of the longest chunk)
    int num_items;  // num_seqs * q_tiles * num_kv_heads
    float qk_scale_log2;
    int32_t *status;
};

// The kernels' DR (decode rows) instantiations: sequence s has one query row, token s, at
// position context_lens[s] - 1 (query_start_loc is not read); a sequence with nothing to
// attend gets zero rows, and a negative or too long context is reported and clamped, as in
// the decode kernels.  The other instantiations never see these branches.

// ---------------------------------------------------------------- work items and their order
// A unit is (sequence s, query tile qt), numbered s * q_tiles + qt; an item is (unit, kv
// head).  Items are ranked unit-major: the units of rank r give items r*Hkv .. r*Hkv+Hkv-1.
// CTA c of P takes one item per round k, item k*P + c in even rounds and k*P + P-1-c in odd
// ones, so that each CTA's total of light and heavy items evens out.
constexpr int kPlanMaxUnits = 4096;  // more units: rank r is unit r (latest tile first)
constexpr int kPlanBins = 1024;      // key-tile counts; longer units share the last bin
constexpr int kMaxRounds = 32;       // more items per CTA: no ranking either

__device__ __forceinline__ int64_t round_item(int k, int P, int c) {
    return (int64_t)k * P + ((k & 1) ? P - 1 - c : c);
}

// Key tiles the unit (s, qt) runs through; 0 for an empty or invalid unit.
template <bool DR>
__device__ __forceinline__ int unit_tiles(const PrefillParams &p, int s, int qt, int TT) {
    int q0, Lq;
    if constexpr (DR) {
        q0 = s;
        Lq = 1;
    } else {
        q0 = p.query_start_loc[s];
        Lq = p.query_start_loc[s + 1] - q0;
    }
    if (q0 < 0 || Lq < 0 || (int64_t)q0 + Lq > p.num_tokens || qt * TT >= Lq) return 0;
    const int C = min(p.context_lens[s], min(p.max_blocks_per_seq * p.block_size, p.max_context_len));
    if (Lq > C) return 0;
    return (C - Lq + min(Lq, (qt + 1) * TT) + kBN - 1) / kBN;
}

// Ranks the units by key tiles, most first, ties in unit order (a stable counting sort in
// shared memory: every CTA computes the same order), and lists the unit of each of this
// CTA's rounds in my_units.  Called by every thread; `scratch` is shared memory that
// nothing else touches until the call returns.
template <bool DR>
__device__ void plan_units(const PrefillParams &p, int TT, int P, int c, unsigned char *scratch,
                           uint16_t *my_units) {
    const int Q = p.q_tiles, U = p.num_seqs * Q;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    constexpr int NT = kPfThreads;
    auto hslot = [](int b) { return b + (b >> 5); };  // padded: a lane's 32 bins hit 32 banks
    int *hist = reinterpret_cast<int *>(scratch);
    uint16_t *wt = reinterpret_cast<uint16_t *>(hist + kPlanBins + kPlanBins / 32);
    uint16_t *order = wt + kPlanMaxUnits;
    for (int i = tid; i < kPlanBins + kPlanBins / 32; i += NT) hist[i] = 0;
    __syncthreads();
    for (int u = tid; u < U; u += NT) {
        const int w = min(unit_tiles<DR>(p, u / Q, u % Q, TT), kPlanBins - 1);
        wt[u] = (uint16_t)w;
        atomicAdd(&hist[hslot(w)], 1);
    }
    __syncthreads();
    if (warp == 0) {
        // hist[b] <- number of units with more key tiles than b; lane l owns the bins
        // 1023-32l down to 992-32l
        int sum = 0;
        for (int i = 0; i < 32; ++i) sum += hist[hslot(kPlanBins - 1 - (lane * 32 + i))];
        int inc = sum;
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFullMask, inc, o);
            if (lane >= o) inc += t;
        }
        int acc = inc - sum;
        for (int i = 0; i < 32; ++i) {
            const int b = hslot(kPlanBins - 1 - (lane * 32 + i)), h = hist[b];
            hist[b] = acc;
            acc += h;
        }
        __syncwarp();
        // scatter 32 units at a time in unit order; lanes of equal weight take consecutive
        // ranks and the lowest of them advances the bin's next rank
        for (int base = 0; base < U; base += 32) {
            const int u = base + lane;
            const int w = u < U ? wt[u] : -1;
            const unsigned peers = __match_any_sync(kFullMask, w);
            if (u < U) order[hist[hslot(w)] + __popc(peers & ((1u << lane) - 1u))] = (uint16_t)u;
            __syncwarp();
            if (u < U && lane == __ffs(peers) - 1) hist[hslot(w)] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int k = tid; k < kMaxRounds; k += NT) {
        const int64_t idx = round_item(k, P, c);
        if (idx < p.num_items) my_units[k] = order[idx / p.num_kv_heads];
    }
    __syncthreads();
    // the scratch becomes a TMA destination: order these generic accesses before it
    fence_async_smem();
}

// One item's scalars.  fetch() issues the loads of round k; resolve() turns them into the
// item (false when it has no rows, with a status bit when the inputs are invalid).
struct PfItem {
    int s, qt, g, q0, Lq, C, tok_begin, pos0, kv_end, n_tiles;
};
struct PfCursor {
    bool have;
    int unit, g, q0, q1, C;

    template <bool DR>
    __device__ __forceinline__ void fetch(const PrefillParams &p, int k, bool planned,
                                          const uint16_t *my_units) {
        const int P = gridDim.x, c = blockIdx.x;
        const int64_t idx = round_item(k, P, c);
        have = idx < p.num_items;
        if (!have) return;
        const int rank = (int)(idx / p.num_kv_heads), Q = p.q_tiles;
        g = (int)(idx % p.num_kv_heads);
        unit = planned ? my_units[k] : (rank / Q) * Q + Q - 1 - rank % Q;
        const int s = unit / Q;
        if constexpr (DR) {
            q0 = s;
            q1 = s + 1;
        } else {
            q0 = p.query_start_loc[s];
            q1 = p.query_start_loc[s + 1];
        }
        C = p.context_lens[s];
    }

    template <bool DR>
    __device__ __forceinline__ bool resolve(const PrefillParams &p, int TT, bool rep, PfItem &it) const {
        it.s = unit / p.q_tiles;
        it.qt = unit % p.q_tiles;
        it.g = g;
        it.q0 = q0;
        it.Lq = q1 - q0;
        if (q0 < 0 || it.Lq < 0 || (int64_t)q0 + it.Lq > p.num_tokens) {  // never index past the query
            if (rep) report(p.status, PA_DEVERR_QUERY);
            return false;
        }
        if (it.qt * TT >= it.Lq) return false;
        const int cap = min(p.max_blocks_per_seq * p.block_size, p.max_context_len);
        int Cc = C;
        if constexpr (DR) {
            if (Cc < 0 || Cc > cap) {
                if (rep) report(p.status, PA_DEVERR_CONTEXT);
                Cc = Cc < 0 ? 0 : cap;
            }
            if (Cc == 0) return false;  // a zero row, written at the start
        }
        if (Cc > cap || it.Lq > Cc) {
            if (rep) report(p.status, Cc > cap ? PA_DEVERR_CONTEXT : PA_DEVERR_QUERY);
            if (Cc > cap) Cc = cap;
            if (it.Lq > Cc) return false;
        }
        it.C = Cc;
        it.tok_begin = it.qt * TT;
        it.pos0 = Cc - it.Lq;                                     // absolute position of chunk row 0
        it.kv_end = it.pos0 + min(it.Lq, it.tok_begin + TT);      // keys visible to the tile's last row
        it.n_tiles = (it.kv_end + kBN - 1) / kBN;
        return true;
    }
};

template <int D>
struct PfShape {
    static constexpr int HALVES = D / 64;             // 128-byte swizzle atoms along D
    static constexpr int Q_BYTES = kBM * D * 2;       // [half][128 rows][128 B]
    static constexpr int KV_BYTES = kBN * D * 2;      // one K (or V) stage: [8-key group][slice][8 keys][128 B]
    static constexpr int GSTR = HALVES * 1024;        // bytes between 8-key groups of a K / V stage
    static constexpr int NQ = D == 64 ? 2 : 1;        // Q buffers
    static constexpr int NK = D == 64 ? 4 : 3;        // K stages
    static constexpr int NV = D == 64 ? 4 : 3;        // V stages
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    // the unit plan borrows the K ring before the first load
    static_assert((kPlanBins + kPlanBins / 32) * 4 + 2 * kPlanMaxUnits * 2 <= NK * KV_BYTES,
                  "plan scratch fits the K ring");
};

// TMEM columns: S (fp32, 128 keys) in three buffers, S_t in buffer t % 3; P_t (two
// bf16/fp16 keys per column) is written over the first 64 columns of S_t's buffer once
// S_t has been read; O (fp32, D) after them.  Three buffers let the S products run up to
// three tiles ahead of the P.V products, so the softmax never waits for an S.
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;
constexpr uint32_t kTmemO = kSBufs * kBN;

template <class T, int D, int G, bool DR>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using Sh = PfShape<D>;
    constexpr int NQ = Sh::NQ, NK = Sh::NK, NV = Sh::NV;
    constexpr int TT = kBM / G;  // query tokens per tile
    constexpr int KSTEPS_S = D / 16, KSTEPS_PV = kBN / 16;
    constexpr bool kBf16 = std::is_same<T, BF16>::value;
    constexpr uint32_t IDESC_S = mma_idesc(128, kBN, kBf16, false);
    constexpr uint32_t IDESC_PV = mma_idesc(128, D, kBf16, true);
    static_assert(kTmemO + D <= kTmemCols, "TMEM budget");

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ0 = sbase + Sh::OFF_Q, sK0 = sbase + Sh::OFF_K, sV0 = sbase + Sh::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sh::OFF_BAR);
    const uint32_t b0 = smem_u32(bars);
    auto bar = [&](int i) { return b0 + 8 * i; };
    constexpr int BQF = 0;              // Q buffer landed
    constexpr int BQE = BQF + NQ;       // last S of that Q's item finished
    constexpr int BKF = BQE + NQ;       // K stage landed
    constexpr int BKE = BKF + NK;       // S of that K finished
    constexpr int BVF = BKE + NK;       // V stage landed
    constexpr int BVE = BVF + NV;       // P.V of that V finished
    constexpr int BSF = BVE + NV;       // S buffer written
    constexpr int BPF = BSF + kSBufs;   // P written over that S buffer
    constexpr int BPV = BPF + kSBufs;   // P.V of that buffer's P finished
    constexpr int NBAR = BPV + kSBufs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
    int *abort_flag = reinterpret_cast<int *>(bars + NBAR) + 1;
    uint16_t *my_units = reinterpret_cast<uint16_t *>(bars + NBAR + 1);
    static_assert((NBAR + 1) * 8 + kMaxRounds * 2 <= 512, "barrier area");

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int Hq = p.num_heads, bs = p.block_size;

    // ---- prologue independent of earlier kernels
    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i >= BPF && i < BPF + kSBufs) ? 8 : 1);
        fence_barrier_init();
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    pdl_wait_previous();
    pdl_launch_dependents();

    const int rounds = (p.num_items + gridDim.x - 1) / gridDim.x;
    const bool planned = p.num_seqs * p.q_tiles <= kPlanMaxUnits && rounds <= kMaxRounds;
    if (planned) plan_units<DR>(p, TT, gridDim.x, blockIdx.x, smem + Sh::OFF_K, my_units);

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int *abort_v = abort_flag;
    // Every role walks the same items (a cursor runs one round ahead so that the next
    // item's scalars are in flight) and counts the same global key tiles t, which pick
    // ring stages, S/P buffers and their phases; vi counts the items with rows and picks
    // the Q buffer.
    PfCursor cur;

    if (warp == 0 || warp == 2) {
        // ============================================ producers (TMA): warp 0 loads Q and K, warp 2 V
        // A K stage frees when its S finishes, a V stage when its P.V does, the Q buffer
        // when its item's last S does.  Lane b fetches the block id of the tile's b-th
        // block two tiles ahead and issues that block's boxes; lane 0 posts the tile's
        // transaction bytes first and arrives after the warp has issued.
        const bool is_k = warp == 0;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t ring = is_k ? sK0 : sV0;
        const int NS = is_k ? NK : NV;
        const int bar_full = is_k ? BKF : BVF, bar_empty = is_k ? BKE : BVE;
        const uint64_t policy = policy_evict_first();
        const int nb = kBN / bs;  // blocks per key tile (4, 8 or 16)
        const uint32_t box_bytes = (uint32_t)bs * 128 * Sh::HALVES;  // one block of one kv head
        bool ok = true;
        int t = 0, vi = 0;
        cur.fetch<DR>(p, 0, planned, my_units);
        for (int k = 0; ok && cur.have; ++k) {
            PfItem it;
            const bool live = cur.resolve<DR>(p, TT, false, it);
            cur.fetch<DR>(p, k + 1, planned, my_units);
            if (!live) continue;
            const int32_t *bt = p.block_tables + (int64_t)it.s * p.max_blocks_per_seq;
            auto block_id = [&](int j) {
                const int key = j * kBN + lane * bs;
                return (lane < nb && j < it.n_tiles && key < it.kv_end) ? bt[key / bs] : -1;
            };
            int id0 = block_id(0), id1 = block_id(1);
            if (is_k) {  // Q: tokens [tok_begin, +TT) x heads [g*G, +G), one D half per box
                const int qb = vi % NQ;
                int q_ok = 1;
                if (lane == 0) {
                    q_ok = !*abort_v && mbar_wait(bar(BQE + qb), ((vi / NQ) & 1) ^ 1, p.status);
                    if (q_ok) {
                        mbar_expect_tx(bar(BQF + qb), Sh::Q_BYTES);
                        for (int hf = 0; hf < Sh::HALVES; ++hf)
                            tma_load_3d(sQ0 + qb * Sh::Q_BYTES + hf * (kBM * 128), &qmap, hf * 64,
                                        it.g * G, it.q0 + it.tok_begin, bar(BQF + qb), policy);
                        mbar_arrive(bar(BQF + qb));
                    }
                }
                if (!__shfl_sync(kFullMask, q_ok, 0)) {
                    ok = false;
                    break;
                }
            }
            for (int j = 0; j < it.n_tiles; ++j, ++t) {
                const int my_id = id0;
                id0 = id1;
                id1 = block_id(j + 2);
                const int st = t % NS;
                const uint32_t full = bar(bar_full + st);
                int w_ok = 1;
                if (lane == 0) w_ok = !*abort_v && mbar_wait(bar(bar_empty + st), ((t / NS) & 1) ^ 1, p.status);
                if (!__shfl_sync(kFullMask, w_ok, 0)) {
                    ok = false;
                    break;
                }
                const bool in_range = lane < nb && j * kBN + lane * bs < it.kv_end;
                const bool valid = in_range && my_id >= 0 && my_id < p.num_blocks;
                if (in_range && !valid) report(p.status, PA_DEVERR_BLOCK_ID);  // never dereferenced
                const unsigned mine = __ballot_sync(kFullMask, valid);
                if (lane == 0) mbar_expect_tx(full, __popc(mine) * box_bytes);
                __syncwarp();
                if (valid) {
                    const uint32_t dst = ring + st * Sh::KV_BYTES + lane * box_bytes;
                    tma_load_5d(dst, map, 0, 0, 0, my_id * (bs / 8), it.g, full, policy);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
            }
            ++vi;
        }
        if (!ok && lane == 0) *abort_v = 1;
    } else if (warp == 1) {
        // ============================================ S issuer: S_t = Q K_t^T
        // The S and P.V products are issued by two threads (warps 1 and 3): one thread
        // waits for each tcgen05.mma to be accepted, so a single issuer keeps the tensor
        // core only about half busy.  S runs up to three tiles ahead of the P.V products;
        // S_t overwrites the P of tile t-3, so it waits until that P.V has finished.
        if (lane == 0) {
            bool ok = true;
            int t = 0, vi = 0;
            cur.fetch<DR>(p, 0, planned, my_units);
            for (int k = 0; ok && cur.have; ++k) {
                PfItem it;
                const bool live = cur.resolve<DR>(p, TT, false, it);
                cur.fetch<DR>(p, k + 1, planned, my_units);
                if (!live) continue;
                const int qb = vi % NQ;
                ok = !*abort_v && mbar_wait(bar(BQF + qb), (vi / NQ) & 1, p.status);
                const uint32_t sQ = sQ0 + qb * Sh::Q_BYTES;
                for (int j = 0; j < it.n_tiles && ok; ++j, ++t) {
                    const int st = t % NK, sb = t % kSBufs;
                    if (t >= kSBufs) ok = mbar_wait(bar(BPV + sb), (t / kSBufs - 1) & 1, p.status);
                    ok = ok && !*abort_v && mbar_wait(bar(BKF + st), (t / NK) & 1, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sK = sK0 + st * Sh::KV_BYTES;
#pragma unroll
                    for (int ks = 0; ks < KSTEPS_S; ++ks) {
                        const uint32_t off = (ks / 4) * (kBM * 128) + (ks % 4) * 32;
                        const uint32_t offk = (ks / 4) * 1024 + (ks % 4) * 32;
                        mma_f16(tmem + sb * kBN, smem_desc(sQ + off, 16, 1024), smem_desc(sK + offk, 16, Sh::GSTR),
                                IDESC_S, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(BSF + sb));
                    mma_commit(bar(BKE + st));
                }
                if (ok) mma_commit(bar(BQE + qb));  // the Q buffer is free once these S finish
                ++vi;
            }
            if (!ok) *abort_v = 1;
        }
    } else if (warp == 3) {
        // ============================================ P.V issuer: O += P_t V_t, P from TMEM
        if (lane == 0) {
            bool ok = true;
            int t = 0;
            cur.fetch<DR>(p, 0, planned, my_units);
            for (int k = 0; ok && cur.have; ++k) {
                PfItem it;
                const bool live = cur.resolve<DR>(p, TT, false, it);
                cur.fetch<DR>(p, k + 1, planned, my_units);
                if (!live) continue;
                for (int j = 0; j < it.n_tiles && ok; ++j, ++t) {
                    const int pb = t % kSBufs, st = t % NV;
                    ok = !*abort_v && mbar_wait(bar(BPF + pb), (t / kSBufs) & 1, p.status) &&
                         mbar_wait(bar(BVF + st), (t / NV) & 1, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sV = sV0 + st * Sh::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_PV; ++kk) {
                        const uint64_t db = smem_desc(sV + kk * 2 * Sh::GSTR, 1024, Sh::GSTR);
                        mma_f16_tmem_a(tmem + kTmemO, tmem + pb * kBN + kk * 8, db, IDESC_PV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(BPV + pb));
                    mma_commit(bar(BVE + st));
                }
            }
            if (!ok) *abort_v = 1;
        }
    } else {
        // ============================================ softmax (row slabs)
        // Warps 4-7 take rows 0-15 and warps 8-11 rows 16-31 of the TMEM lane quarter
        // warp % 4, through the 16-lane TMEM shapes: in 16x256b a thread holds rows t/4 and
        // t/4 + 8 of its slab, keys 8j + 2(t%4) and the next one of each group of 8, so a row
        // is spread over the four lanes 4(t/4) .. 4(t/4)+3 (row maxima and sums are two
        // shuffles among them) and the pair of keys a thread holds packs into the P column
        // 4j + t%4, exactly the 16x128b store layout.  The two warps of a quarter share no
        // state, so each hides the other's latencies.
        const int quarter = warp & 3;
        const int slab = warp >= 8 ? 1 : 0;
        const int gi = lane >> 2, ga = lane & 3;
        const int sidx = (warp - 4) * 32 + lane;      // 0..255 over the softmax threads
        const int lane0 = quarter * 32 + slab * 16;   // first TMEM lane (tile row) of the slab
        const int row0 = lane0 + gi, row1 = row0 + 8; // this thread's two rows of the tile
        const uint32_t lane_off = (uint32_t)lane0 << 16;
        const uint32_t tO = tmem + lane_off + kTmemO;
        const float sc = p.qk_scale_log2;
        bool ok = true;
        int t = 0;
        if constexpr (DR) {  // zero rows for the sequences with nothing to attend
            const int cap = min(p.max_blocks_per_seq * p.block_size, p.max_context_len);
            const int words = p.num_heads * D * (p.out_dtype == PA_F32 ? 4 : 2) / 4;
            for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x) {
                if (min(p.context_lens[s], cap) > 0) continue;
                uint32_t *row = static_cast<uint32_t *>(p.out) + (int64_t)s * words;
                for (int i = sidx; i < words; i += 256) row[i] = 0u;
            }
        }
        cur.fetch<DR>(p, 0, planned, my_units);
        for (int k = 0; ok && cur.have; ++k) {
            PfItem it;
            const bool live = cur.resolve<DR>(p, TT, warp == 4 && lane == 0, it);
            cur.fetch<DR>(p, k + 1, planned, my_units);
            if (!live) continue;
            // rows past the chunk (a ragged last tile) are computed but never stored; they
            // see exactly the keys that were loaded
            const int pos0 = min(it.pos0 + it.tok_begin + row0 / G, it.kv_end - 1);
            const int pos1 = min(it.pos0 + it.tok_begin + row1 / G, it.kv_end - 1);
            const int row0_pos = it.pos0 + it.tok_begin;  // position of the tile's first row
            float m0 = -INFINITY, m1 = -INFINITY;        // reference maxima (log2 domain)
            float l0 = 0.f, l1 = 0.f;                     // this lane's share of the row sums
            for (int j = 0; j < it.n_tiles; ++j, ++t) {
                const int sb = t % kSBufs;
                ok = __all_sync(kFullMask, ok && !*abort_v && mbar_wait(bar(BSF + sb), (t / kSBufs) & 1, p.status));
                if (!ok) break;
                tc_fence_after();
                const int k0 = j * kBN;
                const uint32_t tS = tmem + lane_off + sb * kBN;
                uint32_t s[2][32];  // keys 0-63 and 64-127 of the tile
                tmem_ld_16x256b<8>(tS, s[0]);
                tmem_ld_16x256b<8>(tS + 64, s[1]);
                tmem_wait_ld();
                // mask (keys k0 .. k0+lim-1 are visible to a row; only the last tiles need it)
                if (k0 + kBN > row0_pos + 1 || k0 + kBN > it.C) {  // tile-uniform
                    const int lim0 = min(pos0 + 1, it.C) - k0, lim1 = min(pos1 + 1, it.C) - k0;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int g = 0; g < 8; ++g)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int key = h * 64 + 8 * g + 2 * ga + e;
                                if (key >= lim0) s[h][4 * g + e] = __float_as_uint(-INFINITY);
                                if (key >= lim1) s[h][4 * g + 2 + e] = __float_as_uint(-INFINITY);
                            }
                }
                // row maxima: 32 scores per row in this lane, then over the row's four lanes
                float a0 = -INFINITY, a1 = -INFINITY, b0 = -INFINITY, b1 = -INFINITY;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int g = 0; g < 8; g += 2) {
                        a0 = fmax3(a0, __uint_as_float(s[h][4 * g]), __uint_as_float(s[h][4 * g + 1]));
                        b0 = fmax3(b0, __uint_as_float(s[h][4 * g + 4]), __uint_as_float(s[h][4 * g + 5]));
                        a1 = fmax3(a1, __uint_as_float(s[h][4 * g + 2]), __uint_as_float(s[h][4 * g + 3]));
                        b1 = fmax3(b1, __uint_as_float(s[h][4 * g + 6]), __uint_as_float(s[h][4 * g + 7]));
                    }
                float mx0 = fmaxf(a0, b0), mx1 = fmaxf(a1, b1);
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, 2)) * sc;
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, 2)) * sc;
                // lazy rescale; warp-uniform because the O rows are read and written by the
                // whole warp (tcgen05.ld / st).  The four lanes of a row hold the same maxima.
                const bool grow0 = mx0 > m0 + kRescaleLog2, grow1 = mx1 > m1 + kRescaleLog2;
                if (__any_sync(kFullMask, grow0 || grow1)) {
                    const float n0 = grow0 ? mx0 : m0, n1 = grow1 ? mx1 : m1;
                    const float al0 = n0 == m0 ? 1.f : fast_exp2(m0 - n0);  // 0 from -inf
                    const float al1 = n1 == m1 ? 1.f : fast_exp2(m1 - n1);
                    l0 *= al0;
                    l1 *= al1;
                    m0 = n0;
                    m1 = n1;
                    if (j >= 1) {  // O holds tiles < j: wait for the last P.V, then scale the rows
                        ok = __all_sync(kFullMask, mbar_wait(bar(BPV + (t - 1) % kSBufs), ((t - 1) / kSBufs) & 1,
                                                             p.status));
                        if (ok) {
                            tc_fence_after();
#pragma unroll
                            for (int c0 = 0; c0 < D; c0 += 64) {
                                uint32_t o[32];
                                tmem_ld_16x256b<8>(tO + c0, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int g = 0; g < 8; ++g) {
                                    o[4 * g] = __float_as_uint(__uint_as_float(o[4 * g]) * al0);
                                    o[4 * g + 1] = __float_as_uint(__uint_as_float(o[4 * g + 1]) * al0);
                                    o[4 * g + 2] = __float_as_uint(__uint_as_float(o[4 * g + 2]) * al1);
                                    o[4 * g + 3] = __float_as_uint(__uint_as_float(o[4 * g + 3]) * al1);
                                }
                                tmem_st_16x256b_x8(tO + c0, o);
                            }
                            tmem_wait_st();
                        }
                    }
                }
                // P over the S rows (the P.V of this buffer's previous tile finished before this
                // S was issued): the weights of keys 8j + 2(t%4), +1 pack into P column 4j + t%4
                {
                    const float mb0 = m0 == -INFINITY ? 0.f : m0, mb1 = m1 == -INFINITY ? 0.f : m1;
                    const float2 sc2 = make_float2(sc, sc);
                    const float2 nm0 = make_float2(-mb0, -mb0), nm1 = make_float2(-mb1, -mb1);
                    float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
                    uint32_t pw[32];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const float2 x0 = __ffma2_rn(
                                make_float2(__uint_as_float(s[h][4 * g]), __uint_as_float(s[h][4 * g + 1])), sc2, nm0);
                            const float2 x1 = __ffma2_rn(
                                make_float2(__uint_as_float(s[h][4 * g + 2]), __uint_as_float(s[h][4 * g + 3])), sc2,
                                nm1);
                            const uint32_t w0 = pack2<T>(fast_exp2(x0.x), fast_exp2(x0.y));
                            const uint32_t w1 = pack2<T>(fast_exp2(x1.x), fast_exp2(x1.y));
                            pw[2 * (h * 8 + g)] = w0;
                            pw[2 * (h * 8 + g) + 1] = w1;
                            rs0 = __fadd2_rn(rs0, unpack2<T>(w0));
                            rs1 = __fadd2_rn(rs1, unpack2<T>(w1));
                        }
                    if (ok) {
                        tmem_st_16x128b_x16(tS, pw);
                        tmem_wait_st();
                    }
                    l0 += rs0.x + rs0.y;
                    l1 += rs1.x + rs1.y;
                }
                // keys past kv_end in this tile (not loaded, or past the context): zero V rows,
                // so that 0-weight rows never meet stale or NaN data
                if (k0 + kBN > it.kv_end) {
                    const int valid = it.kv_end - k0, st = t % NV;
                    ok = __all_sync(kFullMask, ok && mbar_wait(bar(BVF + st), (t / NV) & 1, p.status));
                    const uint32_t sV = sV0 + st * Sh::KV_BYTES;
                    if (ok)
                        for (int i = sidx; i < (kBN - valid) * Sh::HALVES * 8; i += 256) {
                            const int rr = valid + i / (Sh::HALVES * 8), rest = i % (Sh::HALVES * 8);
                            sts128(sV + (rr / 8) * Sh::GSTR + (rest / 8) * 1024 + (rr % 8) * 128 + (rest % 8) * 16, 0u,
                                   0u, 0u, 0u);
                        }
                    fence_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (ok && lane == 0) mbar_arrive(bar(BPF + sb));
                if (!ok) break;
            }
            if (!ok) break;
            // ---- epilogue: O / l for the rows of this chunk.  The next item's first P.V
            // (which overwrites O) waits for P written later by all eight warps, each after
            // reading its own rows here.
            const int last = t - 1;
            ok = __all_sync(kFullMask, mbar_wait(bar(BPV + last % kSBufs), (last / kSBufs) & 1, p.status));
            if (!ok) break;
            tc_fence_after();
            float L0 = l0 + __shfl_xor_sync(kFullMask, l0, 1), L1 = l1 + __shfl_xor_sync(kFullMask, l1, 1);
            L0 += __shfl_xor_sync(kFullMask, L0, 2);
            L1 += __shfl_xor_sync(kFullMask, L1, 2);
            const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
            // Output rows straight from the 16x256b layout: one swap with the neighbouring lane
            // gives each lane four consecutive columns, so a store instruction writes 64 (fp32)
            // or 32 (fp16 / bf16) contiguous bytes of each of 8 rows
            const bool odd = (ga & 1) != 0;
            auto write_rows = [&](auto out_tag) {  // one copy of the loops per output type
                using OT = decltype(out_tag);
                OT *outp = static_cast<OT *>(p.out);
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 64) {
                    uint32_t r[32];
                    tmem_ld_16x256b<8>(tO + c0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int trow = rh ? row1 : row0;
                        const float rinv = rh ? inv1 : inv0;
                        const int rtok = it.tok_begin + trow / G;
                        const int64_t obase = ((int64_t)(it.q0 + rtok) * Hq + it.g * G + trow % G) * D + c0;
#pragma unroll
                        for (int g = 0; g < 8; g += 2) {
                            const int e0 = 4 * g + 2 * rh, e1 = 4 * (g + 1) + 2 * rh;  // this row's pair in groups g, g+1
                            const float2 keep = odd ? make_float2(__uint_as_float(r[e1]), __uint_as_float(r[e1 + 1]))
                                                    : make_float2(__uint_as_float(r[e0]), __uint_as_float(r[e0 + 1]));
                            const float2 send = odd ? make_float2(__uint_as_float(r[e0]), __uint_as_float(r[e0 + 1]))
                                                    : make_float2(__uint_as_float(r[e1]), __uint_as_float(r[e1 + 1]));
                            const float2 got = make_float2(__shfl_xor_sync(kFullMask, send.x, 1),
                                                           __shfl_xor_sync(kFullMask, send.y, 1));
                            const int col = odd ? 8 * (g + 1) + 2 * (ga - 1) : 8 * g + 2 * ga;
                            const float4 v = odd ? make_float4(got.x * rinv, got.y * rinv, keep.x * rinv, keep.y * rinv)
                                                 : make_float4(keep.x * rinv, keep.y * rinv, got.x * rinv, got.y * rinv);
                            if (rtok >= it.Lq) continue;
                            if constexpr (std::is_same<OT, float>::value) {
                                *reinterpret_cast<float4 *>(outp + obase + col) = v;
                            } else if constexpr (std::is_same<OT, __half>::value) {
                                __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
                                *reinterpret_cast<uint2 *>(outp + obase + col) =
                                    make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                            } else {
                                __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                                *reinterpret_cast<uint2 *>(outp + obase + col) =
                                    make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                            }
                        }
                    }
                }
            };
            if (p.out_dtype == PA_F32)
                write_rows(float{});
            else if (p.out_dtype == PA_F16)
                write_rows(__half{});
            else
                write_rows(__nv_bfloat16{});
            tc_fence_before();
        }
        if (!ok) *abort_v = 1;
    }
    // ---- teardown: every TMEM access has completed before the columns are released
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

template <class T, int D, int G, bool DR = false>
int launch_typed(const PrefillParams &prm, const CUtensorMap &qm, const CUtensorMap &km,
                 const CUtensorMap &vm, int max_query_len, int num_seqs, cudaStream_t st) {
    constexpr int TT = kBM / G;
    const int smem = PfShape<D>::SMEM;
    static std::atomic<int> smem_ready[kMaxDevices];  // per device: shared-memory limit raised
    PrefillParams p = prm;
    p.q_tiles = (max_query_len + TT - 1) / TT;
    const int64_t items = (int64_t)p.q_tiles * num_seqs * prm.num_kv_heads;
    if (items > INT32_MAX) return PA_ERR_INVALID_ARG;
    p.num_items = (int)items;
    // one persistent CTA per SM (the shared memory allows one)
    const int sms = device_sm_count();
    const int grid = (int)std::min<int64_t>(items, sms > 0 ? sms : 1);
    return launch_pdl_smem(prefill_tc_kernel<T, D, G, DR>, smem_ready, dim3(grid), dim3(kPfThreads), smem, st, qm,
                           km, vm, p) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

template <class T, int D>
int dispatch_g(const PrefillParams &prm, int G, bool decode_rows, const CUtensorMap &qm, const CUtensorMap &km,
               const CUtensorMap &vm, int mq, int S, cudaStream_t st) {
    if (decode_rows)  // built for eight query heads per kv head, the grouping that routes here
        return G == 8 ? launch_typed<T, D, 8, true>(prm, qm, km, vm, mq, S, st) : PA_ERR_UNSUPPORTED;
    switch (G) {
        case 1: return launch_typed<T, D, 1>(prm, qm, km, vm, mq, S, st);
        case 2: return launch_typed<T, D, 2>(prm, qm, km, vm, mq, S, st);
        case 4: return launch_typed<T, D, 4>(prm, qm, km, vm, mq, S, st);
        case 8: return launch_typed<T, D, 8>(prm, qm, km, vm, mq, S, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

template <class T>
int dispatch_d(const PrefillParams &prm, int D, int G, bool dr, const CUtensorMap &qm, const CUtensorMap &km,
               const CUtensorMap &vm, int mq, int S, cudaStream_t st) {
    switch (D) {
        case 64: return dispatch_g<T, 64>(prm, G, dr, qm, km, vm, mq, S, st);
        case 128: return dispatch_g<T, 128>(prm, G, dr, qm, km, vm, mq, S, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_prefill(const PrefillArgs &a) {
    if (a.num_seqs == 0 || a.num_tokens == 0 || a.max_query_len == 0) return PA_OK;
    PrefillParams prm{};
    prm.out = a.out;
    prm.out_dtype = a.out_dtype;
    prm.query_start_loc = a.query_start_loc;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.max_blocks_per_seq = a.max_blocks_per_seq;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.block_size = a.block_size;
    prm.num_blocks = a.num_blocks;
    prm.max_context_len = a.max_context_len;
    prm.num_tokens = a.num_tokens;
    prm.num_seqs = a.num_seqs;
    prm.qk_scale_log2 = a.scale * kLog2e;
    prm.status = a.status;
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t pool_rows = (int64_t)a.num_blocks * a.block_size;
    if (pool_rows <= 0 || pool_rows > INT32_MAX) return PA_ERR_INVALID_ARG;
    // Q boxes are 64 elements (128 bytes, the swizzle span) wide along D and cover the G
    // heads of one kv head for 128/G tokens; a K/V box is one whole block of one kv head,
    // all of D in 64-wide slices (one copy per block).
    CUtensorMap qm, km, vm;
    if (make_tensor_map_3d(&qm, a.query, a.kv_dtype, a.head_dim, a.num_heads, a.num_tokens, 64, G,
                           kBM / G, true) != PA_OK ||
        make_kv_block_map(&km, a.key_cache, a.kv_dtype, a.head_dim, a.num_kv_heads, pool_rows, a.block_size) !=
            PA_OK ||
        make_kv_block_map(&vm, a.value_cache, a.kv_dtype, a.head_dim, a.num_kv_heads, pool_rows, a.block_size) !=
            PA_OK)
        return PA_ERR_CUDA;
    switch (a.kv_dtype) {
        case PA_F16:
            return dispatch_d<F16>(prm, a.head_dim, G, a.decode_rows != 0, qm, km, vm, a.max_query_len, a.num_seqs,
                                   a.stream);
        case PA_BF16:
            return dispatch_d<BF16>(prm, a.head_dim, G, a.decode_rows != 0, qm, km, vm, a.max_query_len, a.num_seqs,
                                    a.stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace pa
