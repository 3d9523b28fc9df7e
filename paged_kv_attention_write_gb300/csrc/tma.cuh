// tma.cuh -- mbarrier and TMA (cp.async.bulk.tensor) helpers for sm_103a.
//
// Every wait is bounded: a wait that has not completed after kWaitLimitNs of
// wall time (%globaltimer) reports PA_DEVERR_TIMEOUT and returns false, so a
// protocol error can never hang the GPU.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace pa {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// Make the barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Add `bytes` to the transaction count of the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false (and a status bit) on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            report(status, PA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 5-D tiled TMA load into shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, int c4, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load into shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// Named barrier over `threads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- host side
// Tensor map over a KV pool viewed as [rows = NB*bs][Hkv][D] (D innermost), box
// {D, box_heads, box_rows}.  Returns PA_OK or PA_ERR_CUDA.
int make_kv_tensor_map(CUtensorMap *map, const void *base, pa_dtype dtype, int head_dim,
                       int num_kv_heads, int64_t rows, int box_heads, int box_rows);

// 5-D tensor map over a KV pool [rows][Hkv][D] (16-bit elements, D a multiple of 64, rows
// and the block size multiples of 8) whose box is one block of one kv head: dimensions
// (column in a 64-wide slice of D, row in a group of 8, slice, group of 8 rows, kv head),
// box {64, 8, D/64, block_size/8, 1}, 128-byte swizzle.  In shared memory the box is
// [group][slice][8 rows][128 B]: every 8-row slab of a slice is one swizzle atom, so the
// block's rows form K-major (and MN-major) operands whose 8-row groups are 1024 * D/64
// bytes apart.  One copy per block instead of one per slice.
int make_kv_block_map(CUtensorMap *map, const void *base, pa_dtype dtype, int head_dim, int num_kv_heads,
                      int64_t rows, int block_size);

// General 3-D tensor map [dim2][dim1][dim0] (dim0 innermost, dense) with box
// {box0, box1, box2}; 128-byte swizzle when asked (box0 * element size must then
// be at most 128 bytes).
int make_tensor_map_3d(CUtensorMap *map, const void *base, pa_dtype dtype, int dim0, int dim1,
                       int64_t dim2, int box0, int box1, int box2, bool swizzle128);

// Streaming multiprocessors of the current device (0 if none can be queried).
int device_sm_count();

}  // namespace pa
