// common.cuh -- device helpers shared by the paged-attention kernels.
//
// Element formats, 16-byte vector loads, the device-side status word and the
// internal launcher declarations.  Nothing here is part of the public ABI
// (include/pa.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/pa.h"

namespace pa {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- element formats
// Tag types: a 16-byte vector holds kPerVec elements of the format.
struct F32 {
    using storage = float;
    static constexpr int kBytes = 4;
    static constexpr int kPerVec = 4;
};
struct F16 {
    using storage = __half;
    static constexpr int kBytes = 2;
    static constexpr int kPerVec = 8;
};
struct BF16 {
    using storage = __nv_bfloat16;
    static constexpr int kBytes = 2;
    static constexpr int kPerVec = 8;
};

// Widen one 16-byte vector to floats.
__device__ __forceinline__ void widen(F32, const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void widen_pair_bf16(uint32_t u, float &lo, float &hi) {
    // bf16 is the top half of an fp32 word: widening is a shift / mask.
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}
__device__ __forceinline__ void widen(BF16, const uint4 &v, float *f) {
    widen_pair_bf16(v.x, f[0], f[1]);
    widen_pair_bf16(v.y, f[2], f[3]);
    widen_pair_bf16(v.z, f[4], f[5]);
    widen_pair_bf16(v.w, f[6], f[7]);
}
__device__ __forceinline__ void widen_pair_f16(uint32_t u, float &lo, float &hi) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
}
__device__ __forceinline__ void widen(F16, const uint4 &v, float *f) {
    widen_pair_f16(v.x, f[0], f[1]);
    widen_pair_f16(v.y, f[2], f[3]);
    widen_pair_f16(v.z, f[4], f[5]);
    widen_pair_f16(v.w, f[6], f[7]);
}

// Store n (even) floats, rounded to the output format.
__device__ __forceinline__ void store_out(float *p, float a, float b) {
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store_out(__half *p, float a, float b) {
    *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(a, b);
}
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}

// ---------------------------------------------------------------- memory helpers
// Streaming 16-byte load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2^-22, flushes
// subnormal results to zero); the softmax weights need nothing more precise.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (cos, sin) of the RoPE angle pos * f, all in fp32 (fp64 runs at a small fraction of the
// fp32 rate on this part).  pos * f = hi + lo exactly (two-product: pos < 2^24 is exact
// in fp32); the angle is reduced by k = rint(hi / 2 pi) turns with 2 pi split in two
// floats, Cody and Waite's additive reduction: hi - k * C1 is exact (both are multiples of
// 2^-21 below 8 in magnitude), the small terms -k * C2 + lo take one rounding, the sum one
// more.  For 0 <= pos < 2^24 the reduced angle is within 2.3e-7 of pos * f mod 2 pi (one
// fp32 ulp at pi); __sincosf adds under 4e-7 on [-pi, pi].
__device__ __forceinline__ float2 rope_cos_sin(int pos, float f) {
    constexpr float kC1 = 6.28318548202514648f;       // 2 pi rounded to fp32 (0x40c90fdb)
    constexpr float kC2 = -1.74845553146951720e-7f;   // 2 pi - kC1 rounded to fp32 (0xb43bbd2e)
    constexpr float kInvTwoPi = 0.159154943091895336f;
    const float pf = (float)pos;
    const float hi = pf * f;
    const float lo = fmaf(pf, f, -hi);
    const float k = rintf(hi * kInvTwoPi);
    const float r1 = fmaf(-k, kC1, hi);
    const float r2 = fmaf(-k, kC2, lo);
    float s, c;
    __sincosf(r1 + r2, &s, &c);
    return make_float2(c, s);
}

__device__ __forceinline__ void report(int32_t *status, int bit) {
    if (status) atomicOr(status, bit);
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_pdl (below) and calls pdl_wait_previous() before it touches memory that
// an earlier kernel in the stream may write; pdl_launch_dependents() lets the
// next kernel's launch and prologue overlap this one.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_previous() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// Devices a process can address in the per-device tables below.
constexpr int kMaxDevices = 64;

// launch_pdl for a kernel that needs more than 48 KB of dynamic shared memory.  The limit
// is raised (cudaFuncSetAttribute) once per device; `ready` is the kernel's own per-device
// table of flags (static storage, zero at start).  Host threads may race through this:
// the flags are atomic and raising the limit twice is harmless.  If a launch still fails
// after the flag was set (the attribute was lost, for instance after cudaDeviceReset),
// the limit is raised again and the launch retried once.
template <class... KArgs, class... Args>
cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), std::atomic<int> *ready, dim3 grid, dim3 block,
                            size_t smem, cudaStream_t stream, const Args &...args) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<int> *flag = (dev >= 0 && dev < kMaxDevices) ? &ready[dev] : nullptr;
    for (int attempt = 0;; ++attempt) {
        const bool was_set = flag && flag->load(std::memory_order_acquire);
        if (!was_set) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (flag) flag->store(1, std::memory_order_release);
        }
        e = launch_pdl(kernel, grid, block, smem, stream, args...);
        if (e == cudaSuccess || !was_set || attempt > 0) return e;
        flag->store(0, std::memory_order_release);
    }
}

}  // namespace pa

// ---------------------------------------------------------------- internal launchers
// Called by the C-ABI layer after host-side validation.  Each returns a
// PA_* code (PA_ERR_CUDA when the launch itself failed).
namespace pa {

struct DecodeArgs {
    void *out;
    pa_dtype out_dtype;
    const void *query;
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    int max_context_len;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    float scale;
    pa_dtype kv_dtype;
    void *workspace;
    size_t workspace_bytes;
    int32_t *status;
    cudaStream_t stream;
    // query RoPE and position-dependent scale (null freqs: none)
    const float *rope_freqs = nullptr;
    int rope_dim = 0;
    float q_scale_beta = 0.f;
    int q_scale_orig_ctx = 0;
    // the new token of every sequence, written to its slot first (null key: no write)
    const void *new_key = nullptr, *new_value = nullptr;
    const int64_t *slot_mapping = nullptr;
};

struct PrefillArgs {
    void *out;
    pa_dtype out_dtype;
    const void *query;
    const int32_t *query_start_loc;
    int num_tokens, max_query_len;
    const void *key_cache;
    const void *value_cache;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    int max_context_len;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    float scale;
    pa_dtype kv_dtype;
    int32_t *status;
    cudaStream_t stream;
    int decode_rows = 0;  // one query row per sequence (token s), no query_start_loc
};

int launch_reshape_and_cache(const void *key, const void *value, void *key_cache,
                             void *value_cache, const int64_t *slot_mapping, int num_tokens,
                             int row_bytes, int block_size, int num_blocks, int32_t *status,
                             cudaStream_t stream);
int launch_reshape_and_cache_rope(const void *key, const void *value, void *key_cache, void *value_cache,
                                  const int64_t *slot_mapping, const int32_t *positions, int num_tokens,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  pa_dtype kv_dtype, const float *freqs, int rope_dim, int32_t *status,
                                  cudaStream_t stream);
int launch_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping,
                       int num_pairs, int64_t block_bytes, int num_blocks, int32_t *status,
                       cudaStream_t stream);
size_t decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int max_context_len);
int launch_decode(const DecodeArgs &a);
int launch_prefill(const PrefillArgs &a);

}  // namespace pa
