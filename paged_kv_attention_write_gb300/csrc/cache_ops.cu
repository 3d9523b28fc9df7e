// cache_ops.cu -- the two data-movement operations on the paged KV pool.
//
// reshape_and_cache: fresh K/V rows scattered to slot = blockId * blockSize +
//   offset (TensorSharp "Mistral 3" page, section 11, K/V scatter via
//   slotMapping).  In the [NB][bs][Hkv][D] pool a token's Hkv*D elements are
//   one contiguous row, so each token is one contiguous 16-byte-vector copy.
// copy_blocks: whole-block K and V copies for prefix-cache reuse (mistral.rs
//   page, block-hash prefix cache).  A block is bs*Hkv*D contiguous elements.
//
// Both are HBM-bound bit copies: 16-byte vector loads and stores, coalesced
// along the row; no arithmetic on the elements.  A third kernel writes the cache with
// the key rotated (RoPE) on the way in.
#include "tma.cuh"  // device_sm_count

namespace pa {
namespace {

constexpr int kCopyThreads = 128;
constexpr int kWriteThreads = 256;
constexpr int kWriteUnroll = 4;  // 16-byte K and V vectors per thread in flight at once

// The fresh rows seen as one flat list of 16-byte vectors (token t owns vectors
// t*vecs_per_row .. +vecs_per_row-1).  Each thread takes kWriteUnroll vectors a grid stride
// apart and issues every load -- K, V and the slot of its token -- before any store, so a
// CTA keeps 32 KB in flight and the kernel costs one round trip for the loads and one for
// the stores (the loads do not depend on the slot; only the stores do).
__global__ void __launch_bounds__(kWriteThreads)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                         const int64_t *__restrict__ slot_mapping, int vecs_per_row, int num_tokens,
                         int64_t num_slots, int32_t *status) {
    pdl_wait_previous();
    pdl_launch_dependents();
    const int64_t total = (int64_t)num_tokens * vecs_per_row;
    const int64_t stride = (int64_t)gridDim.x * kWriteThreads;
    for (int64_t base = (int64_t)blockIdx.x * kWriteThreads + threadIdx.x; base < total;
         base += stride * kWriteUnroll) {
        uint4 k[kWriteUnroll], v[kWriteUnroll];
        int64_t slot[kWriteUnroll];
        int col[kWriteUnroll];
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int64_t i = base + u * stride;
            if (i < total) {
                const int64_t t = i / vecs_per_row;
                col[u] = (int)(i - t * vecs_per_row);
                slot[u] = slot_mapping[t];
                k[u] = ldg_stream(key + i);
                v[u] = ldg_stream(value + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int64_t i = base + u * stride;
            if (i >= total || slot[u] < 0) continue;  // past the end, or a padding token
            if (slot[u] >= num_slots) {
                if (col[u] == 0) report(status, PA_DEVERR_SLOT);
                continue;
            }
            key_cache[slot[u] * vecs_per_row + col[u]] = k[u];
            value_cache[slot[u] * vecs_per_row + col[u]] = v[u];
        }
    }
}

// grid = (num_pairs, chunks); each CTA copies one chunk of one block, K and V.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                   const int64_t *__restrict__ block_mapping, int64_t vecs_per_block,
                   int64_t vecs_per_chunk, int num_blocks, int32_t *status) {
    pdl_wait_previous();
    pdl_launch_dependents();
    const int p = blockIdx.x;
    const int64_t src = block_mapping[2 * p];
    const int64_t dst = block_mapping[2 * p + 1];
    if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) report(status, PA_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t begin = (int64_t)blockIdx.y * vecs_per_chunk;
    const int64_t end = min(vecs_per_block, begin + vecs_per_chunk);
    const uint4 *ks = key_cache + src * vecs_per_block;
    const uint4 *vs = value_cache + src * vecs_per_block;
    uint4 *kd = key_cache + dst * vecs_per_block;
    uint4 *vd = value_cache + dst * vecs_per_block;
    for (int64_t i = begin + threadIdx.x; i < end; i += kCopyThreads) {
        uint4 k = ks[i];
        uint4 v = vs[i];
        kd[i] = k;
        vd[i] = v;
    }
}

// reshape_and_cache with the key rotated on the way in (RoPE, GPT-J pairing: TensorSharp
// "Mistral 3" page, section 4.2).  One CTA per token: the token's cos/sin of every pair
// are computed once into shared memory and shared by its kv heads; each thread
// then rotates 16-byte vectors of the key row in fp32 and writes them, and copies the
// value row.  T is the element type of the cache (F32, F16, BF16 tags).
constexpr int kRopeMaxPairs = 64;  // rope_dim <= head_dim <= 128

template <class T>
__device__ __forceinline__ uint4 narrow16(const float *f);
template <>
__device__ __forceinline__ uint4 narrow16<F32>(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
template <>
__device__ __forceinline__ uint4 narrow16<BF16>(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 narrow16<F16>(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <class T>
__global__ void __launch_bounds__(kCopyThreads)
reshape_and_cache_rope_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                              uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                              const int64_t *__restrict__ slot_mapping, const int32_t *__restrict__ positions,
                              const float *__restrict__ freqs, int rope_dim, int head_dim, int vecs_per_row,
                              int64_t num_slots, int32_t *status) {
    constexpr int EPV = T::kPerVec;  // elements per 16-byte vector
    __shared__ float2 cs[kRopeMaxPairs];                          // (cos, sin) of each pair
    pdl_wait_previous();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    const uint4 *ks = key + (int64_t)t * vecs_per_row;
    const uint4 *vs = value + (int64_t)t * vecs_per_row;
    // the first vectors of the rows, the slot and the position are loaded together (the
    // row loads depend on neither)
    const int64_t slot = slot_mapping[t];
    const int pos = positions[t];
    uint4 k_first = make_uint4(0, 0, 0, 0), v_first = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < vecs_per_row) {
        k_first = ldg_stream(ks + threadIdx.x);
        v_first = ldg_stream(vs + threadIdx.x);
    }
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (threadIdx.x == 0) report(status, PA_DEVERR_SLOT);
        return;
    }
    for (int i = threadIdx.x; i < rope_dim / 2; i += kCopyThreads) cs[i] = rope_cos_sin(pos, freqs[i]);
    __syncthreads();
    uint4 *kd = key_cache + slot * vecs_per_row;
    uint4 *vd = value_cache + slot * vecs_per_row;
    for (int i = threadIdx.x; i < vecs_per_row; i += kCopyThreads) {
        const int d0 = (i * EPV) % head_dim;  // first element of the vector within its head
        uint4 k = i < kCopyThreads ? k_first : ks[i];
        const uint4 vv = i < kCopyThreads ? v_first : vs[i];
        if (d0 < rope_dim) {
            float f[EPV];
            widen(T{}, k, f);
#pragma unroll
            for (int e = 0; e < EPV; e += 2) {
                const int pair = (d0 + e) / 2;
                if (2 * pair < rope_dim) {
                    const float2 r = cs[pair];
                    const float x = f[e], y = f[e + 1];
                    f[e] = x * r.x - y * r.y;
                    f[e + 1] = x * r.y + y * r.x;
                }
            }
            k = narrow16<T>(f);
        }
        kd[i] = k;
        vd[i] = vv;
    }
}

}  // namespace

int launch_reshape_and_cache_rope(const void *key, const void *value, void *key_cache, void *value_cache,
                                  const int64_t *slot_mapping, const int32_t *positions, int num_tokens,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  pa_dtype kv_dtype, const float *freqs, int rope_dim, int32_t *status,
                                  cudaStream_t stream) {
    if (num_tokens == 0) return PA_OK;
    const int eb = kv_dtype == PA_F32 ? 4 : 2;
    const int vecs = num_kv_heads * head_dim * eb / 16;
    const int64_t slots = (int64_t)num_blocks * block_size;
    const uint4 *k = static_cast<const uint4 *>(key), *v = static_cast<const uint4 *>(value);
    uint4 *kc = static_cast<uint4 *>(key_cache), *vc = static_cast<uint4 *>(value_cache);
    cudaError_t e;
    switch (kv_dtype) {
        case PA_F32:
            e = launch_pdl(reshape_and_cache_rope_kernel<F32>, dim3(num_tokens), dim3(kCopyThreads), 0, stream, k,
                           v, kc, vc, slot_mapping, positions, freqs, rope_dim, head_dim, vecs, slots, status);
            break;
        case PA_F16:
            e = launch_pdl(reshape_and_cache_rope_kernel<F16>, dim3(num_tokens), dim3(kCopyThreads), 0, stream, k,
                           v, kc, vc, slot_mapping, positions, freqs, rope_dim, head_dim, vecs, slots, status);
            break;
        case PA_BF16:
            e = launch_pdl(reshape_and_cache_rope_kernel<BF16>, dim3(num_tokens), dim3(kCopyThreads), 0, stream, k,
                           v, kc, vc, slot_mapping, positions, freqs, rope_dim, head_dim, vecs, slots, status);
            break;
        default:
            return PA_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_reshape_and_cache(const void *key, const void *value, void *key_cache,
                             void *value_cache, const int64_t *slot_mapping, int num_tokens,
                             int row_bytes, int block_size, int num_blocks, int32_t *status,
                             cudaStream_t stream) {
    if (num_tokens == 0) return PA_OK;
    const int vecs = row_bytes / 16;
    const int64_t total = (int64_t)num_tokens * vecs;
    const int64_t per_cta = (int64_t)kWriteThreads * kWriteUnroll;
    const int64_t ctas = (total + per_cta - 1) / per_cta;
    const int sms = device_sm_count();
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;  // 8 CTAs per SM are resident at once
    const cudaError_t e = launch_pdl(
        reshape_and_cache_kernel, dim3((unsigned)(ctas < cap ? ctas : cap)), dim3(kWriteThreads), 0, stream,
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), slot_mapping,
        vecs, num_tokens, (int64_t)num_blocks * block_size, status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping,
                       int num_pairs, int64_t block_bytes, int num_blocks, int32_t *status,
                       cudaStream_t stream) {
    if (num_pairs == 0) return PA_OK;
    const int64_t vecs = block_bytes / 16;
    const int64_t per_chunk = kCopyThreads * 8;  // 16 KB of K and 16 KB of V per CTA
    const int64_t chunks = (vecs + per_chunk - 1) / per_chunk;
    dim3 grid(num_pairs, (unsigned)chunks);
    const cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, stream,
                                     static_cast<uint4 *>(key_cache),
                                     static_cast<uint4 *>(value_cache), block_mapping, vecs,
                                     per_chunk, num_blocks, status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
