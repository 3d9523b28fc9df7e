// decode_noalloc.cu -- pa_decode without a caller-supplied workspace.
//
// Some callers cannot allocate device memory when they need to run decode:
// plugin hosts and serving runtimes that own every byte of device memory and
// hand kernels only their tensors, code that must not call cudaMalloc on the
// hot path because it may synchronise the device, and bindings from languages
// that have no device allocator at all.  For them this file keeps the decode
// scratch (the split-K partials and the context scan) in one fixed array that
// lives in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  In host
// code its name is only a stand-in for the device variable, so every call looks
// up its device address with cudaGetSymbolAddress in the current context, and
// that address is what the kernels receive.
#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB, see PA_DECODE_NOALLOC_SCRATCH_BYTES
static_assert(kNoAllocScratchBytes == PA_DECODE_NOALLOC_SCRATCH_BYTES, "header and library agree");

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context.  The address belongs to
// the context's copy of the library's device code, not to the device ordinal: a value
// kept from an earlier call would be stale after cudaDeviceReset, or when the caller
// switches between several contexts on one device, so it is looked up on every call.
// The first lookup in a context loads the library's device code there; later ones are a
// host-side table read.
int scratch_for_current_context(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    *out = p;
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(void *out, pa_dtype out_dtype, const void *query,
                                 const void *key_cache, const void *value_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int max_context_len, int num_seqs,
                                 int num_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, pa_dtype kv_dtype, int32_t *status,
                                 pa_stream_t stream) {
    // Reject a problem whose scratch would not fit before touching the device.  A
    // size of 0 means the arguments are invalid (or there is nothing to do):
    // pa_decode then returns the matching code without launching anything.
    const size_t need = num_seqs > 0 ? pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                                head_dim, max_context_len)
                                     : 0;
    if (need > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_for_current_context(&scratch);
        if (rc != PA_OK) return rc;
    }
    // Every scratch entry the kernels read is written earlier in the same call, so
    // nothing has to be cleared between calls.
    return pa_decode(out, out_dtype, query, key_cache, value_cache, block_tables,
                     max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, kv_dtype, scratch,
                     kNoAllocScratchBytes, status, stream);
}
