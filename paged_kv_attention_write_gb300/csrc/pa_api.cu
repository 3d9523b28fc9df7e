// pa_api.cu -- the extern "C" boundary declared in include/pa.h.
//
// Every entry point validates its arguments on the host before touching the
// GPU (no CUDA call happens on a rejected call), then hands a plain argument
// record to the kernel launcher of its operation.  Nothing is allocated and
// nothing is synchronised here.
#include <cmath>

#include "common.cuh"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int elem_bytes(pa_dtype d) {
    switch (d) {
        case PA_F32: return 4;
        case PA_F16:
        case PA_BF16: return 2;
    }
    return 0;
}

bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool block_size_ok(int b) { return b == 8 || b == 16 || b == 32; }
bool group_ok(int hq, int hkv) {
    if (hq <= 0 || hkv <= 0 || hq % hkv) return false;
    const int g = hq / hkv;
    const bool kv_ok = hkv <= 8 ? 8 % hkv == 0 : hkv % 8 == 0;
    return kv_ok && (g == 1 || g == 2 || g == 4 || g == 8);
}

// Shared checks of the attention calls' cache / table arguments.
int check_attention(const void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
                    const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                    pa_dtype kv_dtype) {
    if (!elem_bytes(kv_dtype) || !elem_bytes(out_dtype)) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_seqs > 65535 || num_blocks < 0 || max_context_len < 0 ||
        max_blocks_per_seq < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size) || !group_ok(num_heads, num_kv_heads))
        return PA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX ||
        (int64_t)num_blocks * block_size > INT32_MAX)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

const char *pa_status_string(int code) {
    switch (code) {
        case PA_OK: return "PA_OK: success";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: null/misaligned pointer, bad size or dtype";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim, block_size, head grouping or dtype not built";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case PA_ERR_CUDA: return "PA_ERR_CUDA: kernel launch failed";
        case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS: not enough free KV-cache blocks";
    }
    return "unknown pa status code";
}

int pa_reshape_and_cache(const void *key, const void *value, void *key_cache, void *value_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype kv_dtype,
                         int32_t *status, pa_stream_t stream) {
    const int eb = elem_bytes(kv_dtype);
    if (!eb || num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16) || !aligned(slot_mapping, 8) || !aligned(status, 4))
        return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * eb;
    if (row_bytes > INT32_MAX) return PA_ERR_INVALID_ARG;
    return pa::launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                                        num_tokens, (int)row_bytes, block_size, num_blocks,
                                        status, reinterpret_cast<cudaStream_t>(stream));
}

int pa_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_dtype kv_dtype, int32_t *status, pa_stream_t stream) {
    const int eb = elem_bytes(kv_dtype);
    if (!eb || num_pairs < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!key_cache || !value_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(block_mapping, 8) ||
        !aligned(status, 4))
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * eb;
    return pa::launch_copy_blocks(key_cache, value_cache, block_mapping, num_pairs, block_bytes,
                                  num_blocks, status, reinterpret_cast<cudaStream_t>(stream));
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int max_context_len) {
    if (num_seqs <= 0 || num_seqs > 65535 || max_context_len < 0 || !head_dim_ok(head_dim) ||
        !group_ok(num_heads, num_kv_heads))
        return 0;
    return pa::decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len);
}

int pa_decode(void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
              const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
              int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
              pa_dtype kv_dtype, void *workspace, size_t workspace_bytes, int32_t *status,
              pa_stream_t stream) {
    int rc = check_attention(out, out_dtype, query, key_cache, value_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             kv_dtype);
    if (rc != PA_OK || num_seqs == 0) return rc;
    if (!aligned(status, 4)) return PA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
    pa::DecodeArgs a{out,          out_dtype,      query,     key_cache,    value_cache,
                     block_tables, max_blocks_per_seq, context_lens, max_context_len,
                     num_seqs,     num_heads,      num_kv_heads, head_dim,  block_size,
                     num_blocks,   scale,          kv_dtype,  workspace,    workspace_bytes,
                     status,       reinterpret_cast<cudaStream_t>(stream)};
    return pa::launch_decode(a);
}

int pa_decode_write(void *out, pa_dtype out_dtype, const void *query, const void *key, const void *value,
                    const int64_t *slot_mapping, void *key_cache, void *value_cache,
                    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, float scale, pa_dtype kv_dtype, void *workspace,
                    size_t workspace_bytes, int32_t *status, pa_stream_t stream) {
    int rc = check_attention(out, out_dtype, query, key_cache, value_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             kv_dtype);
    if (rc != PA_OK || num_seqs == 0) return rc;
    if (!key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8) || !aligned(status, 4))
        return PA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
    pa::DecodeArgs a{out,          out_dtype,      query,     key_cache,    value_cache,
                     block_tables, max_blocks_per_seq, context_lens, max_context_len,
                     num_seqs,     num_heads,      num_kv_heads, head_dim,  block_size,
                     num_blocks,   scale,          kv_dtype,  workspace,    workspace_bytes,
                     status,       reinterpret_cast<cudaStream_t>(stream)};
    a.new_key = key;
    a.new_value = value;
    a.slot_mapping = slot_mapping;
    return pa::launch_decode(a);
}

// The rotary-embedding arguments shared by the two fused entry points.
static int check_rope(const pa_rope *rope, int head_dim) {
    if (!rope || !rope->freqs || !aligned(rope->freqs, 4)) return PA_ERR_INVALID_ARG;
    if (rope->rope_dim < 2 || rope->rope_dim % 2 != 0 || rope->rope_dim > head_dim) return PA_ERR_INVALID_ARG;
    if (rope->q_scale_orig_ctx < 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int pa_decode_rope(void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
                   const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                   pa_dtype kv_dtype, const pa_rope *rope, void *workspace, size_t workspace_bytes,
                   int32_t *status, pa_stream_t stream) {
    int rc = check_attention(out, out_dtype, query, key_cache, value_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             kv_dtype);
    if (rc != PA_OK) return rc;
    if ((rc = check_rope(rope, head_dim)) != PA_OK) return rc;
    if (num_seqs == 0) return PA_OK;
    if (!aligned(status, 4)) return PA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
    pa::DecodeArgs a{out,          out_dtype,      query,     key_cache,    value_cache,
                     block_tables, max_blocks_per_seq, context_lens, max_context_len,
                     num_seqs,     num_heads,      num_kv_heads, head_dim,  block_size,
                     num_blocks,   scale,          kv_dtype,  workspace,    workspace_bytes,
                     status,       reinterpret_cast<cudaStream_t>(stream)};
    a.rope_freqs = rope->freqs;
    a.rope_dim = rope->rope_dim;
    a.q_scale_beta = rope->q_scale_beta;
    a.q_scale_orig_ctx = rope->q_scale_orig_ctx;
    return pa::launch_decode(a);
}

int pa_reshape_and_cache_rope(const void *key, const void *value, void *key_cache, void *value_cache,
                              const int64_t *slot_mapping, const int32_t *positions, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              pa_dtype kv_dtype, const pa_rope *rope, int32_t *status,
                              pa_stream_t stream) {
    const int eb = elem_bytes(kv_dtype);
    if (!eb || num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    int rc = check_rope(rope, head_dim);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping || !positions) return PA_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(slot_mapping, 8) || !aligned(positions, 4) || !aligned(status, 4))
        return PA_ERR_INVALID_ARG;
    return pa::launch_reshape_and_cache_rope(key, value, key_cache, value_cache, slot_mapping, positions,
                                             num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
                                             kv_dtype, rope->freqs, rope->rope_dim, status,
                                             reinterpret_cast<cudaStream_t>(stream));
}

int pa_prefill_chunk(void *out, pa_dtype out_dtype, const void *query,
                     const int32_t *query_start_loc, int num_tokens, int max_query_len,
                     const void *key_cache, const void *value_cache, const int32_t *block_tables,
                     int max_blocks_per_seq, const int32_t *context_lens, int max_context_len,
                     int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, float scale, pa_dtype kv_dtype, int32_t *status,
                     pa_stream_t stream) {
    int rc = check_attention(out, out_dtype, query, key_cache, value_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             kv_dtype);
    if (rc != PA_OK) return rc;
    if (kv_dtype == PA_F32) return PA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || max_query_len < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_tokens == 0) return PA_OK;
    if (!query_start_loc || !aligned(query_start_loc, 4) || !aligned(status, 4))
        return PA_ERR_INVALID_ARG;
    pa::PrefillArgs a{out,          out_dtype,  query,        query_start_loc,   num_tokens,
                      max_query_len, key_cache, value_cache,  block_tables,      max_blocks_per_seq,
                      context_lens, max_context_len, num_seqs, num_heads,        num_kv_heads,
                      head_dim,     block_size, num_blocks,   scale,             kv_dtype,
                      status,       reinterpret_cast<cudaStream_t>(stream)};
    return pa::launch_prefill(a);
}

}  // extern "C"
