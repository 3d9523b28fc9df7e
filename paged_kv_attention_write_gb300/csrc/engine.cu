// engine.cu -- one serving step's device work through the library's public calls
// (include/pa_engine.h): the upload of a packed step and the step's block copies, cache
// write and attention, so that a step loop crosses into the library twice per step.
#include "common.cuh"
#include "pa_engine.h"

extern "C" int pa_engine_upload(void *dev_batch, const void *host_batch, const pa_sched_offsets *offsets,
                                pa_stream_t stream) {
    if (!dev_batch || !host_batch || !offsets || offsets->dev_bytes < 0) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dev_batch) & 15) != 0) return PA_ERR_INVALID_ARG;
    if (offsets->dev_bytes == 0) return PA_OK;
    return cudaMemcpyAsync(dev_batch, host_batch, (size_t)offsets->dev_bytes, cudaMemcpyHostToDevice,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

extern "C" int pa_engine_attend(const pa_engine_cache *c, const pa_sched_batch *b, const pa_sched_offsets *o,
                                const void *dev_batch, const void *q, const void *k, const void *v, void *out,
                                pa_dtype out_dtype, void *workspace, size_t workspace_bytes, int32_t *status,
                                pa_stream_t stream) {
    if (!c || !b || !o || !dev_batch) return PA_ERR_INVALID_ARG;
    if (b->kind == PA_SCHED_IDLE || b->num_seqs == 0) return PA_OK;
    const char *base = static_cast<const char *>(dev_batch);
    const auto *qsl = reinterpret_cast<const int32_t *>(base + o->query_start_loc);
    const auto *cl = reinterpret_cast<const int32_t *>(base + o->context_lens);
    const auto *bt = reinterpret_cast<const int32_t *>(base + o->block_tables);
    const auto *slots = reinterpret_cast<const int64_t *>(base + o->slot_mapping);
    const auto *pairs = reinterpret_cast<const int64_t *>(base + o->copy_pairs);
    int rc = PA_OK;
    if (b->num_copy_pairs > 0)
        rc = pa_copy_blocks(c->key_cache, c->value_cache, pairs, b->num_copy_pairs, c->num_kv_heads, c->head_dim,
                            c->block_size, c->num_blocks, c->kv_dtype, status, stream);
    if (rc != PA_OK) return rc;
    if (b->kind == PA_SCHED_DECODE && b->num_tokens == b->num_seqs)  // one new token per sequence, at its end
        return pa_decode_write(out, out_dtype, q, k, v, slots, c->key_cache, c->value_cache, bt, b->table_width, cl,
                               b->max_context_len, b->num_seqs, c->num_heads, c->num_kv_heads, c->head_dim,
                               c->block_size, c->num_blocks, c->scale, c->kv_dtype, workspace, workspace_bytes,
                               status, stream);
    rc = pa_reshape_and_cache(k, v, c->key_cache, c->value_cache, slots, b->num_tokens, c->num_kv_heads,
                              c->head_dim, c->block_size, c->num_blocks, c->kv_dtype, status, stream);
    if (rc != PA_OK) return rc;
    if (b->kind == PA_SCHED_DECODE)
        return pa_decode(out, out_dtype, q, c->key_cache, c->value_cache, bt, b->table_width, cl,
                         b->max_context_len, b->num_seqs, c->num_heads, c->num_kv_heads, c->head_dim,
                         c->block_size, c->num_blocks, c->scale, c->kv_dtype, workspace, workspace_bytes, status,
                         stream);
    return pa_prefill_chunk(out, out_dtype, q, qsl, b->num_tokens, b->max_query_len, c->key_cache, c->value_cache,
                            bt, b->table_width, cl, b->max_context_len, b->num_seqs, c->num_heads, c->num_kv_heads,
                            c->head_dim, c->block_size, c->num_blocks, c->scale, c->kv_dtype, status, stream);
}
