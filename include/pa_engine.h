/* pa_engine.h -- one serving step's device work, for a step loop over the scheduler
 * (pa_scheduler.h).
 *
 * A step loop plans a step into one host buffer (pa_sched_step_packed), sends the part the
 * device reads over in one copy (pa_engine_upload), lets the model compute the step's
 * queries, keys and values, and then runs the step's paged-attention work with one call
 * (pa_engine_attend): the scheduler's copy-on-write block copies, the fresh K/V written to
 * their cache slots, and decode or chunked-prefill attention -- the all-decode /
 * all-prefill steps of the Pure-Rust engines page's scheduling section, on the paged pool of
 * the TensorSharp "Mistral 3" page, section 11.  Every call only enqueues work on `stream`
 * and returns a PA_* code; nothing is allocated and nothing synchronises.
 */
#ifndef PA_ENGINE_H
#define PA_ENGINE_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"
#include "pa_scheduler.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The paged KV pool of one attention layer (device memory, caller-owned). */
typedef struct {
    void *key_cache, *value_cache; /* [num_blocks][block_size][num_kv_heads][head_dim], kv_dtype */
    int num_blocks, block_size, num_heads, num_kv_heads, head_dim;
    pa_dtype kv_dtype;
    float scale; /* softmax scale of q.k */
} pa_engine_cache;

/*
 * pa_engine_upload -- copy bytes [0, offsets->dev_bytes) of a packed step (host_batch, as
 * pa_sched_step_packed wrote it; pinned memory makes the copy asynchronous) to dev_batch
 * (device, 16-byte aligned, at least dev_bytes), asynchronously on stream.  The host
 * buffer must stay unchanged until the copy has run.
 */
int pa_engine_upload(void *dev_batch, const void *host_batch, const pa_sched_offsets *offsets,
                     pa_stream_t stream);

/*
 * pa_engine_attend -- the paged-attention work of one planned step, on stream, in order:
 * pa_copy_blocks over the step's copy pairs (when it has any), then for a decode step
 * pa_decode_write (its one new token per sequence written through the slot mapping and
 * attended, with `workspace` as for pa_decode), for a prefill step pa_reshape_and_cache of k
 * and v through the slot mapping and pa_prefill_chunk of q into out.
 *
 *   batch, offsets  the step as pa_sched_step_packed described it
 *   dev_batch       the uploaded device copy of the step (pa_engine_upload)
 *   q               [num_tokens][num_heads][head_dim], kv_dtype (device)
 *   k, v            [num_tokens][num_kv_heads][head_dim], kv_dtype (device)
 *   out             [num_tokens][num_heads][head_dim], out_dtype (device, written)
 *
 * Returns the first failing call's code (later calls are not made); an idle step is a
 * no-op.  Errors and the device status word behave as for the four calls.
 */
int pa_engine_attend(const pa_engine_cache *cache, const pa_sched_batch *batch,
                     const pa_sched_offsets *offsets, const void *dev_batch, const void *q,
                     const void *k, const void *v, void *out, pa_dtype out_dtype, void *workspace,
                     size_t workspace_bytes, int32_t *status, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_ENGINE_H */
