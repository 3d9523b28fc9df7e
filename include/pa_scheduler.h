/* pa_scheduler.h -- host step scheduler over the KV-cache manager (pa_kv_manager.h).
 *
 * The scheduler turns a queue of requests (prompt tokens, number of tokens to generate) into
 * batches for the paged-attention kernels, one step at a time, the way the Pure-Rust engines
 * page describes mistral.rs's paged scheduler (scheduling section): every step is either a
 * prefill batch or a decode batch, never both; with prompts waiting, at most 8 decode steps
 * run in a row (DEFAULT_MAX_DECODE_STEPS_BEFORE_PREFILL); a prefill batch holds at most
 * 4096 tokens (DEFAULT_MAX_NUM_BATCHED_TOKENS) and a long prompt is cut into chunks of at
 * most 512 tokens (DEFAULT_MAX_PREFILL_CHUNK_TOKENS).  The three limits are arguments.
 *
 * Policy (exact; the reference scheduler restates it):
 *  - Step decision: with prompt work pending (a prompt being prefilled, or a request
 *    waiting) and either nothing running or max_decode_steps decode steps in a row, try a
 *    prefill batch; if it comes out empty (no block to spare), or without prompt work,
 *    decode every running request; with nothing running either, the step is idle.
 *  - Prefill batch: first the prompts already being prefilled (admission order), each with
 *    its next chunk of at most chunk_tokens tokens while the token budget lasts and blocks
 *    can be allocated; then waiting requests in arrival order, admitted only if the blocks
 *    for their first chunk fit the free blocks (those not taken by their own prefix-cache
 *    hits); a request's prefix-cache hits are not computed again.
 *  - A request's last prompt chunk yields its first generated token; a decode step computes
 *    the newest token of every running request (position = its length - 1) and yields the
 *    next.  A request that has generated max_new_tokens tokens is freed at once.
 *  - Preemption: when a decode step cannot get a block for a request, the most recently
 *    admitted running request is preempted (blocks freed, its tokens so far queued at the
 *    head of the waiting queue as its new prompt, to be recomputed) until it can; when the
 *    next chunk of a prompt being prefilled cannot get its blocks, the most recently
 *    admitted prompt being prefilled is preempted the same way until the chunk fits (or that
 *    prompt itself was preempted).  A chunk of chunk_tokens tokens must fit the pool.
 *
 * Host memory only; calls on one scheduler must not run concurrently.  Errors:
 * PA_ERR_INVALID_ARG, PA_ERR_WORKSPACE (an output array too small: checked before any state
 * changes).
 */
#ifndef PA_SCHEDULER_H
#define PA_SCHEDULER_H

#include <stdint.h>

#include "pa_kv_manager.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_sched pa_sched;

enum { PA_SCHED_IDLE = 0, PA_SCHED_PREFILL = 1, PA_SCHED_DECODE = 2 };

/* One step's batch, described by pa_sched_step. */
typedef struct {
    int kind;            /* PA_SCHED_IDLE, PA_SCHED_PREFILL or PA_SCHED_DECODE */
    int num_seqs;        /* sequences in the batch */
    int num_tokens;      /* query tokens (K/V to write) in the batch */
    int max_query_len;   /* longest chunk (1 for decode) */
    int max_context_len; /* longest context after the step */
    int table_width;     /* block-table row stride written (blocks of the longest sequence) */
    int num_copy_pairs;  /* copy-on-write pairs to apply with pa_copy_blocks first */
} pa_sched_batch;

int pa_sched_create(int num_blocks, int block_size, int token_budget, int chunk_tokens,
                    int max_decode_steps, int enable_prefix_cache, pa_sched **out);
void pa_sched_destroy(pa_sched *s);

/* Queue a request (arrival order).  prompt_len >= 1, max_new_tokens >= 1; a request whose
 * prompt and generated tokens need more blocks than the pool holds is refused
 * (PA_ERR_INVALID_ARG). */
int pa_sched_add_request(pa_sched *s, int64_t req_id, const int32_t *prompt, int prompt_len,
                         int max_new_tokens);

/* Plan the next step.  Writes, for the batch's sequences in order: req_ids[num_seqs],
 * query_start_loc[num_seqs + 1], context_lens[num_seqs], block_tables[num_seqs *
 * table_width] (row-major, unused entries 0); for its query tokens in order: token_ids,
 * positions and slot_mapping[num_tokens]; copy_pairs[2 * num_copy_pairs].  Capacities:
 * max_seqs sequences, max_tokens tokens, table_capacity entries per row, max_pairs pairs;
 * pa_sched_capacity gives sufficient values.  The step's state changes take effect now;
 * pa_sched_complete must follow before the next pa_sched_step. */
int pa_sched_step(pa_sched *s, pa_sched_batch *batch, int64_t *req_ids, int32_t *query_start_loc,
                  int32_t *context_lens, int32_t *block_tables, int table_capacity,
                  int32_t *token_ids, int32_t *positions, int64_t *slot_mapping, int64_t *copy_pairs,
                  int max_seqs, int max_tokens, int max_pairs);

/* Byte offsets of one step's arrays inside the caller's buffer (pa_sched_step_packed).  The
 * arrays the kernels and the model read come first, in one span of dev_bytes bytes (one
 * host-to-device copy): query_start_loc, context_lens, block_tables, slot_mapping,
 * copy_pairs, token_ids, positions; req_ids (host only) follows.  Every array starts on a
 * 16-byte boundary of the buffer and has the element type and length pa_sched_step gives
 * it (block-table rows table_width entries apart). */
typedef struct {
    int64_t query_start_loc, context_lens, block_tables, slot_mapping, copy_pairs, token_ids, positions;
    int64_t dev_bytes;
    int64_t req_ids;
    int64_t total_bytes;
} pa_sched_offsets;

/* Buffer bytes pa_sched_step_packed may need for any step with the requests queued so far
 * (grows when requests are added). */
int64_t pa_sched_packed_bytes(const pa_sched *s);

/* pa_sched_step with every array of the step written into one caller buffer (host memory,
 * 16-byte aligned, for instance pinned so that its device span goes over in one asynchronous
 * copy), laid out for the batch's own sizes as *offsets states.  PA_ERR_WORKSPACE when
 * buf_bytes < pa_sched_packed_bytes(s) (nothing changes); pa_sched_complete follows as for
 * pa_sched_step. */
int pa_sched_step_packed(pa_sched *s, pa_sched_batch *batch, void *buf, int64_t buf_bytes,
                         pa_sched_offsets *offsets);

/* Finish the planned step with one sampled token per batch sequence (a prefill chunk that is
 * not its prompt's last ignores its entry).  Writes the requests that finished (and were
 * freed) to finished (capacity max_finished, count *num_finished). */
int pa_sched_complete(pa_sched *s, const int32_t *sampled, int num_sampled, int64_t *finished,
                      int max_finished, int *num_finished);

/* Output capacities sufficient for every step with the requests queued so far: out[0]
 * sequences, out[1] tokens, out[2] block-table entries per row, out[3] copy pairs. */
int pa_sched_capacity(const pa_sched *s, int out[4]);

/* Counters: out[0] prefill steps, out[1] decode steps, out[2] prompt tokens computed,
 * out[3] tokens generated, out[4] requests finished, out[5] preemptions, out[6] requests
 * still queued or running. */
int pa_sched_stats(const pa_sched *s, int64_t out[7]);

/* The manager the scheduler owns (for queries such as pa_kvm_stats; do not modify). */
pa_kvm *pa_sched_manager(pa_sched *s);

#ifdef __cplusplus
}
#endif

#endif /* PA_SCHEDULER_H */
