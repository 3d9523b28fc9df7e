/* pa_kv_manager.h -- host-side block pool and KV-cache manager for the paged KV cache.
 *
 * The manager hands out the physical blocks of a pool of num_blocks blocks of block_size
 * tokens, keeps each request's block table, and shares full blocks between requests whose
 * token prefixes are equal (prefix caching).  Its operations are the ones the Pure-Rust
 * engines page describes for mistral.rs's port of vLLM v1's KV-cache manager (section on
 * paged attention and block management): find the longest prefix-cache hit of a request,
 * allocate blocks for new tokens, cache newly full blocks, free a request's blocks; the
 * block pool is flat with an LRU free list; blocks are found by content hashes chained
 * along the prefix (prefix-cache section: full blocks are registered and a lookup walks the
 * hash chain to the longest hit).  The TensorSharp "Mistral 3" page, section 11, describes
 * the same block-hash sharing and the slot formula blockId * blockSize + offset.
 *
 * Policy (exact; the oracle restates it):
 *  - Free queue: initially blocks 0..num_blocks-1 in id order.  An allocation takes blocks
 *    from the head.  Freeing a request returns its blocks to the tail, last block first
 *    (the request's tail blocks are the first to be reused).
 *  - A full block (block_size tokens) becomes cached when pa_kvm_cache_blocks registers it,
 *    unless another block already holds the same prefix.  A cached block keeps its content
 *    when its last user frees it; it leaves the cache only when the free queue hands it out
 *    again.  A lookup that hits a cached block in the free queue takes it out of the queue.
 *  - Prefix identity: block i of a token sequence is identified by all tokens up to the end
 *    of block i.  The library keys blocks by a 64-bit FNV-1a hash chained over the parent
 *    key and the block's tokens, and verifies the stored tokens and parent key on a hit.
 *  - A lookup covers at most num_tokens - 1 tokens: the last token is always computed.
 *  - pa_kvm_fork shares all of the parent's blocks with the child.  When a request appends
 *    tokens into a partial last block that another request also holds, that block is first
 *    replaced by a copy (copy-on-write); the (src, dst) pair is returned so that the caller
 *    copies the block's K/V with pa_copy_blocks before writing new tokens.
 *
 * Everything is host memory owned by the manager; calls on one manager must not run
 * concurrently.  Errors: PA_ERR_INVALID_ARG (bad argument, unknown request), PA_ERR_NO_BLOCKS
 * (not enough free blocks: nothing changed), PA_ERR_WORKSPACE (an output array too small:
 * nothing changed).
 */
#ifndef PA_KV_MANAGER_H
#define PA_KV_MANAGER_H

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_kvm pa_kvm;

/* New manager over a pool of num_blocks blocks of block_size tokens (block_size 8, 16 or 32).
 * enable_prefix_cache = 0 turns caching off (lookups miss, nothing is registered). */
int pa_kvm_create(int num_blocks, int block_size, int enable_prefix_cache, pa_kvm **out);
void pa_kvm_destroy(pa_kvm *m);

/* Longest cached prefix of tokens[0..num_tokens): writes the hit block ids (in order) to
 * block_ids (capacity max_blocks) and their count to num_hit_blocks.  Changes no state
 * except the lookup counters. */
int pa_kvm_get_computed_blocks(pa_kvm *m, const int32_t *tokens, int num_tokens, int32_t *block_ids,
                               int max_blocks, int *num_hit_blocks);

/* Register request req_id (new) with its prompt tokens: its block table starts with the
 * prefix-cache hits of the prompt, which it now holds.  *num_computed_tokens = hits *
 * block_size (tokens whose K/V are already in the cache). */
int pa_kvm_admit(pa_kvm *m, int64_t req_id, const int32_t *tokens, int num_tokens,
                 int *num_computed_tokens);

/* Grow request req_id to hold num_tokens tokens in total.  Copy-on-write pairs (at most one)
 * go to copy_pairs as (src, dst) int64 pairs (capacity max_pairs pairs), their count to
 * *num_pairs. */
int pa_kvm_allocate_slots(pa_kvm *m, int64_t req_id, int num_tokens, int64_t *copy_pairs,
                          int max_pairs, int *num_pairs);

/* Register the full blocks among the first num_computed_tokens tokens of request req_id
 * (tokens: the request's whole token sequence so far) in the prefix cache. */
int pa_kvm_cache_blocks(pa_kvm *m, int64_t req_id, const int32_t *tokens, int num_computed_tokens);

/* Release request req_id's blocks (last block first) and forget the request. */
int pa_kvm_free(pa_kvm *m, int64_t req_id);

/* New request child holding all of parent's blocks (shared, e.g. for parallel sampling). */
int pa_kvm_fork(pa_kvm *m, int64_t parent, int64_t child);

/* Block table of request req_id (capacity max_blocks); *num_blocks = its length. */
int pa_kvm_block_table(const pa_kvm *m, int64_t req_id, int32_t *out, int max_blocks, int *num_blocks);

/* Slots of positions first_pos .. first_pos+count-1 of request req_id:
 * block_table[pos / block_size] * block_size + pos % block_size.  The positions must be
 * covered by the request's blocks. */
int pa_kvm_slot_mapping(const pa_kvm *m, int64_t req_id, int first_pos, int count, int64_t *slots);

/* Blocks in the free queue (cached ones included). */
int pa_kvm_num_free_blocks(const pa_kvm *m);

/* Counters: out[0] lookups, out[1] blocks looked up, out[2] blocks hit, out[3] blocks
 * currently cached, out[4] cached blocks evicted (handed out again). */
int pa_kvm_stats(const pa_kvm *m, int64_t out[5]);

#ifdef __cplusplus
}
#endif

#endif /* PA_KV_MANAGER_H */
