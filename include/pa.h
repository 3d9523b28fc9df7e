/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * Paged attention over a block-tabled KV cache, as described on the
 * TensorSharp "Mistral 3" model page, section 11 "Batched / paged forward
 * (continuous batching)", and on the mistral.rs part of the "pure Rust
 * engines" page (paged attention, KV-cache manager, prefix cache and
 * scheduler sections).  Four operations:
 *
 *   pa_reshape_and_cache  write fresh K/V into cache slots through a slot map
 *   pa_decode             one query token per sequence, split-K over the
 *                         context, log-sum-exp reduce
 *   pa_prefill_chunk      a chunk of query tokens per sequence: causal inside
 *                         the chunk, full over the cached prefix
 *   pa_copy_blocks        whole-block copies for prefix-cache reuse
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor argument is a pointer to DEVICE memory owned by the caller,
 *    dense row-major, 16-byte aligned.  The library allocates nothing, keeps
 *    no state between calls and never synchronises the device.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.
 *  - The return value is PA_OK (0) or a negative PA_ERR_* code.  Argument
 *    errors are detected on the host before anything is launched.  A failed
 *    launch returns PA_ERR_CUDA.
 *  - The first call of pa_decode, pa_decode_rope, pa_decode_noalloc or
 *    pa_prefill_chunk on a device raises its kernels' shared-memory limit
 *    (cudaFuncSetAttribute) and may load the library's device code into the
 *    current context; make that first call outside stream capture.  Calls
 *    from several host threads are safe (per-device setup is atomic).
 *  - Values that only the device can see (slot numbers, block ids, context
 *    lengths) are range-checked inside the kernels: an out-of-range value is
 *    never dereferenced; the offending token / block is skipped and, if
 *    `status` is not NULL, the matching PA_DEVERR_* bit is OR-ed into the
 *    device int32 `*status`.  The caller clears *status and reads it after
 *    synchronising.
 *
 * Layouts (S sequences, Hq query heads, Hkv kv heads, D head dim, bs block
 * size, NB blocks in the pool; G = Hq / Hkv; query head h reads kv head h / G)
 *  - key_cache, value_cache: [NB][bs][Hkv][D], the flat
 *    [numBlocks * blockSize * numKvHeads * headDim] per-layer buffer of the
 *    TensorSharp page, section 11.  Token slot `slot` is row slot of the
 *    [NB * bs][Hkv][D] view: block slot / bs, offset slot % bs.
 *  - block_tables: int32 [S][max_blocks_per_seq]; logical token j of sequence
 *    s lives in physical block block_tables[s][j / bs] at offset j % bs.
 *    Entries past ceil(context_lens[s] / bs) are never read.
 *  - context_lens: int32 [S]; the number of keys the sequence's last query row
 *    sees, the freshly written token(s) included.
 *
 * Supported shapes: dtype F32, F16 or BF16 (query and cache share it); D in
 * {64, 128}; bs in {8, 16, 32} (the mistral.rs page's allowed block sizes);
 * Hq a multiple of Hkv with G = Hq / Hkv in {1, 2, 4, 8}; Hkv in {1, 2, 4} or
 * a multiple of 8; num_blocks * block_size < 2^31.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *pa_stream_t;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1, /* null / misaligned pointer, negative size, bad dtype */
    PA_ERR_UNSUPPORTED = -2, /* head_dim, block_size or head grouping not built */
    PA_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required */
    PA_ERR_CUDA = -4,        /* a kernel launch failed (cudaGetLastError) */
    PA_ERR_NO_BLOCKS = -5    /* KV-cache manager: not enough free blocks (nothing changed) */
};

/* Bits OR-ed into the optional device-side `*status` word. */
enum {
    PA_DEVERR_SLOT = 1,      /* slot_mapping entry >= num_blocks * block_size */
    PA_DEVERR_BLOCK_ID = 2,  /* block table / block mapping id outside [0, num_blocks) */
    PA_DEVERR_CONTEXT = 4,   /* context length < 0, > max_context_len, or beyond the block table */
    PA_DEVERR_QUERY = 8,     /* query_start_loc not monotone, or a chunk longer than its context */
    PA_DEVERR_TIMEOUT = 16   /* a bounded wait inside a kernel gave up (internal error; the
                                kernel returned instead of hanging) */
};

/*
 * pa_reshape_and_cache -- write fresh keys and values into their cache slots.
 * TensorSharp "Mistral 3" page, section 11 (K/V scatter via slotMapping to
 * blockId * blockSize + offset; no per-sequence extract / inject).
 *
 *   key, value     [num_tokens][num_kv_heads][head_dim], kv_dtype (read)
 *   key_cache,
 *   value_cache    [num_blocks][block_size][num_kv_heads][head_dim] (written)
 *   slot_mapping   int64 [num_tokens]; slot < 0 skips the token (padding)
 *
 * Each written row is a bit copy.  Tokens must map to distinct slots (two
 * tokens writing one slot race).  num_tokens == 0 is a no-op.
 */
int pa_reshape_and_cache(const void *key, const void *value, void *key_cache, void *value_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype kv_dtype,
                         int32_t *status, pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * these sizes on the current device (0 only when num_seqs == 0).  The value
 * depends on its arguments and on the device's SM count (the split of the
 * contexts is balanced over one CTA per SM); on a machine without a visible
 * device it returns an upper bound.  Returns 0 for arguments pa_decode would
 * reject.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int max_context_len);

/*
 * pa_decode -- decode attention: one query token per sequence against every
 * cached key of that sequence, gathered through its block table.
 * TensorSharp "Mistral 3" page, section 11 (per-sequence paged attention over
 * the paged K/V buffer) and sections 3 / 4.1 (standard causal GQA attention,
 * Q scaled by 1/sqrt(headDim)).
 *
 *   out            [num_seqs][num_heads][head_dim], out_dtype (written)
 *   query          [num_seqs][num_heads][head_dim], kv_dtype
 *   key_cache,
 *   value_cache    [num_blocks][block_size][num_kv_heads][head_dim], kv_dtype
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs]; max_context_len >= every entry (host bound
 *                  used to size the split of the context)
 *   scale          softmax scale applied to q.k (normally 1/sqrt(head_dim))
 *   workspace      device scratch of >= pa_decode_workspace_size(...) bytes,
 *                  16-byte aligned, owned by the caller; it needs no
 *                  initialisation (each call marks what it writes with its own
 *                  64-bit tag), its contents are clobbered, and two calls in
 *                  flight must not share it
 *
 * A call made while `stream` is being captured into a CUDA graph is replayable: the
 * merge of the split context then waits for the whole first pass instead of the
 * per-call tags (a replay repeats the captured tag), a few microseconds slower.
 *
 *   out[s][h] = sum_j softmax_j(scale * q[s][h] . k_j) v_j over j < context_lens[s];
 *   a sequence with context length 0 gets an all-zero row.
 * Accumulation is fp32; the result does not depend on the split.
 * With eight query heads per kv head, an fp16/bf16 cache and num_seqs * num_kv_heads
 * >= 0.4 x the SM count, the rows run on the tensor cores instead (the chunked-prefill
 * kernel with one-token chunks): q.k and p.v in fp32 accumulators, the softmax weights
 * rounded to the cache's type before p.v (as in pa_prefill_chunk), each (sequence, kv
 * head) in one fixed key order, so that a row does not depend on the rest of the batch
 * while the call stays on this path; the workspace is then not touched.  A row computed
 * on the two paths (a small batch and a large one) agrees within the attention tolerance,
 * not bit for bit.  One to four query heads per kv head always take the split path.
 */
int pa_decode(void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
              const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
              int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
              pa_dtype kv_dtype, void *workspace, size_t workspace_bytes, int32_t *status,
              pa_stream_t stream);

/*
 * pa_decode_write -- pa_reshape_and_cache of one new token per sequence followed by
 * pa_decode, in one launch (the decode step of a serving loop: the TensorSharp "Mistral 3"
 * page, section 11, writes the step's K/V through slotMapping, then attends).
 *
 *   key, value     [num_seqs][num_kv_heads][head_dim], kv_dtype (device): token s is the
 *                  newest token of sequence s
 *   slot_mapping   int64 [num_seqs]: its cache slot (blockId * block_size + offset); a
 *                  negative slot writes nothing, a slot past the pool is reported
 *                  (PA_DEVERR_SLOT) and not written
 *   key_cache,
 *   value_cache    written at those slots, then read as by pa_decode
 *   (every other argument as for pa_decode)
 *
 * Precondition (the decode step of any paged KV manager): slot_mapping[s] is the slot that
 * block_tables[s] gives position context_lens[s] - 1, and no other sequence of the call
 * reads that slot (a block being appended to is never shared).  Then out and both pools
 * equal those of pa_reshape_and_cache(key, value, ..., slot_mapping, num_seqs, ...) and
 * pa_decode(...) on the same stream, bit for bit.  Otherwise the pools are written as
 * stated and out is unspecified.  The launch that streams a sequence's last keys stores
 * the token and uses it from the same copy, so no kernel boundary separates the two
 * (where pa_decode runs its rows on the tensor cores, the write is a launch of its own
 * in front of them).
 */
int pa_decode_write(void *out, pa_dtype out_dtype, const void *query, const void *key,
                    const void *value, const int64_t *slot_mapping, void *key_cache,
                    void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                    pa_dtype kv_dtype, void *workspace, size_t workspace_bytes, int32_t *status,
                    pa_stream_t stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory: plugin hosts and serving runtimes that own all device memory and hand
 * kernels only their tensors, hot paths where a cudaMalloc could synchronise
 * the device, and language bindings without a device allocator.  The pages
 * describe no such call; it exists only for these callers.
 *
 * Same arguments, results and error behaviour as pa_decode, without the
 * workspace: the scratch lives in one static device array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES inside the library (held by every GPU that
 * loads the library until the process exits).  A problem whose scratch
 * (pa_decode_workspace_size) exceeds it returns PA_ERR_WORKSPACE before
 * anything runs; with 152 SMs, Hq = 32, Hkv = 8 and D = 128 that allows about 350
 * sequences.  Nothing is allocated and nothing needs clearing between calls.
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress), so the address never goes stale across device resets
 * or contexts.  The first call in a context loads the library's device code
 * there and sets up the decode kernels: make that first call before any stream
 * capture.  All calls on a device share the one array: two calls whose kernels overlap
 * on the GPU (different streams, no ordering between them) race and corrupt
 * each other's results.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int pa_decode_noalloc(void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
                      const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
                      int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                      pa_dtype kv_dtype, int32_t *status, pa_stream_t stream);

/*
 * pa_prefill_chunk -- chunked-prefill attention.  Sequence s owns the packed
 * query rows query_start_loc[s] .. query_start_loc[s+1]-1 (Lq_s rows, the
 * newest tokens of the sequence, whose K/V are already in the cache).  Row i
 * sits at absolute position context_lens[s] - Lq_s + i and attends keys
 * 0 .. that position: full attention over the cached prefix, causal inside
 * the chunk.  mistral.rs page, scheduling section (prompts chunked under a
 * token budget of 4096, 512 per chunk); TensorSharp page, section 11.
 *
 *   out              [num_tokens][num_heads][head_dim], out_dtype (written)
 *   query            [num_tokens][num_heads][head_dim], kv_dtype (F16 or BF16)
 *   query_start_loc  int32 [num_seqs + 1], non-decreasing, [0] = 0,
 *                    [num_seqs] = num_tokens
 *   max_query_len    >= every Lq_s (host bound used to size the grid)
 *   other arguments  as for pa_decode
 *
 * Tensor-core MMA with fp32 accumulation; the softmax weights are rounded to
 * the input dtype before the P.V product.
 */
int pa_prefill_chunk(void *out, pa_dtype out_dtype, const void *query,
                     const int32_t *query_start_loc, int num_tokens, int max_query_len,
                     const void *key_cache, const void *value_cache, const int32_t *block_tables,
                     int max_blocks_per_seq, const int32_t *context_lens, int max_context_len,
                     int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, float scale, pa_dtype kv_dtype, int32_t *status,
                     pa_stream_t stream);

/*
 * pa_copy_blocks -- copy whole cache blocks, K and V, for prefix-cache reuse
 * (mistral.rs page, block-hash prefix cache: full blocks are shared by
 * content; a copy gives a sequence its own writable copy of a shared block).
 *
 *   block_mapping  int64 [num_pairs][2] = (src, dst) block ids
 *
 * Destinations must be distinct and must not appear as sources (then the
 * result equals copying the pairs one after another); otherwise the result
 * is undefined.  num_pairs == 0 is a no-op.
 */
int pa_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_dtype kv_dtype, int32_t *status, pa_stream_t stream);

/*
 * Rotary position embedding fused into the cache write and the decode query load
 * (TensorSharp "Mistral 3" page, section 3 "Forward graph" and section 4.2 "RoPE - GPT-J
 * style with YaRN": RoPE rotates Q and K with the GPT-J pairing -- adjacent elements
 * (x[2i], x[2i+1]) rotate together -- at each token's absolute position, with a frequency
 * table built once at load time (YaRN-corrected when the model asks for it); Q is then
 * scaled by 1 + beta * log(1 + floor(pos / origCtx)) when origCtx > 0).
 *
 * Pair i (i < rope_dim / 2) of a row at position pos is rotated by the angle
 * pos * freqs[i]:  (x, y) -> (x cos - y sin, x sin + y cos).  The angle is formed exactly
 * (as a sum of two floats) and reduced to [-pi, pi] in fp32 (within 2.3e-7 of the exact
 * reduced angle for |pos| < 2^24; positions beyond lose that bound), its sine and cosine
 * taken in fp32 (absolute error below 4e-7), the rotation done in fp32.  Elements past
 * rope_dim are not rotated.  The 1/sqrt(head_dim) factor stays the attention's `scale`
 * argument.
 */
typedef struct {
    const float *freqs;   /* device, [rope_dim / 2]: angular frequency of pair i (pa_rope_yarn_freqs) */
    int rope_dim;         /* even, 2 .. head_dim */
    float q_scale_beta;   /* beta of the position-dependent query scale */
    int q_scale_orig_ctx; /* origCtx of the query scale; 0 turns the scale off */
} pa_rope;

/*
 * pa_rope_yarn_freqs -- host: the frequency table, freqs[i] = base^(-2i / rope_dim), then
 * YaRN-corrected when yarn_scale != 1 and orig_ctx > 0 (section 4.2): with r = orig_ctx /
 * (2 pi / f), the number of turns pair i makes over the original context, a pair with
 * r > beta_fast keeps f (extrapolation), one with r < beta_slow takes f / yarn_scale
 * (interpolation), and in between f mixes linearly in r: f * (1 - g) + f / yarn_scale * g
 * with g = (beta_fast - r) / (beta_fast - beta_slow).  Computed in double, stored fp32.
 * freqs: host array of rope_dim / 2 floats.
 */
int pa_rope_yarn_freqs(float *freqs, int rope_dim, float base, float yarn_scale, int orig_ctx,
                       float beta_fast, float beta_slow);

/*
 * pa_reshape_and_cache_rope -- pa_reshape_and_cache with K rotated on the way in:
 * token t's key row is rotated at position positions[t] (int32 [num_tokens], device)
 * before it is written; values are copied as they are.  Same layouts, skip rule and errors
 * as pa_reshape_and_cache, plus PA_ERR_INVALID_ARG for a missing rope/positions/freqs, an
 * odd rope_dim or one outside 2..head_dim.
 */
int pa_reshape_and_cache_rope(const void *key, const void *value, void *key_cache, void *value_cache,
                              const int64_t *slot_mapping, const int32_t *positions, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              pa_dtype kv_dtype, const pa_rope *rope, int32_t *status,
                              pa_stream_t stream);

/*
 * pa_decode_rope -- pa_decode with the query rotated and scaled as it is loaded: the query
 * of sequence s sits at position context_lens[s] - 1 (the newest token), is rotated there
 * and, when q_scale_orig_ctx > 0, multiplied by 1 + q_scale_beta * log(1 + floor(pos /
 * q_scale_orig_ctx)); `query` holds the unrotated query.  Keys must already be rotated in
 * the cache (pa_reshape_and_cache_rope).  Arguments otherwise as pa_decode.
 */
int pa_decode_rope(void *out, pa_dtype out_dtype, const void *query, const void *key_cache,
                   const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                   pa_dtype kv_dtype, const pa_rope *rope, void *workspace, size_t workspace_bytes,
                   int32_t *status, pa_stream_t stream);

/* Static description of a PA_* return code. */
const char *pa_status_string(int code);

/* Library version as major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
