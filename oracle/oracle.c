/*
 * oracle.c -- plain, slow, fp64 CPU oracle for paged attention over a
 * block-tabled KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA library: it decodes the element formats itself, walks the
 * block table itself and runs dense two-pass softmax attention in double.
 *
 * Sources (TensorSharp "Mistral 3" model page, section 11 "Batched / paged
 * forward (continuous batching)"):
 *   - paged K/V buffers per layer, flat layout
 *     [numBlocks * blockSize * numKvHeads * headDim]  -> pool[NB][bs][Hkv][D];
 *   - fresh K/V scattered through a slot mapping to blockId*blockSize+offset;
 *   - per sequence: gather K/V from the paged buffer, then fused attention.
 * Same page, section 3 "Forward graph" and 4.1 "Attention": causal GQA
 * attention with Q scaled by 1/sqrt(headDim) (the `scale` argument here).
 * mistral.rs page ("pure Rust engines"), paged-attention section: block
 * sizes 8/16/32; block copy is the data side of block-hash prefix reuse.
 *
 * Readings where the pages are silent (each is stated again in the design
 * notes):
 *   - slot < 0 in the slot mapping means "skip this token" (padding);
 *   - GQA heads grouped consecutively: kv head = h / (Hq / Hkv);
 *   - context_lens[s] counts every key visible to the sequence's last query
 *     row, the freshly written token(s) included;
 *   - a chunk of Lq query rows is aligned bottom-right: row i sits at
 *     absolute position context_lens[s] - Lq + i and sees keys 0..pos;
 *   - a sequence with context length 0 produces an all-zero output row;
 *   - block copies run in the order given (sequential semantics).
 *
 * Every entry point returns 0 on success and a negative code on a bad
 * argument (the oracle checks indices instead of reading out of range).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_INDEX -2
#define OR_ERR_NOMEM -3

static int elem_bytes(int dtype)
{
    if (dtype == OR_F32) return 4;
    if (dtype == OR_F16 || dtype == OR_BF16) return 2;
    return 0;
}

/* IEEE-754 binary16 -> double, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = m ? NAN : INFINITY;
    else
        mag = ldexp((double)(m + 1024), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of a binary32 word. */
static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double f32_to_double(const void *p)
{
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/* Element `index` of an array of `dtype`, exactly widened to double. */
static double load_elem(const void *base, int64_t index, int dtype)
{
    const unsigned char *b = (const unsigned char *)base;
    if (dtype == OR_F32) return f32_to_double(b + 4 * index);
    uint16_t h;
    memcpy(&h, b + 2 * index, 2);
    return dtype == OR_F16 ? f16_to_double(h) : bf16_to_double(h);
}

/* Exposed so the tests can pin the element decoders against library
 * conversions over every bit pattern. */
double oracle_decode_elem(const void *base, int64_t index, int dtype)
{
    return load_elem(base, index, dtype);
}

/*
 * reshape_and_cache: for every token t with slot_mapping[t] >= 0, the
 * Hkv*D elements of key[t] and value[t] are copied, bit for bit, to
 * pool[slot / bs][slot % bs][:][:].  Nothing else in the pools changes.
 */
int oracle_reshape_and_cache(const void *key, const void *value,
                             void *key_cache, void *value_cache,
                             const int64_t *slot_mapping, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, int dtype)
{
    int eb = elem_bytes(dtype);
    if (!eb || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0)
        return OR_ERR_ARG;
    size_t row = (size_t)num_kv_heads * head_dim * eb; /* one token, all heads */
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        if (block >= num_blocks) return OR_ERR_INDEX;
        size_t dst = ((size_t)block * block_size + (size_t)offset) * row;
        memcpy((unsigned char *)key_cache + dst, (const unsigned char *)key + (size_t)t * row, row);
        memcpy((unsigned char *)value_cache + dst, (const unsigned char *)value + (size_t)t * row, row);
    }
    return OR_OK;
}

/*
 * copy_blocks: for each pair (src, dst) of block_mapping, in order, the whole
 * block [bs][Hkv][D] of both pools is copied from src to dst.
 */
int oracle_copy_blocks(void *key_cache, void *value_cache,
                       const int64_t *block_mapping, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int dtype)
{
    int eb = elem_bytes(dtype);
    if (!eb || num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0)
        return OR_ERR_ARG;
    size_t blk = (size_t)block_size * num_kv_heads * head_dim * eb;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p];
        int64_t dst = block_mapping[2 * p + 1];
        if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) return OR_ERR_INDEX;
        memmove((unsigned char *)key_cache + (size_t)dst * blk,
                (const unsigned char *)key_cache + (size_t)src * blk, blk);
        memmove((unsigned char *)value_cache + (size_t)dst * blk,
                (const unsigned char *)value_cache + (size_t)src * blk, blk);
    }
    return OR_OK;
}

/*
 * Softmax attention of one query vector over n keys, in double, two passes:
 *   x_j = scale * sum_d q[d] k_j[d];  m = max_j x_j;  w_j = exp(x_j - m);
 *   out[d] = sum_j w_j v_j[d] / sum_j w_j.
 * K and V are dense [n][D] arrays (already gathered).  n == 0 gives zeros.
 */
static void attend_one(double *out, const double *q, const double *K,
                       const double *V, int n, int D, double scale,
                       double *x /* scratch, n entries */)
{
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n <= 0) return;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * K[(size_t)j * D + d];
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
    }
    double den = 0.0;
    for (int j = 0; j < n; ++j) {
        x[j] = exp(x[j] - m);
        den += x[j];
    }
    for (int j = 0; j < n; ++j)
        for (int d = 0; d < D; ++d) out[d] += x[j] * V[(size_t)j * D + d];
    for (int d = 0; d < D; ++d) out[d] /= den;
}

/*
 * Shared tail of the paged and the dense oracle: given the gathered keys and
 * values of one (sequence, kv head) pair, run every query row and every
 * query head of the group.
 *   q rows:  query[(q0 + i) * Hq * D + h * D + d], i in [0, Lq)
 *   row i sits at position C - Lq + i and attends keys 0..C-Lq+i.
 */
static void attend_group(double *out, const void *query, int q_dtype,
                         int64_t q0, int Lq, int C, int g, int Hq, int Hkv,
                         int D, double scale, const double *K, const double *V,
                         double *qv, double *x)
{
    int G = Hq / Hkv;
    for (int i = 0; i < Lq; ++i) {
        int pos = C - Lq + i;
        for (int hh = 0; hh < G; ++hh) {
            int h = g * G + hh;
            int64_t base = ((q0 + i) * Hq + h) * (int64_t)D;
            for (int d = 0; d < D; ++d) qv[d] = load_elem(query, base + d, q_dtype);
            attend_one(out + base, qv, K, V, pos + 1, D, scale, x);
        }
    }
}

/*
 * Paged attention (decode is the case Lq = 1 for every sequence).
 *   query            [Tq][Hq][D] packed rows, q_dtype
 *   query_start_loc  [S+1]; sequence s owns rows qsl[s] .. qsl[s+1]-1
 *   key/value_cache  [NB][bs][Hkv][D], kv_dtype
 *   block_tables     [S][max_blocks_per_seq] int32
 *   context_lens     [S] int32, keys visible to the sequence's last row
 *   out              [Tq][Hq][D] double
 * Logical key j of sequence s lives at
 *   pool[block_tables[s][j / bs]][j % bs][kv_head][:].
 */
int oracle_paged_attention(double *out, const void *query, int q_dtype,
                           const int32_t *query_start_loc, int num_seqs,
                           const void *key_cache, const void *value_cache,
                           int kv_dtype, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens,
                           int num_heads, int num_kv_heads, int head_dim,
                           int block_size, int num_blocks, float scale)
{
    if (!elem_bytes(q_dtype) || !elem_bytes(kv_dtype) || num_seqs < 0 ||
        num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        head_dim <= 0 || block_size <= 0 || max_blocks_per_seq < 0)
        return OR_ERR_ARG;
    /* Check every index before touching memory. */
    for (int s = 0; s < num_seqs; ++s) {
        int C = context_lens[s];
        int Lq = query_start_loc[s + 1] - query_start_loc[s];
        if (C < 0 || Lq < 0 || (Lq > C && C > 0)) return OR_ERR_INDEX;
        if (C == 0 || Lq == 0) continue; /* nothing is read */
        int nblk = (C + block_size - 1) / block_size;
        if (nblk > max_blocks_per_seq) return OR_ERR_INDEX;
        for (int b = 0; b < nblk; ++b) {
            int32_t id = block_tables[(size_t)s * max_blocks_per_seq + b];
            if (id < 0 || id >= num_blocks) return OR_ERR_INDEX;
        }
    }
    const int Hq = num_heads, Hkv = num_kv_heads, D = head_dim, bs = block_size;
    const double sc = (double)scale;
    int status = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int task = 0; task < num_seqs * Hkv; ++task) {
        int s = task / Hkv, g = task % Hkv;
        int C = context_lens[s];
        int64_t q0 = query_start_loc[s];
        int Lq = query_start_loc[s + 1] - query_start_loc[s];
        if (Lq == 0) continue;
        size_t n = C > 0 ? (size_t)C : 1;
        double *K = (double *)malloc(n * D * sizeof(double));
        double *V = (double *)malloc(n * D * sizeof(double));
        double *qv = (double *)malloc((size_t)D * sizeof(double));
        double *x = (double *)malloc(n * sizeof(double));
        if (!K || !V || !qv || !x) {
            status = OR_ERR_NOMEM;
        } else {
            /* Gather logical keys/values 0..C-1 through the block table. */
            for (int j = 0; j < C; ++j) {
                int32_t blk = block_tables[(size_t)s * max_blocks_per_seq + j / bs];
                int64_t row = (((int64_t)blk * bs + j % bs) * Hkv + g) * (int64_t)D;
                for (int d = 0; d < D; ++d) {
                    K[(size_t)j * D + d] = load_elem(key_cache, row + d, kv_dtype);
                    V[(size_t)j * D + d] = load_elem(value_cache, row + d, kv_dtype);
                }
            }
            attend_group(out, query, q_dtype, q0, Lq, C, g, Hq, Hkv, D, sc, K, V, qv, x);
        }
        free(K); free(V); free(qv); free(x);
    }
    return status;
}

/*
 * Dense attention over a contiguous per-sequence cache [Hkv][Lmax][D] of
 * doubles (the layout of the per-sequence KV-swap path on the same page,
 * section 10).  Same row/position rules as the paged oracle.  Used only to
 * check the paged oracle's gather.
 *   k_dense, v_dense  [S][Hkv][Lmax][D] double
 */
int oracle_dense_attention(double *out, const void *query, int q_dtype,
                           const int32_t *query_start_loc, int num_seqs,
                           const double *k_dense, const double *v_dense,
                           int max_len, const int32_t *context_lens,
                           int num_heads, int num_kv_heads, int head_dim,
                           float scale)
{
    if (!elem_bytes(q_dtype) || num_seqs < 0 || num_heads <= 0 ||
        num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
        max_len < 0)
        return OR_ERR_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int C = context_lens[s];
        int Lq = query_start_loc[s + 1] - query_start_loc[s];
        if (C < 0 || C > max_len || Lq < 0 || (Lq > C && C > 0)) return OR_ERR_INDEX;
    }
    const int Hkv = num_kv_heads, D = head_dim;
    int status = OR_OK;
    for (int s = 0; s < num_seqs; ++s) {
        for (int g = 0; g < Hkv; ++g) {
            int C = context_lens[s];
            int Lq = query_start_loc[s + 1] - query_start_loc[s];
            if (Lq == 0) continue;
            size_t off = ((size_t)s * Hkv + g) * (size_t)max_len * D;
            size_t n = C > 0 ? (size_t)C : 1;
            double *qv = (double *)malloc((size_t)D * sizeof(double));
            double *x = (double *)malloc(n * sizeof(double));
            if (!qv || !x) status = OR_ERR_NOMEM;
            else attend_group(out, query, q_dtype, query_start_loc[s], Lq, C, g,
                              num_heads, Hkv, D, (double)scale, k_dense + off,
                              v_dense + off, qv, x);
            free(qv); free(x);
        }
    }
    return status;
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
