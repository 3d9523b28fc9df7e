// decode.cu -- host side of paged decode: workspace layout, parameters, tensor maps,
// and the plain (query not rotated) kernel instantiations.  The kernels and the
// design are described in decode_kernels.cuh.
#include <atomic>
#include <chrono>
#include <random>

#include "decode_kernels.cuh"

namespace pa {
namespace {

// ------------------------------------------------------------------------------ host side

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    int HG, groups, HGq, K, C;
    size_t seg, k0, m, l, o, tag, total;
};

// Query slices per kv head: two when a kv head has eight query heads (each consumer warp then
// holds four of them), else one.
int query_slices(int num_heads, int num_kv_heads) { return num_heads / num_kv_heads > 4 ? 2 : 1; }

Layout layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int sms) {
    Layout L{};
    const int hg_max = 8 / query_slices(num_heads, num_kv_heads);  // kv heads a stage holds
    L.HG = num_kv_heads < hg_max ? num_kv_heads : hg_max;
    L.groups = num_kv_heads / L.HG;
    L.HGq = L.HG * (num_heads / num_kv_heads);
    L.K = L.groups * num_seqs;
    L.C = sms;
    const size_t pieces = (size_t)(L.C + L.K) * L.HGq;
    L.seg = 0;
    L.k0 = L.seg + align_up(sizeof(int32_t) * (L.K + 1));
    L.m = L.k0 + align_up(sizeof(int32_t) * L.C);
    L.l = L.m + align_up(sizeof(float) * pieces);
    L.o = L.l + align_up(sizeof(float) * pieces);
    L.tag = L.o + align_up(sizeof(float) * pieces * head_dim);
    L.total = L.tag + align_up(sizeof(unsigned long long) * (1 + L.C + L.K));
    return L;
}

// A 64-bit value no earlier launch of this process used and that data left in a workspace
// is vanishingly unlikely to hold: a counter mixed with a per-process seed through the
// SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", 2014).
unsigned long long next_launch_tag() {
    static std::atomic<unsigned long long> counter{0};
    static const unsigned long long seed = [] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ rd() ^
               (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
    }();
    unsigned long long z = seed + 0x9E3779B97F4A7C15ull * (counter.fetch_add(1) + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (z ^ (z >> 31)) | 1ull;
}

int grid_ctas() {
    const int sms = device_sm_count();
    return sms > 0 ? (sms < kMaxPieces ? sms : kMaxPieces) : kMaxPieces;  // no device: upper bound
}

}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int max_context_len) {
    (void)max_context_len;
    return layout(num_seqs, num_heads, num_kv_heads, head_dim, grid_ctas()).total;
}

int launch_decode(const DecodeArgs &a) {
    if (a.num_seqs == 0) return PA_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    const Layout L = layout(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                            sms < kMaxPieces ? sms : kMaxPieces);
    if (a.workspace_bytes < L.total) return PA_ERR_WORKSPACE;
    // Eight query heads per kv head on a 16-bit cache, with (sequence, kv head) pairs enough
    // to occupy most SMs: each sequence's query row goes through the tensor-core chunk kernel
    // as a one-token chunk (q.k and p.v on the tensor cores, the weights rounded to the
    // cache's type before p.v), which outruns the CUDA-core split for this grouping; a fused
    // cache write becomes the cache-write launch in front of it.
    const int G8 = a.num_heads / a.num_kv_heads;
    if (G8 == 8 && a.kv_dtype != PA_F32 && !a.rope_freqs && 5 * (int64_t)a.num_seqs * a.num_kv_heads >= 2 * (int64_t)sms) {
        if (a.new_key) {
            const int eb16 = 2;
            const int rc = launch_reshape_and_cache(a.new_key, a.new_value, const_cast<void *>(a.key_cache),
                                                    const_cast<void *>(a.value_cache), a.slot_mapping, a.num_seqs,
                                                    a.num_kv_heads * a.head_dim * eb16, a.block_size, a.num_blocks,
                                                    a.status, a.stream);
            if (rc != PA_OK) return rc;
        }
        PrefillArgs pf{a.out,          a.out_dtype,       a.query,        nullptr,      a.num_seqs,
                       1,              a.key_cache,       a.value_cache,  a.block_tables, a.max_blocks_per_seq,
                       a.context_lens, a.max_context_len, a.num_seqs,     a.num_heads,  a.num_kv_heads,
                       a.head_dim,     a.block_size,      a.num_blocks,   a.scale,      a.kv_dtype,
                       a.status,       a.stream};
        pf.decode_rows = 1;
        return launch_prefill(pf);
    }
    char *ws = static_cast<char *>(a.workspace);
    DecodeParams prm{};
    prm.out = a.out;
    prm.out_dtype = a.out_dtype;
    prm.query = a.query;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.seg_start = reinterpret_cast<int32_t *>(ws + L.seg);
    prm.cta_k0 = reinterpret_cast<int32_t *>(ws + L.k0);
    prm.part_m = reinterpret_cast<float *>(ws + L.m);
    prm.part_l = reinterpret_cast<float *>(ws + L.l);
    prm.part_o = reinterpret_cast<float *>(ws + L.o);
    prm.tags = reinterpret_cast<unsigned long long *>(ws + L.tag);
    prm.launch_tag = next_launch_tag();
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(a.stream, &capture) != cudaSuccess) return PA_ERR_CUDA;
    prm.tagged = capture == cudaStreamCaptureStatusNone ? 1 : 0;
    prm.max_blocks_per_seq = a.max_blocks_per_seq;
    prm.num_seqs = a.num_seqs;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.block_size = a.block_size;
    prm.num_blocks = a.num_blocks;
    prm.max_context_len = a.max_context_len;
    prm.head_dim = a.head_dim;
    prm.heads_per_group = L.HG;
    prm.num_groups = L.groups;
    prm.grid = L.C;
    prm.qk_scale_log2 = a.scale * kLog2e;
    prm.status = a.status;
    prm.rope_freqs = a.rope_freqs;
    prm.rope_dim = a.rope_dim;
    prm.q_scale_beta = a.q_scale_beta;
    prm.q_scale_orig_ctx = a.q_scale_orig_ctx;
    prm.new_key = a.new_key;
    prm.new_value = a.new_value;
    prm.slot_mapping = a.slot_mapping;
    prm.key_cache_w = const_cast<void *>(a.key_cache);
    prm.value_cache_w = const_cast<void *>(a.value_cache);
    prm.num_slots = (int64_t)a.num_blocks * a.block_size;

    // box rows are set per instantiation (they depend on the stage shape); encode the
    // tensor maps with the largest box the shape can use and re-encode if smaller.
    const int eb = a.kv_dtype == PA_F32 ? 4 : 2;
    const int G = a.num_heads / a.num_kv_heads;
    const int qs = query_slices(a.num_heads, a.num_kv_heads);
    const int nt = a.head_dim * eb <= 256 ? 16 : 8;  // DecodeShape::NT (at most four heads per warp)
    const int tu = nt * (kConsumerWarps / (L.HG * qs));
    const int rows = a.block_size < tu ? a.block_size : tu;
    const int64_t pool_rows = (int64_t)a.num_blocks * a.block_size;
    if (pool_rows <= 0 || pool_rows > INT32_MAX) return PA_ERR_INVALID_ARG;
    CUtensorMap km, vm;
    if (make_kv_tensor_map(&km, a.key_cache, a.kv_dtype, a.head_dim, a.num_kv_heads, pool_rows, L.HG,
                           rows) != PA_OK ||
        make_kv_tensor_map(&vm, a.value_cache, a.kv_dtype, a.head_dim, a.num_kv_heads, pool_rows,
                           L.HG, rows) != PA_OK)
        return PA_ERR_CUDA;
    if (a.rope_freqs) return dispatch_decode_rope(prm, a.kv_dtype, a.head_dim, G, km, vm, a.stream);
    if (a.new_key) return dispatch_decode_write(prm, a.kv_dtype, a.head_dim, G, km, vm, a.stream);
    return dispatch_kv<false>(prm, a.kv_dtype, a.head_dim, G, km, vm, a.stream);
}

}  // namespace pa
