// kv_manager.cpp -- host block pool and KV-cache manager (prefix caching, LRU free queue,
// copy-on-write for forked requests).  The policy is stated in include/pa_kv_manager.h;
// the operations follow the Pure-Rust engines page (paged-attention block management and
// prefix-cache sections) and the TensorSharp "Mistral 3" page, section 11.
//
// Data layout: one record per physical block (reference count, free-queue links, prefix
// key and, while cached, the block's tokens and its parent's key), an intrusive doubly
// linked free queue (O(1) removal when a lookup revives a free cached block), a hash map
// from prefix key to block, and a map from request id to its block table.
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_kv_manager.h"

namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;  // FNV-1a 64-bit parameters
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) {
        h ^= (v >> (8 * i)) & 0xffu;
        h *= kFnvPrime;
    }
    return h;
}

// Key of a full block: FNV-1a over the parent's key and the block's tokens (little-endian
// bytes, independent of the host's byte order).
uint64_t block_key(uint64_t parent, const int32_t *tok, int bs) {
    uint64_t h = fnv_bytes(kFnvOffset, parent, 8);
    for (int i = 0; i < bs; ++i) h = fnv_bytes(h, (uint32_t)tok[i], 4);
    return h;
}

struct Block {
    int32_t ref = 0;
    int32_t prev = -1, next = -1;  // free-queue links
    bool in_free = false;
    bool cached = false;
    uint64_t key = 0, parent = 0;
    std::vector<int32_t> tokens;   // content while cached (verified on a hit)
};

struct Request {
    std::vector<int32_t> blocks;
    int num_tokens = 0;   // tokens the blocks were sized for
    int num_cached = 0;   // leading blocks already registered (or hit) in the cache
    uint64_t chain = 0;   // prefix key of block num_cached - 1 (the next block's parent)
};

}  // namespace

struct pa_kvm {
    int num_blocks, bs;
    bool prefix_cache;
    std::vector<Block> blk;
    int32_t head = -1, tail = -1;
    int num_free = 0;
    std::unordered_map<uint64_t, int32_t> cache;
    std::unordered_map<int64_t, Request> reqs;
    int64_t lookups = 0, looked_blocks = 0, hit_blocks = 0, evictions = 0;

    void push_back(int32_t b) {
        Block &x = blk[b];
        x.prev = tail;
        x.next = -1;
        if (tail >= 0) blk[tail].next = b; else head = b;
        tail = b;
        x.in_free = true;
        ++num_free;
    }
    void unlink(int32_t b) {
        Block &x = blk[b];
        if (x.prev >= 0) blk[x.prev].next = x.next; else head = x.next;
        if (x.next >= 0) blk[x.next].prev = x.prev; else tail = x.prev;
        x.prev = x.next = -1;
        x.in_free = false;
        --num_free;
    }
    // Take the block at the head of the free queue; a cached block leaves the cache.
    int32_t pop_front() {
        const int32_t b = head;
        unlink(b);
        Block &x = blk[b];
        if (x.cached) {
            auto it = cache.find(x.key);
            if (it != cache.end() && it->second == b) cache.erase(it);
            x.cached = false;
            x.tokens.clear();
            ++evictions;
        }
        x.ref = 1;
        return b;
    }
    // Longest verified chain of cached blocks for tokens[0..n), at most (n - 1) / bs blocks;
    // *chain_out = prefix key of the last hit (the offset basis when there is none).
    void lookup(const int32_t *tokens, int n, std::vector<int32_t> &hits, uint64_t *chain_out = nullptr) {
        hits.clear();
        ++lookups;
        if (chain_out) *chain_out = kFnvOffset;
        if (!prefix_cache || n <= 1) return;
        const int nb = (n - 1) / bs;
        looked_blocks += nb;
        uint64_t parent = kFnvOffset;
        for (int i = 0; i < nb; ++i) {
            const int32_t *t = tokens + (size_t)i * bs;
            const uint64_t k = block_key(parent, t, bs);
            auto it = cache.find(k);
            if (it == cache.end()) break;
            const Block &x = blk[it->second];
            if (!x.cached || x.parent != parent || std::memcmp(x.tokens.data(), t, sizeof(int32_t) * bs) != 0)
                break;
            hits.push_back(it->second);
            parent = k;
        }
        if (chain_out) *chain_out = parent;
        hit_blocks += (int64_t)hits.size();
    }
};

extern "C" {

int pa_kvm_create(int num_blocks, int block_size, int enable_prefix_cache, pa_kvm **out) {
    if (!out || num_blocks <= 0 || !(block_size == 8 || block_size == 16 || block_size == 32))
        return PA_ERR_INVALID_ARG;
    pa_kvm *m = new (std::nothrow) pa_kvm();
    if (!m) return PA_ERR_INVALID_ARG;
    m->num_blocks = num_blocks;
    m->bs = block_size;
    m->prefix_cache = enable_prefix_cache != 0;
    m->blk.resize(num_blocks);
    for (int b = 0; b < num_blocks; ++b) m->push_back(b);
    *out = m;
    return PA_OK;
}

void pa_kvm_destroy(pa_kvm *m) { delete m; }

int pa_kvm_get_computed_blocks(pa_kvm *m, const int32_t *tokens, int num_tokens, int32_t *block_ids,
                               int max_blocks, int *num_hit_blocks) {
    if (!m || num_tokens < 0 || (num_tokens > 0 && !tokens) || !num_hit_blocks || max_blocks < 0)
        return PA_ERR_INVALID_ARG;
    std::vector<int32_t> hits;
    m->lookup(tokens, num_tokens, hits);
    if ((int)hits.size() > max_blocks || (!hits.empty() && !block_ids)) return PA_ERR_WORKSPACE;
    for (size_t i = 0; i < hits.size(); ++i) block_ids[i] = hits[i];
    *num_hit_blocks = (int)hits.size();
    return PA_OK;
}

int pa_kvm_admit(pa_kvm *m, int64_t req_id, const int32_t *tokens, int num_tokens,
                 int *num_computed_tokens) {
    if (!m || num_tokens < 0 || (num_tokens > 0 && !tokens) || !num_computed_tokens ||
        m->reqs.count(req_id))
        return PA_ERR_INVALID_ARG;
    std::vector<int32_t> hits;
    Request r;
    m->lookup(tokens, num_tokens, hits, &r.chain);
    for (int32_t b : hits) {
        Block &x = m->blk[b];
        if (x.ref == 0 && x.in_free) m->unlink(b);
        ++x.ref;
        r.blocks.push_back(b);
    }
    r.num_tokens = (int)hits.size() * m->bs;
    r.num_cached = (int)hits.size();
    m->reqs.emplace(req_id, std::move(r));
    *num_computed_tokens = (int)hits.size() * m->bs;
    return PA_OK;
}

int pa_kvm_allocate_slots(pa_kvm *m, int64_t req_id, int num_tokens, int64_t *copy_pairs,
                          int max_pairs, int *num_pairs) {
    if (!m || num_tokens < 0 || !num_pairs || max_pairs < 0) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(req_id);
    if (it == m->reqs.end()) return PA_ERR_INVALID_ARG;
    Request &r = it->second;
    const int bs = m->bs;
    const int want = (num_tokens + bs - 1) / bs;
    const int grow = want > (int)r.blocks.size() ? want - (int)r.blocks.size() : 0;
    // copy-on-write: new tokens go into a partial last block that another request holds
    const bool cow = num_tokens > r.num_tokens && r.num_tokens % bs != 0 && !r.blocks.empty() &&
                     m->blk[r.blocks.back()].ref > 1;
    if (grow + (cow ? 1 : 0) > m->num_free) return PA_ERR_NO_BLOCKS;
    if (cow && (max_pairs < 1 || !copy_pairs)) return PA_ERR_WORKSPACE;
    int pairs = 0;
    if (cow) {
        const int32_t old = r.blocks.back();
        const int32_t nb = m->pop_front();
        --m->blk[old].ref;
        r.blocks.back() = nb;
        copy_pairs[0] = old;
        copy_pairs[1] = nb;
        pairs = 1;
    }
    for (int i = 0; i < grow; ++i) r.blocks.push_back(m->pop_front());
    if (num_tokens > r.num_tokens) r.num_tokens = num_tokens;
    *num_pairs = pairs;
    return PA_OK;
}

int pa_kvm_cache_blocks(pa_kvm *m, int64_t req_id, const int32_t *tokens, int num_computed_tokens) {
    if (!m || num_computed_tokens < 0 || (num_computed_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(req_id);
    if (it == m->reqs.end()) return PA_ERR_INVALID_ARG;
    Request &r = it->second;
    const int bs = m->bs;
    const int full = num_computed_tokens / bs;
    if (full > (int)r.blocks.size()) return PA_ERR_INVALID_ARG;
    if (full <= r.num_cached) return PA_OK;
    if (!m->prefix_cache) {  // nothing is registered: no keys needed
        r.num_cached = full;
        return PA_OK;
    }
    // only the blocks that became full since the last call are hashed: the chain key of the
    // last counted block is kept with the request
    uint64_t parent = r.num_cached == 0 ? kFnvOffset : r.chain;
    for (int i = r.num_cached; i < full; ++i) {
        const int32_t *t = tokens + (size_t)i * bs;
        const uint64_t k = block_key(parent, t, bs);
        Block &x = m->blk[r.blocks[i]];
        if (!x.cached && !m->cache.count(k)) {
            x.cached = true;
            x.key = k;
            x.parent = parent;
            x.tokens.assign(t, t + bs);
            m->cache.emplace(k, r.blocks[i]);
        }
        parent = k;
    }
    r.num_cached = full;
    r.chain = parent;
    return PA_OK;
}

int pa_kvm_free(pa_kvm *m, int64_t req_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(req_id);
    if (it == m->reqs.end()) return PA_ERR_INVALID_ARG;
    const std::vector<int32_t> &bl = it->second.blocks;
    for (auto b = bl.rbegin(); b != bl.rend(); ++b) {
        Block &x = m->blk[*b];
        if (--x.ref == 0) m->push_back(*b);
    }
    m->reqs.erase(it);
    return PA_OK;
}

int pa_kvm_fork(pa_kvm *m, int64_t parent, int64_t child) {
    if (!m || parent == child) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(parent);
    if (it == m->reqs.end() || m->reqs.count(child)) return PA_ERR_INVALID_ARG;
    Request r = it->second;
    for (int32_t b : r.blocks) ++m->blk[b].ref;
    m->reqs.emplace(child, std::move(r));
    return PA_OK;
}

int pa_kvm_block_table(const pa_kvm *m, int64_t req_id, int32_t *out, int max_blocks, int *num_blocks) {
    if (!m || !num_blocks || max_blocks < 0) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(req_id);
    if (it == m->reqs.end()) return PA_ERR_INVALID_ARG;
    const std::vector<int32_t> &bl = it->second.blocks;
    if ((int)bl.size() > max_blocks || (!bl.empty() && !out)) return PA_ERR_WORKSPACE;
    for (size_t i = 0; i < bl.size(); ++i) out[i] = bl[i];
    *num_blocks = (int)bl.size();
    return PA_OK;
}

int pa_kvm_slot_mapping(const pa_kvm *m, int64_t req_id, int first_pos, int count, int64_t *slots) {
    if (!m || first_pos < 0 || count < 0 || (count > 0 && !slots)) return PA_ERR_INVALID_ARG;
    auto it = m->reqs.find(req_id);
    if (it == m->reqs.end()) return PA_ERR_INVALID_ARG;
    const std::vector<int32_t> &bl = it->second.blocks;
    const int bs = m->bs;
    if ((int64_t)first_pos + count > (int64_t)bl.size() * bs) return PA_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const int pos = first_pos + i;
        slots[i] = (int64_t)bl[pos / bs] * bs + pos % bs;
    }
    return PA_OK;
}

int pa_kvm_num_free_blocks(const pa_kvm *m) { return m ? m->num_free : PA_ERR_INVALID_ARG; }

int pa_kvm_stats(const pa_kvm *m, int64_t out[5]) {
    if (!m || !out) return PA_ERR_INVALID_ARG;
    out[0] = m->lookups;
    out[1] = m->looked_blocks;
    out[2] = m->hit_blocks;
    out[3] = (int64_t)m->cache.size();
    out[4] = m->evictions;
    return PA_OK;
}

}  // extern "C"
