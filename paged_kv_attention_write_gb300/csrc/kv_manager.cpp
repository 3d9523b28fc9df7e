// kv_manager.cpp -- host block pool and KV-cache manager (prefix caching, LRU free queue,
// copy-on-write for forked requests).  The policy is stated in include/pa_kv_manager.h;
// the operations follow the Pure-Rust engines page (paged-attention block management and
// prefix-cache sections) and the TensorSharp "Mistral 3" page, section 11.
//
// Data layout (kv_manager_impl.h): one record per physical block (reference count, free-queue links, prefix
// key and, while cached, the block's tokens and its parent's key), an intrusive doubly
// linked free queue (O(1) removal when a lookup revives a free cached block), a hash map
// from prefix key to block, and a map from request id to its block table.
#include "kv_manager_impl.h"

using pa_kvm_impl::block_key;
using pa_kvm_impl::kFnvOffset;
using pa_kvm_impl::Block;
using pa_kvm_impl::Request;

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
