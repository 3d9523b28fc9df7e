// kv_manager_impl.h -- internal data structures of the host KV-cache manager, shared by
// kv_manager.cpp (the pa_kvm_* C ABI) and scheduler.cpp (which drives the manager and needs
// lookups that do not count and the blocks' reference counts).  Not part of the ABI.
#pragma once

#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_kv_manager.h"

namespace pa_kvm_impl {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;  // FNV-1a 64-bit parameters
constexpr uint64_t kFnvPrime = 1099511628211ull;

inline uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) {
        h ^= (v >> (8 * i)) & 0xffu;
        h *= kFnvPrime;
    }
    return h;
}

// Key of a full block: FNV-1a over the parent's key and the block's tokens (little-endian
// bytes, independent of the host's byte order).
inline uint64_t block_key(uint64_t parent, const int32_t *tok, int bs) {
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

}  // namespace pa_kvm_impl

struct pa_kvm {
    using Block = pa_kvm_impl::Block;
    using Request = pa_kvm_impl::Request;
    static constexpr uint64_t kFnvOffset = pa_kvm_impl::kFnvOffset;
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
    void lookup(const int32_t *tokens, int n, std::vector<int32_t> &hits, uint64_t *chain_out = nullptr,
                bool count = true) {
        hits.clear();
        if (count) ++lookups;
        if (chain_out) *chain_out = kFnvOffset;
        if (!prefix_cache || n <= 1) return;
        const int nb = (n - 1) / bs;
        if (count) looked_blocks += nb;
        uint64_t parent = kFnvOffset;
        for (int i = 0; i < nb; ++i) {
            const int32_t *t = tokens + (size_t)i * bs;
            const uint64_t k = pa_kvm_impl::block_key(parent, t, bs);
            auto it = cache.find(k);
            if (it == cache.end()) break;
            const Block &x = blk[it->second];
            if (!x.cached || x.parent != parent || std::memcmp(x.tokens.data(), t, sizeof(int32_t) * bs) != 0)
                break;
            hits.push_back(it->second);
            parent = k;
        }
        if (chain_out) *chain_out = parent;
        if (count) hit_blocks += (int64_t)hits.size();
    }
};

