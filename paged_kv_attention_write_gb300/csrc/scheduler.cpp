// scheduler.cpp -- host step scheduler over the KV-cache manager: alternating prefill and
// decode batches under a token budget with chunked prompts (the Pure-Rust engines page,
// scheduling section, describes the policy for mistral.rs).  The exact policy is stated in
// include/pa_scheduler.h.
#include <algorithm>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "kv_manager_impl.h"
#include "pa_scheduler.h"

namespace {

struct SReq {
    std::vector<int32_t> tokens;  // prompt, then generated tokens
    int prompt_len = 0;           // tokens to prefill (grows to all tokens after a preemption)
    int computed = 0;             // tokens whose K/V are in the cache
    int max_new = 0, generated = 0;
};

struct Entry {
    int64_t rid;
    int start, count;  // query positions start .. start + count - 1
};

void erase_value(std::vector<int64_t> &v, int64_t x) {
    auto it = std::find(v.begin(), v.end(), x);
    if (it != v.end()) v.erase(it);
}

}  // namespace

struct pa_sched {
    pa_kvm *kv = nullptr;
    int bs, budget, chunk, max_decode;
    std::unordered_map<int64_t, SReq> req;
    std::deque<int64_t> waiting;
    std::vector<int64_t> prefilling, running;
    int decode_streak = 0;
    int last_kind = PA_SCHED_IDLE;
    bool planned = false;
    std::vector<Entry> last;
    std::vector<int64_t> pairs;
    int max_blocks_per_req = 1;
    int64_t prefill_steps = 0, decode_steps = 0, prefill_tokens = 0, generated = 0, finished = 0,
            preemptions = 0;

    // (hit tokens, chunk) when waiting request rid's first chunk fits the free blocks not
    // taken by its own prefix-cache hits; changes nothing (the lookup is not counted).
    bool admissible(int64_t rid, int left, int *got, int *n) {
        SReq &r = req[rid];
        std::vector<int32_t> hits;
        kv->lookup(r.tokens.data(), (int)r.tokens.size(), hits, nullptr, false);
        *got = (int)hits.size() * bs;
        *n = std::min(chunk, std::min((int)r.tokens.size() - *got, left));
        const int need = (*got + *n + bs - 1) / bs - (int)hits.size();
        int free_hits = 0;
        for (int32_t b : hits) free_hits += kv->blk[b].ref == 0;
        return need <= kv->num_free - free_hits;
    }
    bool alloc(int64_t rid, int num_tokens) {
        int64_t p[2];
        int np = 0;
        if (pa_kvm_allocate_slots(kv, rid, num_tokens, p, 1, &np) != PA_OK) return false;
        if (np) pairs.insert(pairs.end(), p, p + 2);
        return true;
    }
    void prefill_batch() {
        int left = budget;
        for (int64_t rid : std::vector<int64_t>(prefilling)) {
            if (left == 0) break;
            if (std::find(prefilling.begin(), prefilling.end(), rid) == prefilling.end()) continue;
            SReq &r = req[rid];
            const int n = std::min(chunk, std::min(r.prompt_len - r.computed, left));
            bool ok = true;
            while (!alloc(rid, r.computed + n)) {  // the most recently admitted prompt makes room
                const int64_t victim = prefilling.back();
                prefilling.pop_back();
                preempt(victim);
                if (victim == rid) {
                    ok = false;
                    break;
                }
            }
            if (!ok) continue;
            last.push_back({rid, r.computed, n});
            left -= n;
        }
        while (!waiting.empty() && left > 0) {
            const int64_t rid = waiting.front();
            int got = 0, n = 0;
            if (!admissible(rid, left, &got, &n)) break;
            SReq &r = req[rid];
            int got2 = 0;
            pa_kvm_admit(kv, rid, r.tokens.data(), (int)r.tokens.size(), &got2);
            alloc(rid, got + n);  // fits: checked above
            waiting.pop_front();
            r.computed = got;
            r.prompt_len = (int)r.tokens.size();
            prefilling.push_back(rid);
            last.push_back({rid, got, n});
            left -= n;
        }
    }
    void preempt(int64_t rid) {
        SReq &r = req[rid];
        pa_kvm_free(kv, rid);
        r.computed = 0;
        r.prompt_len = (int)r.tokens.size();
        waiting.push_front(rid);
        ++preemptions;
    }
    void decode_batch() {
        size_t i = 0;
        while (i < running.size()) {
            const int64_t rid = running[i];
            if (alloc(rid, (int)req[rid].tokens.size())) {
                ++i;
            } else {  // the most recently admitted request makes room
                const int64_t victim = running.back();
                running.pop_back();
                preempt(victim);
            }
        }
        for (int64_t rid : running) last.push_back({rid, (int)req[rid].tokens.size() - 1, 1});
    }
    int64_t in_flight() const { return (int64_t)req.size(); }
};

extern "C" {

int pa_sched_create(int num_blocks, int block_size, int token_budget, int chunk_tokens,
                    int max_decode_steps, int enable_prefix_cache, pa_sched **out) {
    if (!out || token_budget <= 0 || chunk_tokens <= 0 || max_decode_steps <= 0) return PA_ERR_INVALID_ARG;
    pa_sched *s = new (std::nothrow) pa_sched();
    if (!s) return PA_ERR_INVALID_ARG;
    const int rc = pa_kvm_create(num_blocks, block_size, enable_prefix_cache, &s->kv);
    if (rc != PA_OK) {
        delete s;
        return rc;
    }
    s->bs = block_size;
    s->budget = token_budget;
    s->chunk = chunk_tokens;
    s->max_decode = max_decode_steps;
    *out = s;
    return PA_OK;
}

void pa_sched_destroy(pa_sched *s) {
    if (!s) return;
    pa_kvm_destroy(s->kv);
    delete s;
}

int pa_sched_add_request(pa_sched *s, int64_t req_id, const int32_t *prompt, int prompt_len,
                         int max_new_tokens) {
    if (!s || !prompt || prompt_len <= 0 || max_new_tokens <= 0 || s->req.count(req_id)) return PA_ERR_INVALID_ARG;
    if (((int64_t)prompt_len + max_new_tokens + s->bs - 1) / s->bs > s->kv->num_blocks)
        return PA_ERR_INVALID_ARG;  // could never fit the pool
    SReq r;
    r.tokens.assign(prompt, prompt + prompt_len);
    r.prompt_len = prompt_len;
    r.max_new = max_new_tokens;
    s->req.emplace(req_id, std::move(r));
    s->waiting.push_back(req_id);
    s->max_blocks_per_req = std::max(s->max_blocks_per_req, (prompt_len + max_new_tokens + s->bs - 1) / s->bs);
    return PA_OK;
}

int pa_sched_capacity(const pa_sched *s, int out[4]) {
    if (!s || !out) return PA_ERR_INVALID_ARG;
    const int n = (int)std::max<int64_t>(1, s->in_flight());
    out[0] = n;
    out[1] = std::max(s->budget, n);
    out[2] = s->max_blocks_per_req;
    out[3] = n;
    return PA_OK;
}

}  // extern "C"

namespace {

// Plans the next step (sets the batch entries, the copy pairs and the kind).
void plan_step(pa_sched *s) {
    s->last.clear();
    s->pairs.clear();
    s->last_kind = PA_SCHED_IDLE;
    const bool pending = !s->prefilling.empty() || !s->waiting.empty();
    if (pending && (s->running.empty() || s->decode_streak >= s->max_decode)) {
        s->prefill_batch();
        if (!s->last.empty()) s->last_kind = PA_SCHED_PREFILL;
    }
    if (s->last_kind == PA_SCHED_IDLE && !s->running.empty()) {
        s->decode_batch();
        s->last_kind = PA_SCHED_DECODE;
    }
}

// Sizes of the planned batch.
void describe(const pa_sched *s, pa_sched_batch *b) {
    int width = 1, tokens = 0, max_q = 0, max_c = 0;
    for (const Entry &e : s->last) {
        const auto &bl = s->kv->reqs.at(e.rid).blocks;
        width = std::max(width, (int)bl.size());
        max_q = std::max(max_q, e.count);
        max_c = std::max(max_c, e.start + e.count);
        tokens += e.count;
    }
    b->kind = s->last_kind;
    b->num_seqs = (int)s->last.size();
    b->num_tokens = tokens;
    b->max_query_len = max_q;
    b->max_context_len = max_c;
    b->table_width = width;
    b->num_copy_pairs = (int)s->pairs.size() / 2;
}

// Writes the planned batch's arrays (block-table rows table_width entries apart).
void write_batch(const pa_sched *s, int table_width, int64_t *req_ids, int32_t *query_start_loc,
                 int32_t *context_lens, int32_t *block_tables, int32_t *token_ids, int32_t *positions,
                 int64_t *slot_mapping, int64_t *copy_pairs) {
    int tokens = 0;
    query_start_loc[0] = 0;
    for (size_t i = 0; i < s->last.size(); ++i) {
        const Entry &e = s->last[i];
        const auto &bl = s->kv->reqs.at(e.rid).blocks;
        const SReq &r = s->req.at(e.rid);
        req_ids[i] = e.rid;
        context_lens[i] = e.start + e.count;
        int32_t *row = block_tables + i * (size_t)table_width;
        for (int j = 0; j < table_width; ++j) row[j] = j < (int)bl.size() ? bl[j] : 0;
        for (int p = e.start; p < e.start + e.count; ++p, ++tokens) {
            token_ids[tokens] = r.tokens[p];
            positions[tokens] = p;
            slot_mapping[tokens] = (int64_t)bl[p / s->bs] * s->bs + p % s->bs;
        }
        query_start_loc[i + 1] = tokens;
    }
    for (size_t i = 0; i < s->pairs.size(); ++i) copy_pairs[i] = s->pairs[i];
}

int64_t round16(int64_t x) { return (x + 15) & ~int64_t(15); }

// Byte layout of a packed step with S sequences, T tokens, table rows of W entries and P
// copy pairs (the device span first).
pa_sched_offsets packed_layout(int64_t S, int64_t T, int64_t W, int64_t P) {
    pa_sched_offsets o{};
    int64_t at = 0;
    o.query_start_loc = at; at += round16(4 * (S + 1));
    o.context_lens = at;    at += round16(4 * S);
    o.block_tables = at;    at += round16(4 * S * W);
    o.slot_mapping = at;    at += round16(8 * T);
    o.copy_pairs = at;      at += round16(16 * P);
    o.token_ids = at;       at += round16(4 * T);
    o.positions = at;       at += round16(4 * T);
    o.dev_bytes = at;
    o.req_ids = at;         at += round16(8 * S);
    o.total_bytes = at;
    return o;
}

}  // namespace

extern "C" {

int pa_sched_step(pa_sched *s, pa_sched_batch *b, int64_t *req_ids, int32_t *query_start_loc,
                  int32_t *context_lens, int32_t *block_tables, int table_capacity,
                  int32_t *token_ids, int32_t *positions, int64_t *slot_mapping, int64_t *copy_pairs,
                  int max_seqs, int max_tokens, int max_pairs) {
    if (!s || !b || s->planned) return PA_ERR_INVALID_ARG;
    int cap[4];
    pa_sched_capacity(s, cap);
    if (max_seqs < cap[0] || max_tokens < cap[1] || table_capacity < cap[2] || max_pairs < cap[3])
        return PA_ERR_WORKSPACE;
    if (!req_ids || !query_start_loc || !context_lens || !block_tables || !token_ids || !positions ||
        !slot_mapping || !copy_pairs)
        return PA_ERR_INVALID_ARG;
    plan_step(s);
    describe(s, b);
    write_batch(s, b->table_width, req_ids, query_start_loc, context_lens, block_tables, token_ids, positions,
                slot_mapping, copy_pairs);
    s->planned = true;
    return PA_OK;
}

int64_t pa_sched_packed_bytes(const pa_sched *s) {
    int cap[4];
    if (pa_sched_capacity(s, cap) != PA_OK) return 0;
    return packed_layout(cap[0], cap[1], cap[2], cap[3]).total_bytes;
}

int pa_sched_step_packed(pa_sched *s, pa_sched_batch *b, void *buf, int64_t buf_bytes, pa_sched_offsets *offsets) {
    if (!s || !b || !buf || !offsets || s->planned || (reinterpret_cast<uintptr_t>(buf) & 15))
        return PA_ERR_INVALID_ARG;
    if (buf_bytes < pa_sched_packed_bytes(s)) return PA_ERR_WORKSPACE;
    plan_step(s);
    describe(s, b);
    const pa_sched_offsets o = packed_layout(b->num_seqs, b->num_tokens, b->table_width, b->num_copy_pairs);
    char *base = static_cast<char *>(buf);
    write_batch(s, b->table_width, reinterpret_cast<int64_t *>(base + o.req_ids),
                reinterpret_cast<int32_t *>(base + o.query_start_loc), reinterpret_cast<int32_t *>(base + o.context_lens),
                reinterpret_cast<int32_t *>(base + o.block_tables), reinterpret_cast<int32_t *>(base + o.token_ids),
                reinterpret_cast<int32_t *>(base + o.positions), reinterpret_cast<int64_t *>(base + o.slot_mapping),
                reinterpret_cast<int64_t *>(base + o.copy_pairs));
    *offsets = o;
    s->planned = true;
    return PA_OK;
}

int pa_sched_complete(pa_sched *s, const int32_t *sampled, int num_sampled, int64_t *finished,
                      int max_finished, int *num_finished) {
    if (!s || !s->planned || !num_finished || num_sampled != (int)s->last.size() ||
        (num_sampled > 0 && !sampled))
        return PA_ERR_INVALID_ARG;
    if (max_finished < num_sampled || (num_sampled > 0 && !finished)) return PA_ERR_WORKSPACE;
    if (s->last_kind == PA_SCHED_PREFILL) {
        ++s->prefill_steps;
        s->decode_streak = 0;
    } else if (s->last_kind == PA_SCHED_DECODE) {
        ++s->decode_steps;
        ++s->decode_streak;
    }
    int nf = 0;
    for (size_t i = 0; i < s->last.size(); ++i) {
        const Entry &e = s->last[i];
        SReq &r = s->req.at(e.rid);
        const int done = e.start + e.count;
        r.computed = done;
        pa_kvm_cache_blocks(s->kv, e.rid, r.tokens.data(), done);
        if (s->last_kind == PA_SCHED_PREFILL) {
            s->prefill_tokens += e.count;
            if (done < r.prompt_len) continue;
            erase_value(s->prefilling, e.rid);
            s->running.push_back(e.rid);
        }
        r.tokens.push_back(sampled[i]);
        ++r.generated;
        ++s->generated;
        if (r.generated >= r.max_new) {
            erase_value(s->running, e.rid);
            pa_kvm_free(s->kv, e.rid);
            s->req.erase(e.rid);
            ++s->finished;
            finished[nf++] = e.rid;
        }
    }
    *num_finished = nf;
    s->last.clear();
    s->planned = false;
    return PA_OK;
}

int pa_sched_stats(const pa_sched *s, int64_t out[7]) {
    if (!s || !out) return PA_ERR_INVALID_ARG;
    out[0] = s->prefill_steps;
    out[1] = s->decode_steps;
    out[2] = s->prefill_tokens;
    out[3] = s->generated;
    out[4] = s->finished;
    out[5] = s->preemptions;
    out[6] = s->in_flight();
    return PA_OK;
}

pa_kvm *pa_sched_manager(pa_sched *s) { return s ? s->kv : nullptr; }

}  // extern "C"
