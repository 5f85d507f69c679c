// pa_blocks.cpp -- host-side block manager and serving loop (include/pa_blocks.h).
//
// The block manager owns the pool's physical block ids: a free list kept as
// an intrusive doubly linked list (pop at the tail, release at the head, any
// cached block taken out in O(1) when a new request matches it), reference
// counts, per-sequence block tables and tokens, and -- with prefix caching --
// a map from block identity to the block holding it.
//
// A full block's identity is a pair of 64-bit chained hashes over (extra key,
// every token up to the block's end): each step folds the previous pair, the
// extra key and the block's own tokens through two independent 64-bit mixing
// functions (the splitmix64 finaliser of Steele, Lea and Flood, with
// different stream constants).  A match also compares the block's own tokens
// and extra key, so sharing the wrong block needs a collision of both chains
// and not just of one map bucket.
#include <algorithm>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "../../include/pa_blocks.h"

namespace {

inline uint64_t mix(uint64_t x) {
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    x ^= x >> 31;
    return x;
}

struct Ident {
    uint64_t a = 0, b = 0;
    bool operator==(const Ident &o) const { return a == o.a && b == o.b; }
};

struct IdentHash {
    size_t operator()(const Ident &k) const { return (size_t)(k.a ^ (k.b * 0x9e3779b97f4a7c15ull)); }
};

// identity of the next full block given the previous one (root: {0, 0})
Ident chain(const Ident &prev, int64_t extra, const int32_t *tok, int bs) {
    uint64_t a = mix(prev.a ^ 0x6a09e667f3bcc909ull) ^ mix((uint64_t)extra + 0x3c6ef372fe94f82bull);
    uint64_t b = mix(prev.b ^ 0xbb67ae8584caa73bull) ^ mix((uint64_t)extra * 0x9e3779b97f4a7c15ull + 1);
    for (int i = 0; i < bs; ++i) {
        const uint64_t t = (uint64_t)(uint32_t)tok[i];
        a = mix(a + t * 0xa54ff53a5f1d36f1ull + (uint64_t)i);
        b = mix(b ^ (t + 0x510e527fade682d1ull + ((uint64_t)i << 32)));
    }
    return Ident{a, b};
}

struct Seq {
    std::vector<int32_t> table;
    std::vector<int32_t> tokens;
    int64_t extra = 0;
    std::vector<Ident> ident;     // identity of each full block (prefix caching)
};

}  // namespace

struct pa_bm {
    int32_t nb = 0, bs = 16;
    bool pc = false;
    // free list: head = front (released blocks go here), tail = end (popped)
    std::vector<int32_t> prev, next;
    int32_t head = -1, tail = -1, nfree = 0;
    std::vector<uint8_t> on_free;
    std::vector<int32_t> ref;
    // committed identities
    std::vector<uint8_t> committed;
    std::vector<Ident> ident;
    std::vector<int64_t> bextra;
    std::vector<int32_t> btok;    // nb * bs
    std::unordered_map<Ident, int32_t, IdentHash> cached;
    std::unordered_map<int64_t, Seq> seqs;

    void unlink(int32_t b) {
        const int32_t p = prev[b], n = next[b];
        if (p >= 0) next[p] = n; else head = n;
        if (n >= 0) prev[n] = p; else tail = p;
        prev[b] = next[b] = -1;
        on_free[b] = 0;
        --nfree;
    }
    void push_front(int32_t b) {
        prev[b] = -1;
        next[b] = head;
        if (head >= 0) prev[head] = b; else tail = b;
        head = b;
        on_free[b] = 1;
        ++nfree;
    }
    void push_back(int32_t b) {
        next[b] = -1;
        prev[b] = tail;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        on_free[b] = 1;
        ++nfree;
    }
    int32_t pop() {                      // caller checked nfree > 0
        const int32_t b = tail;
        unlink(b);
        if (committed[b]) {              // evicted: its contents will be overwritten
            cached.erase(ident[b]);
            committed[b] = 0;
        }
        ref[b] = 1;
        return b;
    }
    void release(const std::vector<int32_t> &table) {
        for (size_t i = table.size(); i-- > 0;) {   // leaves before roots
            const int32_t b = table[i];
            if (--ref[b] == 0) push_front(b);
        }
    }
    // the block holding identity id with these own tokens and extra key, or -1
    int32_t match(const Ident &id, const int32_t *tok, int64_t extra) const {
        auto it = cached.find(id);
        if (it == cached.end()) return -1;
        const int32_t b = it->second;
        if (bextra[b] != extra) return -1;
        if (std::memcmp(&btok[(size_t)b * bs], tok, sizeof(int32_t) * bs) != 0) return -1;
        return b;
    }
    void commit(int32_t b, const Ident &id, const int32_t *tok, int64_t extra) {
        if (cached.count(id)) return;    // already cached elsewhere: b stays private
        cached.emplace(id, b);
        committed[b] = 1;
        ident[b] = id;
        bextra[b] = extra;
        std::memcpy(&btok[(size_t)b * bs], tok, sizeof(int32_t) * bs);
    }
    int64_t blocks_for(int64_t n) const { return (n + bs - 1) / bs; }
};

extern "C" {

pa_bm *pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order,
                    int32_t prefix_caching) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (!bm) return nullptr;
    try {
        bm->nb = num_blocks;
        bm->bs = block_size;
        bm->pc = prefix_caching != 0;
        bm->prev.assign(num_blocks, -1);
        bm->next.assign(num_blocks, -1);
        bm->on_free.assign(num_blocks, 0);
        bm->ref.assign(num_blocks, 0);
        bm->committed.assign(num_blocks, 0);
        bm->ident.assign(num_blocks, Ident{});
        bm->bextra.assign(num_blocks, 0);
        bm->btok.assign((size_t)num_blocks * block_size, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            const int32_t b = free_order ? free_order[i] : i;
            if (b < 0 || b >= num_blocks || bm->on_free[b]) {   // not a permutation
                delete bm;
                return nullptr;
            }
            bm->push_back(b);
        }
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

int32_t pa_bm_num_free(const pa_bm *bm) { return bm ? bm->nfree : 0; }

int32_t pa_bm_can_allocate(const pa_bm *bm, int64_t num_tokens) {
    if (!bm || num_tokens < 0) return 0;
    return bm->nfree >= bm->blocks_for(num_tokens) ? 1 : 0;
}

int pa_bm_add_sequence(pa_bm *bm, int64_t seq_id, const int32_t *tokens, int64_t n,
                       int64_t extra, int64_t *num_cached) {
    if (!bm || n < 0) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
    try {
        Seq s;
        s.extra = extra;
        s.tokens.assign((size_t)n, 0);
        if (tokens && n) std::memcpy(s.tokens.data(), tokens, sizeof(int32_t) * (size_t)n);
        const int bs = bm->bs;
        const int64_t nb = bm->blocks_for(n), full = n / bs;
        // identities of the full blocks, and the leading ones already cached
        std::vector<int32_t> hits;
        if (bm->pc) {
            Ident id;
            s.ident.reserve((size_t)full);
            for (int64_t i = 0; i < full; ++i) {
                id = chain(id, extra, &s.tokens[(size_t)i * bs], bs);
                s.ident.push_back(id);
            }
            for (int64_t i = 0; i < full; ++i) {
                const int32_t b = bm->match(s.ident[(size_t)i], &s.tokens[(size_t)i * bs], extra);
                if (b < 0) break;
                hits.push_back(b);
            }
        }
        int64_t revived = 0;
        for (int32_t b : hits) revived += bm->ref[b] == 0;
        if (bm->nfree - revived < nb - (int64_t)hits.size()) return PA_BM_FULL;
        s.table.reserve((size_t)nb);
        for (int32_t b : hits) {
            if (bm->ref[b] == 0) bm->unlink(b);
            ++bm->ref[b];
            s.table.push_back(b);
        }
        for (int64_t i = (int64_t)hits.size(); i < nb; ++i) {
            const int32_t b = bm->pop();
            s.table.push_back(b);
            if (bm->pc && i < full)
                bm->commit(b, s.ident[(size_t)i], &s.tokens[(size_t)i * bs], extra);
        }
        if (num_cached) *num_cached = (int64_t)hits.size() * bs;
        bm->seqs.emplace(seq_id, std::move(s));
    } catch (...) {
        return PA_ERR_INVALID_ARG;
    }
    return PA_OK;
}

int pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return PA_ERR_INVALID_ARG;
    try {
        Seq c = it->second;
        for (int32_t b : c.table) ++bm->ref[b];
        bm->seqs.emplace(child, std::move(c));
    } catch (...) {
        return PA_ERR_INVALID_ARG;
    }
    return PA_OK;
}

int pa_bm_append(pa_bm *bm, int64_t seq_id, int32_t token, int64_t *slot, int32_t *copy_src,
                 int32_t *copy_dst) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    Seq &s = it->second;
    const int bs = bm->bs;
    const int64_t pos = (int64_t)s.tokens.size();
    int32_t cs = -1, cd = -1;
    try {
        if (pos % bs == 0) {                         // the token starts a new block
            if (bm->nfree == 0) return PA_BM_FULL;
            s.table.push_back(bm->pop());
        } else {
            const int32_t last = s.table.back();
            if (bm->ref[last] > 1) {                 // shared: copy before writing
                if (bm->nfree == 0) return PA_BM_FULL;
                const int32_t fresh = bm->pop();
                --bm->ref[last];
                s.table.back() = fresh;
                cs = last;
                cd = fresh;
            }
        }
        s.tokens.push_back(token);
        const int64_t n = pos + 1;
        const int32_t blk = s.table[(size_t)(pos / bs)];
        if (bm->pc && n % bs == 0) {                 // the block is now full
            const int64_t i = n / bs - 1;
            const Ident prev = i > 0 ? s.ident[(size_t)(i - 1)] : Ident{};
            const Ident id = chain(prev, s.extra, &s.tokens[(size_t)i * bs], bs);
            s.ident.push_back(id);
            bm->commit(blk, id, &s.tokens[(size_t)i * bs], s.extra);
        }
        if (slot) *slot = (int64_t)blk * bs + pos % bs;
    } catch (...) {
        return PA_ERR_INVALID_ARG;
    }
    if (copy_src) *copy_src = cs;
    if (copy_dst) *copy_dst = cd;
    return PA_OK;
}

int pa_bm_free(pa_bm *bm, int64_t seq_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
    bm->release(it->second.table);
    bm->seqs.erase(it);
    return PA_OK;
}

int32_t pa_bm_table(const pa_bm *bm, int64_t seq_id, int32_t *out, int32_t cap) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return -1;
    const auto &t = it->second.table;
    if (out)
        for (int32_t i = 0; i < cap && i < (int32_t)t.size(); ++i) out[i] = t[(size_t)i];
    return (int32_t)t.size();
}

int64_t pa_bm_seq_len(const pa_bm *bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : (int64_t)it->second.tokens.size();
}

int32_t pa_bm_refcount(const pa_bm *bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->nb) return -1;
    return bm->ref[block];
}

int pa_bm_batch(const pa_bm *bm, const int64_t *seq_ids, int32_t n, int32_t *tables,
                int32_t width, int32_t pad, int32_t *seq_lens) {
    if (!bm || n < 0 || width < 0 || (n > 0 && (!seq_ids || !tables || !seq_lens)))
        return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
        const auto &t = it->second.table;
        if ((int64_t)t.size() > width) return PA_ERR_INVALID_ARG;
        int32_t *row = tables + (size_t)i * width;
        for (int32_t j = 0; j < width; ++j) row[j] = j < (int32_t)t.size() ? t[(size_t)j] : pad;
        seq_lens[i] = (int32_t)it->second.tokens.size();
    }
    return PA_OK;
}

int32_t pa_bm_common_prefix(const pa_bm *bm, const int64_t *seq_ids, int32_t n) {
    if (!bm || n < 0 || (n > 0 && !seq_ids)) return PA_ERR_INVALID_ARG;
    if (n == 0) return 0;
    const std::vector<int32_t> *first = nullptr;
    size_t common = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PA_ERR_INVALID_ARG;
        const auto &t = it->second.table;
        const size_t full = it->second.tokens.size() / (size_t)bm->bs;
        if (!first) {
            first = &t;
            common = full < t.size() ? full : t.size();
            continue;
        }
        size_t k = 0;
        const size_t lim = common < full ? common : full;
        while (k < lim && k < t.size() && t[k] == (*first)[k]) ++k;
        common = k;
    }
    return (int32_t)common;
}

}  // extern "C"

// ---- serving loop ---------------------------------------------------------

namespace {

struct Req {
    int64_t id, tokens, left;
};

}  // namespace

struct pa_loop {
    pa_bm *bm = nullptr;
    std::deque<Req> queue;
    std::vector<Req> running;             // admission order
    int64_t step = 0;
};

extern "C" {

pa_loop *pa_loop_create(pa_bm *bm) {
    if (!bm) return nullptr;
    pa_loop *l = new (std::nothrow) pa_loop();
    if (l) l->bm = bm;
    return l;
}

void pa_loop_destroy(pa_loop *loop) { delete loop; }

int pa_loop_submit(pa_loop *loop, int64_t id, int64_t tokens, int64_t max_new) {
    if (!loop || tokens < 0 || max_new <= 0) return PA_ERR_INVALID_ARG;
    try {
        loop->queue.push_back(Req{id, tokens, max_new});
    } catch (...) {
        return PA_ERR_INVALID_ARG;
    }
    return PA_OK;
}

int pa_loop_step(pa_loop *loop, int64_t *events, int32_t events_cap, int32_t *num_events,
                 int64_t *written, int32_t written_cap, int32_t *num_written, int64_t *step) {
    if (!loop || !num_events || !num_written) return PA_ERR_INVALID_ARG;
    pa_bm *bm = loop->bm;
    int32_t ne = 0, nw = 0;
    bool overflow = false;
    auto event = [&](int kind, const Req &r) {
        if (ne < events_cap && events) {
            int64_t *e = events + (size_t)ne * 5;
            e[0] = loop->step; e[1] = kind; e[2] = r.id; e[3] = r.tokens;
            e[4] = pa_bm_num_free(bm);
        } else {
            overflow = true;
        }
        ++ne;
    };
    // admit while the first queued request fits
    while (!loop->queue.empty() && pa_bm_can_allocate(bm, loop->queue.front().tokens)) {
        Req r = loop->queue.front();
        loop->queue.pop_front();
        if (pa_bm_add_sequence(bm, r.id, nullptr, r.tokens, 0, nullptr) != PA_OK)
            return PA_ERR_INVALID_ARG;                 // duplicate id
        loop->running.push_back(r);
        event(PA_EV_ADMIT, r);
    }
    if (loop->queue.empty() && loop->running.empty()) {
        *num_events = ne;
        *num_written = 0;
        if (step) *step = loop->step;
        return overflow ? PA_ERR_INVALID_ARG : 0;
    }
    if (loop->running.empty()) {
        // the first queued request does not fit even in an empty pool
        *num_events = ne;
        *num_written = 0;
        if (step) *step = loop->step;
        return PA_ERR_INVALID_ARG;
    }
    ++loop->step;
    // one token per running request, in admission order
    std::vector<int64_t> order;
    order.reserve(loop->running.size());
    for (const Req &r : loop->running) order.push_back(r.id);
    auto find = [&](int64_t id) -> int64_t {
        for (size_t i = 0; i < loop->running.size(); ++i)
            if (loop->running[i].id == id) return (int64_t)i;
        return -1;
    };
    for (int64_t id : order) {
        if (find(id) < 0) continue;                    // preempted earlier in this step
        int64_t slot = -1;
        bool gone = false;
        for (;;) {
            const int rc = pa_bm_append(bm, id, 0, &slot, nullptr, nullptr);
            if (rc == PA_OK) break;
            if (rc != PA_BM_FULL) return rc;
            // no block for the next token: preempt the newest running request
            Req victim = loop->running.back();
            loop->running.pop_back();
            pa_bm_free(bm, victim.id);
            loop->queue.push_front(victim);
            event(PA_EV_PREEMPT, victim);
            if (victim.id == id) { gone = true; break; }
        }
        if (gone) continue;
        const int64_t i = find(id);
        Req &r = loop->running[(size_t)i];
        r.tokens += 1;
        r.left -= 1;
        if (nw < written_cap && written) {
            written[(size_t)nw * 2] = id;
            written[(size_t)nw * 2 + 1] = slot;
        } else {
            overflow = true;
        }
        ++nw;
        if (r.left == 0) {
            const Req done = r;
            loop->running.erase(loop->running.begin() + i);
            pa_bm_free(bm, id);
            event(PA_EV_FINISH, done);
        }
    }
    *num_events = ne;
    *num_written = nw;
    if (step) *step = loop->step;
    if (overflow) return PA_ERR_INVALID_ARG;
    return (loop->queue.empty() && loop->running.empty()) ? 0 : 1;
}

}  // extern "C"
