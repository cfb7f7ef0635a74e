// Prefix-state cache with second-hit admission (host only, no device code).
//
// "vLLM Kimi K3 지원", section "하이브리드 KV-Cache 관리": the KDA state blocks
// are kept apart from prefix matching, so a prompt sharing a prefix resumes
// from the state saved at that prefix; section "에이전틱 캐시 유지 정책":
// Marconi-style selective retention saves a prefix's state only on the
// prefix's second hit.
//
// A prefix is the first i * block tokens of a prompt.  Each plan counts a hit
// on every block prefix of its prompt, reuses the longest saved prefix that
// leaves at least one token to compute, and admits at most one longer prefix
// with two or more hits into a slot of the cache's own list (lowest free
// first; when full, the least recently counted saved prefix other than the
// reused one gives its slot up and stays tracked, unsaved).  Unsaved prefixes
// beyond max_tracked are dropped least recently counted first.
//
// Prefixes are found by a 64-bit chained hash of their blocks; a saved
// prefix also keeps its tokens, so a hash collision can never resume a
// prompt from another prompt's state (it only merges two hit counts).

#include <cstdint>
#include <cstring>
#include <iterator>
#include <list>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "kda.h"

namespace {

struct Entry {
    int32_t hits = 0;
    int32_t slot = -1;  // -1: tracked, not saved
    uint64_t stamp = 0;  // the count clock at its last count
    std::list<uint64_t>::iterator pos;  // its node in the saved or the unsaved recency list
    std::vector<int32_t> tokens;        // the prefix, while saved
};

// splitmix64's output function (Steele, Lea, Flood: "Fast splittable
// pseudorandom number generators", OOPSLA 2014)
inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

}  // namespace

// Recency: each prefix key sits in one of two lists (saved, unsaved), least
// recently counted first; counting a prefix splices its node to the back, so
// the order is the order of the last counts and no touch allocates.
struct kda_prefix_cache {
    int32_t block = 0, max_tracked = 0;
    std::set<int32_t> free_slots;
    std::unordered_map<uint64_t, Entry> map;
    std::list<uint64_t> unsaved, saved;
    uint64_t clock = 0;
    kda_prefix_cache_stats stats{};

    // Moves entry e (key k) from one list to the other, at its place by last
    // count (a scan from the back; admissions, evictions and forgets only).
    void move_entry(Entry &e, std::list<uint64_t> &from, std::list<uint64_t> &to) {
        auto at = to.end();
        while (at != to.begin()) {
            auto prev = std::prev(at);
            if (map.at(*prev).stamp < e.stamp) break;
            at = prev;
        }
        to.splice(at, from, e.pos);
    }

    // keys[i] = hash of the first i blocks, i = 1 .. n / block.  A block's
    // tokens go through four independent mixing chains (token t into chain
    // t % 4; block is a multiple of 64), folded into the running hash at the
    // block's end: four times the instruction-level parallelism of one chain.
    void keys_of(const int32_t *tok, int32_t n, std::vector<uint64_t> &keys) const {
        const int32_t nb = n / block;
        keys.assign(size_t(nb) + 1, 0);
        uint64_t h = 0x6a09e667f3bcc909ull;
        for (int32_t i = 1; i <= nb; ++i) {
            uint64_t a0 = h, a1 = h ^ 0xbb67ae8584caa73bull, a2 = h ^ 0x3c6ef372fe94f82bull, a3 = h ^ 0xa54ff53a5f1d36f1ull;
            const int32_t *b = tok + size_t(i - 1) * size_t(block);
            for (int32_t t = 0; t < block; t += 4) {
                a0 = mix64(a0 ^ uint64_t(uint32_t(b[t])));
                a1 = mix64(a1 ^ uint64_t(uint32_t(b[t + 1])));
                a2 = mix64(a2 ^ uint64_t(uint32_t(b[t + 2])));
                a3 = mix64(a3 ^ uint64_t(uint32_t(b[t + 3])));
            }
            h = mix64(a0 ^ ((a1 << 16) | (a1 >> 48)) ^ ((a2 << 32) | (a2 >> 32)) ^ ((a3 << 48) | (a3 >> 16)));
            keys[size_t(i)] = mix64(h + uint64_t(i));
        }
    }
    std::list<uint64_t> &list_of(const Entry &e) { return e.slot >= 0 ? saved : unsaved; }

    void plan(const int32_t *tok, int32_t n, kda_prefix_plan *out) {
        const int32_t B = block, nb = n / B, cap = n > 0 ? (n - 1) / B : 0;
        std::vector<uint64_t> keys;
        keys_of(tok, n, keys);
        int32_t hit = 0;
        for (int32_t i = cap; i >= 1; --i) {
            auto it = map.find(keys[size_t(i)]);
            if (it != map.end() && it->second.slot >= 0 && it->second.tokens.size() == size_t(i) * size_t(B) &&
                std::memcmp(it->second.tokens.data(), tok, sizeof(int32_t) * size_t(i) * size_t(B)) == 0) {
                hit = i;
                break;
            }
        }
        for (int32_t i = 1; i <= nb; ++i) {
            const uint64_t k = keys[size_t(i)];
            auto ins = map.try_emplace(k);
            Entry &e = ins.first->second;
            std::list<uint64_t> &l = list_of(e);
            if (ins.second) {
                e.pos = l.insert(l.end(), k);
            } else {
                l.splice(l.end(), l, e.pos);
            }
            e.hits += 1;
            e.stamp = ++clock;
        }
        int32_t admit = 0, slot = -1;
        for (int32_t i = nb; i > hit; --i) {
            const Entry &e = map.at(keys[size_t(i)]);
            if (e.hits >= 2 && e.slot < 0) {
                admit = i;
                break;
            }
        }
        if (admit) {
            if (!free_slots.empty()) {
                slot = *free_slots.begin();
                free_slots.erase(free_slots.begin());
            } else {
                const uint64_t keep = hit ? keys[size_t(hit)] : 0;
                for (auto it = saved.begin(); it != saved.end(); ++it) {
                    if (hit && *it == keep) continue;
                    Entry &v = map.at(*it);
                    slot = v.slot;
                    v.slot = -1;
                    std::vector<int32_t>().swap(v.tokens);
                    move_entry(v, saved, unsaved);
                    stats.evictions += 1;
                    break;
                }
            }
            if (slot >= 0) {
                Entry &e = map.at(keys[size_t(admit)]);
                e.tokens.assign(tok, tok + size_t(admit) * size_t(B));
                e.slot = slot;
                move_entry(e, unsaved, saved);
                stats.admissions += 1;
            } else {
                admit = 0;
            }
        }
        while (unsaved.size() > size_t(max_tracked)) {
            map.erase(unsaved.front());
            unsaved.pop_front();
        }
        stats.plans += 1;
        if (hit) stats.hits += 1;
        out->hit_len = hit * B;
        out->hit_slot = hit ? map.at(keys[size_t(hit)]).slot : -1;
        out->admit_pos = admit ? admit * B : -1;
        out->admit_slot = admit ? slot : -1;
    }
};

extern "C" {

kda_status kda_prefix_cache_create(int32_t block, const int32_t *slots, int32_t n_slots, int32_t max_tracked,
                                   kda_prefix_cache **out) {
    if (!out) return KDA_ERR_INVALID_ARG;
    *out = nullptr;
    if (block <= 0 || block % 64 != 0 || n_slots < 0 || max_tracked < 0 || (n_slots > 0 && !slots))
        return KDA_ERR_INVALID_ARG;
    try {
        auto *c = new kda_prefix_cache;
        c->block = block;
        c->max_tracked = max_tracked;
        for (int32_t i = 0; i < n_slots; ++i) {
            if (slots[i] < 0 || !c->free_slots.insert(slots[i]).second) {
                const kda_status st = slots[i] < 0 ? KDA_ERR_SLOT_RANGE : KDA_ERR_ALIAS;
                delete c;
                return st;
            }
        }
        *out = c;
        return KDA_OK;
    } catch (const std::bad_alloc &) {
        return KDA_ERR_HOST_MEMORY;
    }
}

void kda_prefix_cache_destroy(kda_prefix_cache *cache) { delete cache; }

kda_status kda_prefix_cache_plan(kda_prefix_cache *cache, const int32_t *tokens, int32_t n, kda_prefix_plan *out) {
    if (!cache || !out || n < 0 || (n > 0 && !tokens)) return KDA_ERR_INVALID_ARG;
    try {
        cache->plan(tokens, n, out);
        return KDA_OK;
    } catch (const std::bad_alloc &) {
        return KDA_ERR_HOST_MEMORY;
    }
}

kda_status kda_prefix_cache_forget(kda_prefix_cache *cache, int32_t slot) {
    if (!cache) return KDA_ERR_INVALID_ARG;
    for (auto it = cache->saved.begin(); it != cache->saved.end(); ++it) {
        Entry &e = cache->map.at(*it);
        if (e.slot != slot) continue;
        try {
            cache->free_slots.insert(slot);
        } catch (const std::bad_alloc &) {
            return KDA_ERR_HOST_MEMORY;
        }
        e.slot = -1;
        std::vector<int32_t>().swap(e.tokens);
        cache->move_entry(e, cache->saved, cache->unsaved);
        return KDA_OK;  // the tracked bound applies again at the next plan
    }
    return KDA_ERR_INVALID_ARG;
}

kda_status kda_prefix_cache_get_stats(const kda_prefix_cache *cache, kda_prefix_cache_stats *out) {
    if (!cache || !out) return KDA_ERR_INVALID_ARG;
    *out = cache->stats;
    out->n_saved = int64_t(cache->saved.size());
    out->n_unsaved = int64_t(cache->unsaved.size());
    out->n_free = int64_t(cache->free_slots.size());
    return KDA_OK;
}

int32_t kda_prefix_cache_saved(const kda_prefix_cache *cache, int32_t *lens, int32_t *slots, int32_t cap) {
    if (!cache || cap < 0 || (cap > 0 && (!lens || !slots))) return -1;
    int32_t n = 0;
    for (const uint64_t k : cache->saved) {
        const Entry &e = cache->map.at(k);
        if (n < cap) {
            lens[n] = int32_t(e.tokens.size());
            slots[n] = e.slot;
        }
        ++n;
    }
    return n;
}

}  // extern "C"
