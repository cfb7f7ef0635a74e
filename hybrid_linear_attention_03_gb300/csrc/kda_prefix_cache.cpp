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
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "kda.h"

namespace {

struct Entry {
    int32_t hits = 0;
    int32_t slot = -1;  // -1: tracked, not saved
    uint64_t stamp = 0;
    std::vector<int32_t> tokens;  // the prefix, while saved
};

// splitmix64's output function (Steele, Lea, Flood: "Fast splittable
// pseudorandom number generators", OOPSLA 2014)
inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

}  // namespace

struct kda_prefix_cache {
    int32_t block = 0, max_tracked = 0;
    std::set<int32_t> free_slots;
    std::unordered_map<uint64_t, Entry> map;
    std::set<std::pair<uint64_t, uint64_t>> unsaved, saved;  // (stamp, key), oldest first
    uint64_t clock = 0;
    kda_prefix_cache_stats stats{};

    // keys[i] = hash of the first i blocks, i = 1 .. n / block
    void keys_of(const int32_t *tok, int32_t n, std::vector<uint64_t> &keys) const {
        const int32_t nb = n / block;
        keys.assign(size_t(nb) + 1, 0);
        uint64_t h = 0x6a09e667f3bcc909ull;
        for (int32_t i = 1; i <= nb; ++i) {
            for (int32_t t = (i - 1) * block; t < i * block; ++t) h = mix64(h ^ uint64_t(uint32_t(tok[t])));
            keys[size_t(i)] = mix64(h + uint64_t(i));
        }
    }
    std::set<std::pair<uint64_t, uint64_t>> &set_of(const Entry &e) { return e.slot >= 0 ? saved : unsaved; }

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
            if (!ins.second) set_of(e).erase({e.stamp, k});
            e.hits += 1;
            e.stamp = ++clock;
            set_of(e).insert({e.stamp, k});
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
                    if (hit && it->second == keep) continue;
                    Entry &v = map.at(it->second);
                    slot = v.slot;
                    const std::pair<uint64_t, uint64_t> sk = *it;
                    saved.erase(it);
                    v.slot = -1;
                    std::vector<int32_t>().swap(v.tokens);
                    unsaved.insert(sk);
                    stats.evictions += 1;
                    break;
                }
            }
            if (slot >= 0) {
                const uint64_t k = keys[size_t(admit)];
                Entry &e = map.at(k);
                unsaved.erase({e.stamp, k});
                e.slot = slot;
                e.tokens.assign(tok, tok + size_t(admit) * size_t(B));
                saved.insert({e.stamp, k});
                stats.admissions += 1;
            } else {
                admit = 0;
            }
        }
        while (unsaved.size() > size_t(max_tracked)) {
            map.erase(unsaved.begin()->second);
            unsaved.erase(unsaved.begin());
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
        Entry &e = cache->map.at(it->second);
        if (e.slot != slot) continue;
        try {
            cache->unsaved.insert(*it);
            cache->free_slots.insert(slot);
        } catch (const std::bad_alloc &) {
            return KDA_ERR_HOST_MEMORY;
        }
        cache->saved.erase(it);
        e.slot = -1;
        std::vector<int32_t>().swap(e.tokens);
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
    for (const auto &sk : cache->saved) {
        const Entry &e = cache->map.at(sk.second);
        if (n < cap) {
            lens[n] = int32_t(e.tokens.size());
            slots[n] = e.slot;
        }
        ++n;
    }
    return n;
}

}  // extern "C"
