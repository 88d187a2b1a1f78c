// adapter_cache.cpp -- host side: which adapters stay resident in the device pool.
//
// What it decides ("m07 -- Multi-Adapter (LoRA) Serving", section 7 "Deep Dive B: The
// Cold-Start Long Tail", "Eviction, and the trap in it"; the same page's revision R3 "The
// pinning guard was inconsistent"; "12. Adapter Serving and Multi-Tenant Customization",
// section "Tiered storage: hot, warm, cold"):
//
//   * an adapter's value is the requests it received in the last `window_s` seconds divided by
//     the bytes it holds; to make room, resident adapters are evicted lowest value first (ties:
//     the one whose latest request is older, then the smaller id);
//   * an adapter with in-flight sequences (reference count > 0) is never evicted: a sequence
//     needs its adapter for every step of its generation;
//   * the pinning guard: while the pinned bytes (resident adapters with a reference) exceed
//     `guard_fraction` of the budget, no NEW adapter is admitted -- existing ones keep serving.
//
// The cache only decides; the caller carries the decisions out on the device pool (unload the
// listed adapters, then load the new one, on any stream it likes).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <deque>
#include <map>
#include <vector>

#include "../../include/lora_gb300.h"

struct lora_cache {
    struct Entry {
        int64_t bytes = 0;
        int32_t ref = 0;
        bool resident = false;
        std::deque<double> hits;  // request times inside the window, oldest first
        double last = -INFINITY;  // latest request time
    };
    int64_t budget = 0;
    double guard = 0.5;
    double window = 3600.0;
    int64_t used = 0;
    double clock = -INFINITY;  // latest request time seen; times never go back
    std::map<int32_t, Entry> entries;

    void prune(Entry &e, double now) const {
        while (!e.hits.empty() && e.hits.front() <= now - window) e.hits.pop_front();
    }
    int64_t pinned() const {
        int64_t b = 0;
        for (const auto &kv : entries)
            if (kv.second.resident && kv.second.ref > 0) b += kv.second.bytes;
        return b;
    }
};

extern "C" {

int lora_cache_create(int64_t budget_bytes, double guard_fraction, double window_s, lora_cache **out) {
    if (!out || budget_bytes < 0 || !(guard_fraction >= 0.0 && guard_fraction <= 1.0) || !(window_s > 0.0))
        return LORA_EINVAL;
    lora_cache *c = new lora_cache;
    c->budget = budget_bytes;
    c->guard = guard_fraction;
    c->window = window_s;
    *out = c;
    return LORA_OK;
}

int lora_cache_destroy(lora_cache *c) {
    if (!c) return LORA_EINVAL;
    delete c;
    return LORA_OK;
}

int lora_cache_acquire(lora_cache *c, int32_t adapter, int64_t bytes, double now_s, int32_t *evict, int32_t evict_cap,
                       int32_t *n_evict, int32_t *must_load) {
    if (!c || adapter < 0 || bytes <= 0 || std::isnan(now_s) || !n_evict || !must_load || evict_cap < 0 ||
        (evict_cap > 0 && !evict))
        return LORA_EINVAL;
    *n_evict = 0;
    *must_load = 0;
    if (now_s < c->clock) return LORA_EINVAL;
    c->clock = now_s;
    auto found = c->entries.find(adapter);
    if (found != c->entries.end() && found->second.resident) {
        lora_cache::Entry &e = found->second;
        if (e.bytes != bytes) return LORA_EINVAL;
        e.hits.push_back(now_s);
        e.last = now_s;
        c->prune(e, now_s);
        ++e.ref;
        return LORA_OK;
    }
    // a new adapter: the pinning guard, then room
    if ((double)c->pinned() > c->guard * (double)c->budget) return LORA_EPINNED;
    if (bytes > c->budget) return LORA_ENOMEM;
    std::vector<std::pair<int32_t, lora_cache::Entry *>> cand;
    for (auto &kv : c->entries)
        if (kv.second.resident && kv.second.ref == 0 && kv.first != adapter) {
            c->prune(kv.second, now_s);
            cand.push_back({kv.first, &kv.second});
        }
    // lowest value (requests in the window per byte) first; compared exactly as cross products
    std::sort(cand.begin(), cand.end(), [](const auto &a, const auto &b) {
        const __int128 va = (__int128)a.second->hits.size() * b.second->bytes;
        const __int128 vb = (__int128)b.second->hits.size() * a.second->bytes;
        if (va != vb) return va < vb;
        if (a.second->last != b.second->last) return a.second->last < b.second->last;
        return a.first < b.first;
    });
    int64_t free_bytes = c->budget - c->used;
    size_t k = 0;
    while (free_bytes < bytes && k < cand.size()) free_bytes += cand[k++].second->bytes;
    if (free_bytes < bytes) return LORA_ENOMEM;  // everything unpinned would not make room: nothing changes
    if ((int32_t)k > evict_cap) return LORA_EINVAL;
    for (size_t i = 0; i < k; ++i) {
        evict[i] = cand[i].first;
        cand[i].second->resident = false;
        c->used -= cand[i].second->bytes;
    }
    *n_evict = (int32_t)k;
    lora_cache::Entry &e = c->entries[adapter];
    e.bytes = bytes;
    e.resident = true;
    e.ref = 1;
    e.hits.push_back(now_s);
    e.last = now_s;
    c->prune(e, now_s);
    c->used += bytes;
    *must_load = 1;
    return LORA_OK;
}

int lora_cache_release(lora_cache *c, int32_t adapter) {
    if (!c) return LORA_EINVAL;
    auto it = c->entries.find(adapter);
    if (it == c->entries.end() || !it->second.resident || it->second.ref <= 0) return LORA_EINVAL;
    --it->second.ref;
    return LORA_OK;
}

int lora_cache_stats(const lora_cache *c, int64_t *used_bytes, int64_t *pinned_bytes, int32_t *resident) {
    if (!c || !used_bytes || !pinned_bytes || !resident) return LORA_EINVAL;
    *used_bytes = c->used;
    *pinned_bytes = c->pinned();
    int32_t n = 0;
    for (const auto &kv : c->entries) n += kv.second.resident ? 1 : 0;
    *resident = n;
    return LORA_OK;
}

int lora_cache_resident(const lora_cache *c, int32_t adapter, int32_t *resident, int32_t *ref) {
    if (!c || !resident || !ref) return LORA_EINVAL;
    auto it = c->entries.find(adapter);
    *resident = (it != c->entries.end() && it->second.resident) ? 1 : 0;
    *ref = *resident ? it->second.ref : 0;
    return LORA_OK;
}

}  // extern "C"
