// batch_former.cpp -- host side: the adapter-aware batch former that picks the rows of the next
// step from the waiting requests.
//
// What it computes ("m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A: Batching
// Heterogeneous Adapters", "The adapter-aware scheduler" and "The fairness cost, which must be
// stated"; the same page's revision R1 "The long tail needs a reserved batch slot"; "12. Adapter
// Serving and Multi-Tenant Customization", section "Scheduling with adapter awareness"):
//
//   1. age override: every request that has waited longer than the deadline is admitted first,
//      oldest first, and its adapter counts as one of the batch's adapters;
//   2. reserved tail slots: of the remaining requests, the oldest ones whose adapter has exactly
//      one waiting request fill up to `tail_slots` places;
//   3. grouping: the remaining requests are grouped by adapter (groups in order of first arrival),
//      the groups are visited largest first (ties keep that order), and each group is taken
//      whole while the batch has room (the last one is cut to fit).  Once the batch holds
//      `max_distinct` adapters and at least `min_batch` requests, no group that would add a new
//      adapter is admitted; groups of adapters already in the batch, and the base-only group,
//      still are.
//
// A step's adapter bytes are proportional to its distinct adapters (the same section, "The cost
// is bandwidth, not compute"), so the cap bounds them whatever the traffic looks like.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/lora_gb300.h"

namespace {

struct Group {
    int32_t adapter;
    std::vector<int32_t> members;  // queue indices, in queue order
};

// the requests of `cand` ordered oldest first (ties: queue order)
void oldest_first(std::vector<int32_t> &cand, const double *waited) {
    std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) { return waited[a] > waited[b]; });
}

}  // namespace

extern "C" int lora_form_batch(const int32_t *queue_adapter, const double *queue_waited_ms, int32_t n_queue,
                               const lora_batch_policy *policy, int32_t *out_idx, int32_t *out_n,
                               int32_t *out_distinct) {
    if (!policy || !out_n || !out_distinct || n_queue < 0) return LORA_EINVAL;
    const lora_batch_policy P = *policy;
    if (P.max_batch < 1 || P.max_distinct < 0 || P.min_batch < 0 || P.tail_slots < 0 || std::isnan(P.max_queue_ms))
        return LORA_EINVAL;
    if (n_queue > 0 && (!queue_adapter || !queue_waited_ms || !out_idx)) return LORA_EINVAL;
    for (int32_t i = 0; i < n_queue; ++i)
        if (queue_adapter[i] < -1 || std::isnan(queue_waited_ms[i])) return LORA_EINVAL;

    std::vector<char> taken((size_t)n_queue, 0);
    std::vector<int32_t> batch;
    batch.reserve((size_t)std::min(n_queue, P.max_batch));
    std::unordered_set<int32_t> present;  // adapter ids (>= 0) in the batch
    auto admit = [&](int32_t i) {
        taken[(size_t)i] = 1;
        batch.push_back(i);
        if (queue_adapter[i] >= 0) present.insert(queue_adapter[i]);
    };
    const auto room = [&]() { return (int32_t)batch.size() < P.max_batch; };

    // 1. age override
    if (P.max_queue_ms > 0) {
        std::vector<int32_t> urgent;
        for (int32_t i = 0; i < n_queue; ++i)
            if (queue_waited_ms[i] > P.max_queue_ms) urgent.push_back(i);
        oldest_first(urgent, queue_waited_ms);
        for (int32_t i : urgent) {
            if (!room()) break;
            admit(i);
        }
    }

    // 2. reserved tail slots: adapters with exactly one waiting request (not yet admitted)
    if (P.tail_slots > 0 && room()) {
        std::unordered_map<int32_t, int32_t> count;
        for (int32_t i = 0; i < n_queue; ++i)
            if (!taken[(size_t)i] && queue_adapter[i] >= 0) ++count[queue_adapter[i]];
        std::vector<int32_t> singles;
        for (int32_t i = 0; i < n_queue; ++i)
            if (!taken[(size_t)i] && queue_adapter[i] >= 0 && count[queue_adapter[i]] == 1) singles.push_back(i);
        oldest_first(singles, queue_waited_ms);
        int32_t used = 0;
        for (int32_t i : singles) {
            if (used == P.tail_slots || !room()) break;
            admit(i);
            ++used;
        }
    }

    // 3. grouping, largest groups first
    if (room()) {
        std::vector<Group> groups;
        std::unordered_map<int32_t, size_t> where;
        for (int32_t i = 0; i < n_queue; ++i) {
            if (taken[(size_t)i]) continue;
            const int32_t a = queue_adapter[i];
            auto it = where.find(a);
            if (it == where.end()) {
                where.emplace(a, groups.size());
                groups.push_back(Group{a, {i}});
            } else {
                groups[it->second].members.push_back(i);
            }
        }
        std::stable_sort(groups.begin(), groups.end(),
                         [](const Group &x, const Group &y) { return x.members.size() > y.members.size(); });
        for (const Group &g : groups) {
            const bool is_new = g.adapter >= 0 && present.count(g.adapter) == 0;
            if (is_new && (int32_t)present.size() >= P.max_distinct && (int32_t)batch.size() >= P.min_batch)
                continue;  // no new adapters once the cap binds
            for (int32_t i : g.members) {
                if (!room()) break;
                admit(i);
            }
            if (!room()) break;
        }
    }

    std::copy(batch.begin(), batch.end(), out_idx);
    *out_n = (int32_t)batch.size();
    *out_distinct = (int32_t)present.size();
    return LORA_OK;
}
