// Launch orders for grids of work items of unequal length (host code, shared by the forward
// and backward kernels). One CTA of these kernels is resident per SM at a time and the
// hardware gives the next block to the first SM that frees up, so the block order decides the
// makespan: the items (weight + fixed each) are packed best-fit decreasing into one bin per SM
// at the smallest capacity that packs, and the blocks go out in order of their start time in
// that packing, which list scheduling then follows.
#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "attn_internal.h"

namespace attn {

namespace {

// Best-fit-decreasing packing of the items (weight + fixed each) into `bins` bins at the smallest
// capacity that packs. Any capacity of at least the even split plus the heaviest item packs, so
// the unit steps end within wmax tries; past 64 tries the step doubles to bound the host time for
// callers with very large weights (the kernels' own weights stay far below that). Fills each
// item's bin and start offset within it, and returns the items heaviest first.
std::vector<int> pack_best_fit(const std::vector<int>& weights, int fixed, int bins, std::vector<int>& w,
                               std::vector<int>& bin_of, std::vector<int64_t>& start) {
    const int items = static_cast<int>(weights.size());
    w.assign(weights.begin(), weights.end());
    int64_t total = 0;
    int wmax = 0;
    for (int& x : w) {
        x += fixed;
        total += x;
        wmax = std::max(wmax, x);
    }
    std::vector<int> idx(static_cast<size_t>(items));
    for (int i = 0; i < items; ++i) idx[static_cast<size_t>(i)] = i;
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return w[a] > w[b]; });
    bins = std::max(1, bins);
    std::vector<int64_t> load(static_cast<size_t>(bins));
    bin_of.assign(static_cast<size_t>(items), 0);
    start.assign(static_cast<size_t>(items), 0);
    int tries = 0;
    for (int64_t cap = std::max<int64_t>(wmax, (total + bins - 1) / bins);;
         cap += tries < 64 ? 1 : (int64_t{1} << std::min(tries - 64, 40))) {
        ++tries;
        std::fill(load.begin(), load.end(), 0);
        bool fits = true;
        for (int i : idx) {
            int best = -1;
            for (int b = 0; b < bins; ++b)
                if (load[b] + w[i] <= cap && (best < 0 || load[b] > load[best])) best = b;
            if (best < 0) {
                fits = false;
                break;
            }
            bin_of[static_cast<size_t>(i)] = best;
            start[static_cast<size_t>(i)] = load[best];
            load[best] += w[i];
        }
        if (fits) break;
    }
    return idx;
}

}  // namespace

std::vector<uint16_t> plan_order_compute(const std::vector<int>& weights, int fixed, int num_sms) {
    std::vector<int> w, bin_of;
    std::vector<int64_t> start;
    std::vector<int> idx = pack_best_fit(weights, fixed, num_sms, w, bin_of, start);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
        return start[a] != start[b] ? start[a] < start[b] : w[a] > w[b];
    });
    return std::vector<uint16_t>(idx.begin(), idx.end());
}

void plan_bins_compute(const std::vector<int>& weights, int fixed, int bins, std::vector<uint16_t>& order,
                       std::vector<uint16_t>& bin_start) {
    std::vector<int> w, bin_of;
    std::vector<int64_t> start;
    std::vector<int> idx = pack_best_fit(weights, fixed, bins, w, bin_of, start);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
        return bin_of[a] != bin_of[b] ? bin_of[a] < bin_of[b] : start[a] < start[b];
    });
    order.assign(idx.begin(), idx.end());
    bin_start.assign(static_cast<size_t>(bins) + 1, 0);
    for (int i : idx) ++bin_start[static_cast<size_t>(bin_of[i]) + 1];
    for (int b = 0; b < bins; ++b) bin_start[static_cast<size_t>(b) + 1] += bin_start[static_cast<size_t>(b)];
}

int plan_launch_order(const PlanKey& key, int fixed, int num_sms, const std::function<std::vector<int>()>& weights,
                      uint16_t* out) {
    static std::mutex mu;
    static std::map<std::tuple<PlanKey, int, int>, std::vector<uint16_t>> cache;
    const auto full = std::make_tuple(key, num_sms, fixed);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(full);
    if (it == cache.end()) {
        if (cache.size() >= 256) cache.clear();
        it = cache.emplace(full, plan_order_compute(weights(), fixed, num_sms)).first;
    }
    std::copy(it->second.begin(), it->second.end(), out);
    return static_cast<int>(it->second.size());
}

bool once_per_device(uint64_t* done, int dev, const std::function<bool()>& setup) {
    if (dev < 0 || dev >= 64) return setup();
    const uint64_t bit = uint64_t{1} << dev;
    if (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit) return true;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit) return true;
    if (!setup()) return false;
    __atomic_fetch_or(done, bit, __ATOMIC_RELEASE);
    return true;
}

}  // namespace attn
