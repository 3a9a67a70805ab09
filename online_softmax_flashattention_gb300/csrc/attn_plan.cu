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
#include <vector>

#include "attn_internal.h"

namespace attn {

std::vector<uint16_t> plan_order_compute(const std::vector<int>& weights, int fixed, int num_sms) {
    const int items = static_cast<int>(weights.size());
    std::vector<int> w(weights);
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
    const int bins = std::max(1, num_sms);
    std::vector<int64_t> load(static_cast<size_t>(bins));
    std::vector<int64_t> start(static_cast<size_t>(items));
    // Any capacity of at least the even split plus the heaviest item packs, so the unit steps
    // end within wmax tries; past 64 tries the step doubles to bound the host time for callers
    // with very large weights (the kernels' own weights stay far below that).
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
            start[static_cast<size_t>(i)] = load[best];
            load[best] += w[i];
        }
        if (fits) break;
    }
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
        return start[a] != start[b] ? start[a] < start[b] : w[a] > w[b];
    });
    return std::vector<uint16_t>(idx.begin(), idx.end());
}

int plan_launch_order(const std::vector<int>& weights, int fixed, int num_sms, const std::string& key,
                      uint16_t* out) {
    static std::mutex mu;
    static std::map<std::string, std::vector<uint16_t>> cache;
    const std::string full = key + " @" + std::to_string(num_sms) + "/" + std::to_string(fixed);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(full);
    if (it == cache.end()) {
        if (cache.size() >= 256) cache.clear();
        it = cache.emplace(full, plan_order_compute(weights, fixed, num_sms)).first;
    }
    std::copy(it->second.begin(), it->second.end(), out);
    return static_cast<int>(it->second.size());
}

}  // namespace attn
