// Internal launchers behind the C ABI. Each validates nothing (attn_capi.cu has already
// checked every argument) and returns an attn_status_t.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <functional>
#include <string>
#include <vector>

#include "attn.h"

namespace attn {

// Online-softmax forward on FFMA for float32 tensors ([BH, N, d] contiguous, d = 64 or 128).
// `lse` is null or receives each row's base-2 log-sum-exp ([BH, N] float32).
int launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int64_t BH,
                   int64_t N, int64_t d, bool causal, int num_sms, cudaStream_t stream);

// Online-softmax forward on tcgen05 tensor cores for bf16 (bf16 = true) or fp16 tensors,
// d = 64 or 128; `lse` as above.
int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH,
                  int64_t N, int64_t d, bool causal, bool bf16, int num_sms, cudaStream_t stream);

// Backward pass for float32 tensors (two FFMA kernels): dq, dk, dv from q, k, v, the forward's
// o, the output gradient dout and the forward's base-2 log-sum-exps lse ([BH, N] float32);
// head width d = 64 or 128.
int launch_bwd_f32(const float* q, const float* k, const float* v, const float* o, const float* dout,
                   const float* lse, float* dq, float* dk, float* dv, int64_t BH, int64_t N, int64_t d, bool causal,
                   cudaStream_t stream);

// The same for bf16 (bf16 = true) or fp16 tensors on tcgen05 tensor cores (two kernels).
int launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, int64_t BH, int64_t N, int64_t d, bool causal, bool bf16,
                  int num_sms, cudaStream_t stream);

// Identifies one launch-order plan: the kernel (kind), its shape and any tile sizes that change
// the item weights. Plans are cached per key, SM count and fixed cost.
struct PlanKey {
    int kind;
    int64_t n;
    int64_t bh;
    int a;
    int b;
    bool operator<(const PlanKey& o) const {
        if (kind != o.kind) return kind < o.kind;
        if (n != o.n) return n < o.n;
        if (bh != o.bh) return bh < o.bh;
        if (a != o.a) return a < o.a;
        return b < o.b;
    }
};

// Launch order for a grid of work items of unequal length, one CTA resident per SM at a time
// (the hardware gives the next block to the first SM that frees up; attn_plan.cu): a
// best-fit-decreasing packing of the items, weight[i] + fixed each, into num_sms bins at the
// smallest capacity that packs (tried upward from the even split, the step doubling after 64
// tries), then the items in order of their start time in that packing. Writes the permutation
// (block -> item) to out and returns its length. Plans are cached by key (at most 256 plans,
// thread-safe); `weights` is called only on a cache miss and must return at most 65536 weights.
int plan_launch_order(const PlanKey& key, int fixed, int num_sms, const std::function<std::vector<int>()>& weights,
                      uint16_t* out);
// The same plan without the cache (for the attn_plan_launch_order entry point).
std::vector<uint16_t> plan_order_compute(const std::vector<int>& weights, int fixed, int num_sms);

// The same packing for persistent grids: the items of bin b (one bin per persistent CTA or
// cluster) are order[bin_start[b] .. bin_start[b+1]), in order of their start in the packing.
// The item count must not exceed 65536 and bins must be at least 1.
void plan_bins_compute(const std::vector<int>& weights, int fixed, int bins, std::vector<uint16_t>& order,
                       std::vector<uint16_t>& bin_start);

// Runs `setup` once per device ordinal (0..63) for the calling site's `done` mask: the first call on
// a device runs it under a lock and records success; later calls return at once. Returns false if
// setup failed (it is then tried again on the next call).
bool once_per_device(uint64_t* done, int dev, const std::function<bool()>& setup);

// Reads (and optionally clears) the tensor-core backward kernels' device error word.
int bwd_tc_device_error(bool clear, unsigned* err);

// Reads (and optionally clears) the tensor-core kernel's device error word after
// synchronising `stream`. *err receives the word.
int tc_device_error(cudaStream_t stream, bool clear, unsigned* err);

// Materialised path: scores, three-pass softmax, weighted values, for `heads` heads whose
// scratch starts at `ws` (per-head stride `head_ws_bytes`).
int launch_materialized(const void* q, const void* k, const void* v, void* o, void* ws,
                        size_t head_ws_bytes, int64_t heads, int64_t N, bool causal, int dtype,
                        cudaStream_t stream);

// Per-head scratch of the materialised path: S and P (N x N fp32 each) and N row totals,
// each region rounded up to 256 bytes. Returns 0 on overflow.
size_t materialized_head_bytes(int64_t N);

// Key-value cache attention (attn_decode.cu): Nq queries [BH, Nq, d] against Nk keys and
// values [BH, Nk, d], d = 64 or 128. splits == 0 balances the tiles over a persistent grid;
// splits >= 1 cuts every (head, query group) into that many shares. Pieces of a segment are
// merged by a second kernel through the workspace; ATTN_ERR_WORKSPACE if it is smaller than
// the plan needs.
int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                  size_t workspace_bytes, int64_t BH, int64_t Nq, int64_t Nk, int64_t d, bool causal, int dtype,
                  int splits, int num_sms, cudaStream_t stream);

// Workspace bytes launch_decode needs (0 when no segment has more than one piece, or on
// overflow). For splits == 0 the plan depends on the device: num_sms and the kernel's
// occupancy, which this queries on the current device.
size_t decode_workspace_bytes(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int splits, int dtype, int num_sms);

// Launches one warp whose only wait (on an mbarrier nobody arrives on) runs out after
// timeout_ns; it then records a timeout in the decode kernel's device error word.
int launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream);

// Reads (and optionally clears) the decode kernel's device error word.
int decode_device_error(bool clear, unsigned* err);

// Reads (and optionally clears) the tensor-core decode kernel's device error word.
int decode_tc_device_error(bool clear, unsigned* err);

}  // namespace attn
