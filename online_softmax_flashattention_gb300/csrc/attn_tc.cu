// Online-softmax attention forward for bf16 / fp16 on GB300 (sm_103a) tensor cores.
//
// What it computes is exact attention, o = softmax(q k^T / sqrt(d) + causal mask) v, per
// head ("Flash attention in PyTorch, then in Triton", sections "Attention's table of
// scores" and "Flash attention"). The keys are consumed in tiles; each query row carries a
// running maximum m, a running denominator l and a running output O, and when a tile
// raises the maximum, l and O are multiplied by exp(m_old - m_new) before the tile's own
// terms are added (the online normaliser of that page's "Flash attention" section and of
// attention.cu's attentionOnline). After the last tile O / l is the softmax-weighted sum.
// Scores are kept in base-2 units, s * log2(e) / sqrt(d), so every exponential is an exp2
// (section "A kernel in Triton" scales its scores by log2(e) for the same reason), and the
// probabilities are rounded to the input type before they weigh v so the tensor cores can
// take them (same section). Causal tiles past a query tile's last row are skipped
// (section "The online softmax, in PyTorch"); ragged N is masked on keys and clipped on
// stores.
//
// The reference m only has to be the same for l and O, not the exact running maximum:
// any common reference gives the same O / l. The kernel therefore keeps a stale maximum
// until a tile exceeds it by more than 2^8 (then probabilities stay below 256, well inside
// bf16/fp16 and fp32 range), which makes the O rescale rare instead of nearly every tile.
//
// GB300 mapping (a fresh design; the pages' kernels target sm_75 CUDA cores and a Triton
// kernel on sm_89):
//   * One CTA owns two query tiles A and B of 128 rows (rows 256c .. 256c+255 of one head)
//     and streams K/V tiles of BN keys past both (BN = 128 at head width 64, 64 at 128), so
//     each K/V tile is fetched once for 256 queries.
//   * Warp 8 issues TMA loads (128-byte swizzle) into a 4-stage K ring and a 3-stage V ring
//     guarded by full/empty mbarriers. Warp 9 owns the tensor memory and issues the S = Q K^T
//     products, warp 10 the O += P V products, each for whichever tile's inputs are ready
//     first: the PV products from one thread, the S products from one thread at head width 64
//     and from the whole warp (elect.sync) at 128. Warps 0-3 (tile A) and 4-7 (tile B) are the softmax warpgroups:
//     thread t of a group owns query row t, which is TMEM lane t, so row reductions need no
//     shuffles. The third warpgroup (warps 8-11) gives up registers so the softmax groups can
//     hold a whole row of scores.
//   * Causal grids launch their blocks in the order of a best-fit-decreasing packing of the
//     work items into one bin per SM (plan_launch_order), so the hardware's first-free-SM
//     dispatch balances the uneven causal items.
//   * Tensor memory (512 columns x 128 lanes x 32 bit): S_A, S_B fp32 scores (BN columns
//     each), O_A, O_B fp32 outputs (d each), P_A, P_B probabilities as 16-bit pairs (BN/2
//     each). S = Q K^T runs with both operands in shared memory; O += P V takes P from
//     tensor memory and V (dims contiguous, "MN-major") from shared memory.
//   * S_X(j+1) is issued as soon as softmax X has copied S_X(j) into registers, so the
//     next QK^T overlaps the exponentials, and the two groups' products interleave.
//   * Epilogue: each tile's softmax warps write O / l, rounded to the output type, into the
//     tile's Q buffer (free once its last S product has completed) in the 128-byte-swizzled
//     layout of the output's TMA box, and one thread stores the box with a TMA bulk store; the
//     tensor map clips rows >= N.
//   * With an `lse` pointer the epilogue also stores each row's log-sum-exp in base 2,
//     m + log2 l, as the page's forward kernel keeps it for the backward pass ("Backwards,
//     and training with it"); any common reference m gives the same value.
//   * Every mbarrier wait is bounded. A wait that exceeds its deadline sets the device
//     error word and an abort flag; all roles then leave their loops, drain copies and MMAs
//     still in flight (with a deadline of their own), free tensor memory and return.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <map>
#include <string>
#include <mutex>
#include <tuple>
#include <vector>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per tile = TMEM lanes
constexpr int kBlockBytes = kBM * 64 * 2;  // one 128-row x 128-byte column block of a Q tile
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kSIssuerWarp = 9;   // also owns the tensor memory
constexpr int kPVIssuerWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s for any single wait
constexpr uint64_t kDrainTimeoutNs = 100000000ull;  // 100 ms to drain after an abort
constexpr unsigned kPollSleepNs = 32;  // MMA issuers' back-off between unproductive polls
constexpr float kLazyLog2 = 8.f;  // keep a stale max until a tile exceeds it by 2^8
constexpr float kLazyBound = 256.f;  // 2^kLazyLog2
// Register split: launch at 168 per thread (384 x 168 = 64512); the third warpgroup
// drops to 56 and the two softmax groups rise to 224 (256 x 224 + 128 x 56 = 64512).
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 224;
constexpr int kRegsOther = 56;
static_assert(2 * 128 * kRegsSoftmax + (kThreads - 2 * 128) * kRegsOther <= kThreads * kRegsLaunch,
              "register split must fit the launch allocation");
static_assert(kThreads * kRegsLaunch <= 65536, "launch allocation must fit the register file");

// Everything that depends on the head width D (64 or 128) and the key-tile size BN (128 keys at
// D = 64, 64 at D = 128). A Q tile of 128 rows x D 16-bit values is D/64 column blocks of 128
// rows x 128 bytes, a K or V tile D/64 blocks of BN rows x 128 bytes, each loaded by its own TMA
// box. Tensor memory: S_X (BN fp32 columns) at BN X, O_X (D columns) at 2 BN + D X, P_X (the
// probabilities as 16-bit pairs, BN/2 columns) at 2 BN + 2 D + BN/2 X: 512 columns at D = 64,
// 448 at D = 128. (With 128-key tiles at D = 128, S and O alone would fill the 512 columns, P
// would have to sit over S and S_X(j+1) would wait for PV_X(j); 64-key tiles avoid that.)
template <int D>
struct Lay {
    static_assert(D == 64 || D == 128, "head width 64 or 128");
    static constexpr int kBN = D == 64 ? 128 : 64;
    static constexpr int kBlocks = D / 64;
    static constexpr int kTileBytes = kBlocks * kBlockBytes;     // Q tile: 16 or 32 KiB
    static constexpr int kKVBlockBytes = kBN * 128;              // one column block of a K/V tile
    static constexpr int kKVTileBytes = kBlocks * kKVBlockBytes; // K or V tile: 16 KiB
    static constexpr int kKStages = 4;  // K ring depth (QK^T reads K one step ahead)
    static constexpr int kVStages = 3;  // V ring depth
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 2 * kBN;
    static constexpr uint32_t kColP0 = 2 * kBN + 2 * D;
    __host__ __device__ static constexpr uint32_t colS(int X) { return kColS + kBN * static_cast<uint32_t>(X); }
    __host__ __device__ static constexpr uint32_t colO(int X) { return kColO + D * static_cast<uint32_t>(X); }
    __host__ __device__ static constexpr uint32_t colP(int X) { return kColP0 + (kBN / 2) * static_cast<uint32_t>(X); }
    // Shared-memory layout (byte offsets from a 1024-byte aligned base).
    static constexpr int kOffQ = 0;                                  // 2 tiles
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;             // kKStages tiles
    static constexpr int kOffV = kOffK + kKStages * kKVTileBytes;    // kVStages tiles
    static constexpr int kOffBar = kOffV + kVStages * kKVTileBytes;  // mbarriers, 8 bytes each
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kBarSFull = kBarVEmpty + kVStages;  // [2] S_X(j) computed
    static constexpr int kBarSFree = kBarSFull + 2;          // [2] softmax X copied S_X(j) out (4 warps)
    static constexpr int kBarPFull = kBarSFree + 2;          // [2] softmax X wrote P_X(j) (4 warps)
    static constexpr int kBarOReady = kBarPFull + 2;         // [2] PV_X(j) done: O_X stable, P_X reusable
    static constexpr int kBarDrain = kBarOReady + 2;         // [2] every MMA of issuer 0 (S) / 1 (PV) done
    static constexpr int kBarEpi = kBarDrain + 2;            // [2] tile X's output rows are in shared memory (4 warps)
    static constexpr int kNumBars = kBarEpi + 2;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;  // TMEM base address written by tcgen05.alloc
    static constexpr int kOffAbort = kOffSlot + 4;
    static constexpr int kSmemUsed = kOffAbort + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
    static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms need 1024-byte alignment");
    static_assert(kColP0 + kBN <= kTmemCols, "tensor memory budget");
};

__device__ unsigned int g_tc_error = 0;

// Launch order of the work items (item = pair * BH + head) for causal calls with at most
// kOrderMax items: block b runs item order[b] (see plan_launch_order). Longer calls, and
// non-causal ones, run heaviest pairs first without a table.
constexpr int kOrderMax = 2048;

struct TcParams {
    void* o;
    float* lse;  // null, or [BH, N] base-2 log-sum-exps
    int N;
    int BH;
    int num_pairs;
    int causal;
    float scale_log2;  // log2(e) / sqrt(d)
    int order_len;     // 0: no table
    uint16_t order[kOrderMax];
};

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_tc_error, 1u);
}

// A decision of an issuer loop: with kWarp the whole warp runs the loop, so the lanes' results
// are combined into one (every lane reads the same barrier or flag in the same instruction, so
// they agree anyway; the vote makes the branch provably uniform for elect.sync); a single-lane
// issuer passes its own result through.
template <bool kWarp>
__device__ __forceinline__ bool warp_vote(bool v) {
    if constexpr (kWarp) return __all_sync(0xffffffffu, v);
    return v;
}
template <bool kWarp>
__device__ __forceinline__ bool warp_vote_any(bool v) {
    if constexpr (kWarp) return __any_sync(0xffffffffu, v);
    return v;
}

// All lanes of a warp wait; the result is the same in every lane, so a warp never splits
// in front of a warp-collective tcgen05.ld / tcgen05.st.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag, kWaitTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t* r) {
    ATTN_TMEM_ST_X32(taddr, r);
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Row maximum of BN (64 or 128) scores as eight independent chains of 3-input max, then a tree.
template <int BN>
__device__ __forceinline__ float row_max(const float (&s)[BN]) {
    static_assert(BN / 8 % 2 == 0 && BN >= 32, "an even number of 8-wide groups");
    float mx[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) mx[g] = fmax3(s[g], s[g + 8], s[g + 16]);
#pragma unroll
    for (int t = 3; t < BN / 8 - 1; t += 2)
#pragma unroll
        for (int g = 0; g < 8; ++g) mx[g] = fmax3(mx[g], s[g + 8 * t], s[g + 8 * t + 8]);
#pragma unroll
    for (int g = 0; g < 8; ++g) mx[g] = fmaxf(mx[g], s[g + BN - 8]);
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
}

// p = 2^(s * c - m) for the BN scores of a row, packed to 16-bit pairs (round to nearest
// even) in `pk`; returns the fp32 sum of the unrounded p (four independent partial sums).
template <bool BF16, int BN>
__device__ __forceinline__ float row_exp2_t(const uint32_t (&su)[BN], float2 c2, float2 negm,
                                            uint32_t (&pk)[BN / 2]) {
    float2 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) {
        const float2 t = ffma2(make_float2(__uint_as_float(su[2 * i]), __uint_as_float(su[2 * i + 1])), c2, negm);
        const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        acc[i & 3] = fadd2(acc[i & 3], pp);
        pk[i] = pack2<BF16>(pp.x, pp.y);
    }
    const float2 at = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    return at.x + at.y;
}

// One softmax warpgroup's view: its lanes of S_X, O_X, P_X and its barriers.
struct SoftmaxCtx {
    uint32_t tS, tO, tP;
    uint32_t bar_s_full, bar_s_free, bar_p_full, bar_o_ready;
    volatile int* abort_flag;
    float c;    // log2(e) / sqrt(d)
    int limit;  // keys >= limit are masked for this row
    int lane;
};

template <int BN>
__device__ __forceinline__ void load_s(const SoftmaxCtx& cx, uint32_t (&su)[BN]) {
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) ATTN_TMEM_LD_X32(cx.tS + 32 * c, (su + 32 * c));
}

__device__ __forceinline__ void release_s(const SoftmaxCtx& cx) {
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (cx.lane == 0) mbar_arrive(cx.bar_s_free);
}

// One key tile of the online softmax for this thread's query row: scores in `su`, running
// reference m and denominator l. Writes P(j) to tensor memory, rescales O when the
// reference moves, starts loading S(j+1) and signals the MMA issuers. Returns false when a
// wait timed out or the CTA is aborting (the result is the same in all lanes of a warp).
template <bool BF16, bool kMasked, int D>
__device__ __forceinline__ bool softmax_step(const SoftmaxCtx& cx, uint32_t (&su)[Lay<D>::kBN], float& m,
                                             float& l, int j, int nX) {
    constexpr int kBN = Lay<D>::kBN;
    // The scores stay in the registers tcgen05.ld filled (as bit patterns); masked keys get
    // the bit pattern of -inf.
    if constexpr (kMasked) {
        const int nvalid = cx.limit - j * kBN;
#pragma unroll
        for (int i = 0; i < kBN; ++i) su[i] = (i < nvalid) ? su[i] : 0xFF800000u;
    }
    const float c = cx.c;
    const float2 c2 = make_float2(c, c);
    // Optimistic pass: exponentials against the current (possibly stale) reference m. If
    // some p exceeded 2^kLazyLog2 (the lazy rule would then move m), the tile's sum of p
    // would exceed 2^kLazyLog2 too; so a sum within that bound proves m may stay, and only
    // otherwise (or on the first tile) the row maximum is computed and p redone if m moves.
    uint32_t pk[kBN / 2];
    float tile_sum = INFINITY;
    if (m != -INFINITY) tile_sum = row_exp2_t<BF16, kBN>(su, c2, make_float2(-m, -m), pk);
    float alpha = 1.f;
    if (!(tile_sum <= kLazyBound)) {
        float s[kBN];
#pragma unroll
        for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(su[i]);
        const float mt = row_max<kBN>(s) * c;
        if (mt > m + kLazyLog2) {
            alpha = ex2_approx(m - mt);  // 0 on the first tile (m = -inf)
            m = mt;
            l *= alpha;
        }
        // A row with every key masked so far keeps a zero reference (no inf - inf).
        const float m_use = (m == -INFINITY) ? 0.f : m;
        if (alpha != 1.f || tile_sum == INFINITY || tile_sum != tile_sum)
            tile_sum = row_exp2_t<BF16, kBN>(su, c2, make_float2(-m_use, -m_use), pk);
    }
    bool rescale = false;
    if (j > 0) {
        if (!warp_wait(cx.bar_o_ready, (j - 1) & 1, cx.abort_flag)) return false;
        tc_fence_after();
        rescale = __any_sync(0xffffffffu, alpha != 1.f);
    }
#pragma unroll
    for (int c = 0; c < kBN / 64; ++c) tmem_st_x32(cx.tP + 32 * c, pk + 32 * c);
    if (rescale) {
        // O <- alpha * O (rare: only when some row of this warp moved its reference); done in
        // 16-column pieces so it adds few registers to the step.
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
        for (int h = 0; h < D / 16; ++h) {
            uint32_t ou[16];
            tmem_ld_x16(cx.tO + 16 * h, ou);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float2 v = fmul2(make_float2(__uint_as_float(ou[i]), __uint_as_float(ou[i + 1])), a2);
                ou[i] = __float_as_uint(v.x);
                ou[i + 1] = __float_as_uint(v.y);
            }
            tmem_st_x16(cx.tO + 16 * h, ou);
        }
    }
    l += tile_sum;
    const bool more = j + 1 < nX;
    bool ok = true;
    if (more) {  // the next scores start moving while P drains
        ok = warp_wait(cx.bar_s_full, (j + 1) & 1, cx.abort_flag);
        if (ok) load_s<kBN>(cx, su);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (cx.lane == 0) mbar_arrive(cx.bar_p_full);
    if (more && ok) release_s(cx);
    return ok;
}

// S_X(j) = Q_X K_j^T : M=128, N=BN, K=D as D/16 steps of K=16 (32 bytes of a 128-byte row;
// steps 4..7 of D = 128 read the second column block of each tile). kWarp: issued by a whole
// converged warp, elect.sync picking the lane (see the S issuer); else by the calling thread.
template <bool BF16, int D, bool kWarp>
__device__ __forceinline__ void issue_s(uint32_t tmem, uint32_t sQx, uint32_t sKs, int X, uint32_t bar_s_full) {
    using L = Lay<D>;
    constexpr uint32_t kIdescQK = idesc_f16(BF16, kBM, L::kBN, false, false);
    // The descriptors of the K=16 steps differ only in their start address (bits 0-13, in
    // 16-byte units; shared addresses stay below 2^18 bytes, so the field cannot carry over).
    const uint64_t a0 = smem_desc_sw128(sQx, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(sKs, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a = a0 + static_cast<uint64_t>(((kk >> 2) * kBlockBytes + 32 * (kk & 3)) >> 4);
        const uint64_t b = b0 + static_cast<uint64_t>(((kk >> 2) * L::kKVBlockBytes + 32 * (kk & 3)) >> 4);
        if constexpr (kWarp)
            umma_ss_elect(tmem + L::colS(X), a, b, kIdescQK, kk > 0 ? 1u : 0u);
        else
            umma_ss(tmem + L::colS(X), a, b, kIdescQK, kk > 0 ? 1u : 0u);
    }
    if constexpr (kWarp)
        umma_commit_elect(bar_s_full);
    else
        umma_commit(bar_s_full);
}

// O_X += P_X V_j : M=128, N=D, K=BN as BN/16 steps of K=16 (16 keys = 2048 bytes of each V
// column block), P from tensor memory. V is the MN-major operand (dims contiguous); for D = 128
// its two 64-dim column blocks are one K/V block apart, the descriptor's leading byte offset.
template <bool BF16, int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t sVs, int X, bool accumulate, uint32_t bar_o_ready) {
    using L = Lay<D>;
    constexpr uint32_t kIdescPV = idesc_f16(BF16, kBM, D, false, true);
    constexpr uint32_t kLbo = D == 64 ? 16u : static_cast<uint32_t>(L::kKVBlockBytes);
    const uint64_t b0 = smem_desc_sw128(sVs, kLbo, 1024);
#pragma unroll
    for (int kk = 0; kk < L::kBN / 16; ++kk) {
        const uint64_t b = b0 + static_cast<uint64_t>((2048 * kk) >> 4);
        umma_ts(tmem + L::colO(X), tmem + L::colP(X) + 8u * kk, b, kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
    }
    umma_commit(bar_o_ready);
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                       const TcParams p) {
    using L = Lay<D>;
    // Who issues S = Q K^T. At D = 128 a step's S is eight N = 64 products, and issuing them
    // from a whole converged warp (operands in uniform registers, elect.sync picking the lane)
    // is what keeps them fed: B1 H12 N8192 causal 1153 -> 1383 TFLOP/s. At D = 64 (four N = 128
    // products a step, the softmax warps heavier) the single-lane issuer measured faster
    // (981 against 953).
    constexpr bool kWarpS = D == 128;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);

    const uint32_t sQ = base + L::kOffQ;
    const uint32_t sK = base + L::kOffK;
    const uint32_t sV = base + L::kOffV;
    auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kOffSlot);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: pair of query tiles (A, B) of head bh, from the launch-order table when
    // the host sent one, else heaviest causal pairs first ----
    const int N = p.N;
    int bh, pair;
    if (p.order_len > 0) {
        const int item = p.order[blockIdx.x];
        bh = item % p.BH;
        pair = item / p.BH;
    } else {
        bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.BH));
        const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.BH));
        pair = p.causal ? (p.num_pairs - 1 - slot) : slot;
    }
    const int rowA = pair * 2 * kBM;
    const int rowB = rowA + kBM;
    constexpr int kBN = L::kBN;
    const int nkv = (N + kBN - 1) / kBN;
    const int nA = p.causal ? min(nkv, (rowA + kBM - 1) / kBN + 1) : nkv;
    const int nB = (rowB < N) ? (p.causal ? min(nkv, (rowB + kBM - 1) / kBN + 1) : nkv) : 0;
    const int nmax = max(nA, nB);

    // ---- setup: barriers (thread 0), tensor memory (S-issuer warp) ----
    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarQFull), 1);
        for (int s = 0; s < L::kKStages; ++s) {
            mbar_init(bar(L::kBarKFull + s), 1);
            mbar_init(bar(L::kBarKEmpty + s), 1);  // released by the last query tile that reads it
        }
        for (int s = 0; s < L::kVStages; ++s) {
            mbar_init(bar(L::kBarVFull + s), 1);
            mbar_init(bar(L::kBarVEmpty + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(L::kBarSFull + x), 1);
            mbar_init(bar(L::kBarSFree + x), 4);
            mbar_init(bar(L::kBarPFull + x), 4);
            mbar_init(bar(L::kBarOReady + x), 1);
            mbar_init(bar(L::kBarDrain + x), 1);
            mbar_init(bar(L::kBarEpi + x), 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kSIssuerWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        // =========================== softmax warpgroups ===========================
        regs_increase<kRegsSoftmax>();
        const int X = warp >> 2;
        const int nX = X ? nB : nA;
        const int row = (X ? rowB : rowA) + ((warp & 3) << 5) + lane;
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const SoftmaxCtx cx{tmem + lane_addr + L::colS(X), tmem + lane_addr + L::colO(X),
                            tmem + lane_addr + L::colP(X), bar(L::kBarSFull + X), bar(L::kBarSFree + X),
                            bar(L::kBarPFull + X), bar(L::kBarOReady + X), abort_flag, p.scale_log2,
                            p.causal ? min(row + 1, N) : N, lane};
        float m = -INFINITY;  // reference max of scaled scores (base-2 units), possibly stale
        float l = 0.f;        // running denominator relative to m
        bool ok = true;
        // `su` holds the scores of the tile about to be used; S(j+1) is copied out of tensor
        // memory while P(j) drains (software pipelining).
        uint32_t su[kBN];
        if (nX > 0) {
            ok = warp_wait(cx.bar_s_full, 0, abort_flag);
            if (ok) {
                load_s<kBN>(cx, su);
                release_s(cx);
            }
        }
        if constexpr (kBN == kBM) {
            // Only a query tile's last key tile can hold masked keys (the causal diagonal or
            // keys past N), so the loop runs mask-free and the last step is peeled off.
            for (int j = 0; ok && j + 1 < nX; ++j) ok = softmax_step<BF16, false, D>(cx, su, m, l, j, nX);
            if (ok && nX > 0) ok = softmax_step<BF16, true, D>(cx, su, m, l, nX - 1, nX);
        } else {
            // Key tiles wholly below the tile's first row (causal) and below N need no mask; the
            // diagonal tiles (two with 64-key tiles) and a ragged last tile take the masked step.
            const int rowX = X ? rowB : rowA;
            const int nfree = min(nX, (p.causal ? min(rowX + 1, N) : N) / kBN);
            int j = 0;
            for (; ok && j < nfree; ++j) ok = softmax_step<BF16, false, D>(cx, su, m, l, j, nX);
            for (; ok && j < nX; ++j) ok = softmax_step<BF16, true, D>(cx, su, m, l, j, nX);
        }

        // ---- epilogue: O / l, rounded to the output type, written into this tile's Q buffer (the
        // tile's last S product has completed) in the 128-byte-swizzled layout of the output's TMA
        // box; then one thread stores the box, which drops rows >= N. ----
        if (ok && nX > 0) {
            if (warp_wait(cx.bar_o_ready, (nX - 1) & 1, abort_flag)) {
                tc_fence_after();
                const float inv = 1.f / l;
                const int r = ((warp & 3) << 5) + lane;  // row of the tile
                const uint32_t sO = sQ + static_cast<uint32_t>(X) * L::kTileBytes;
#pragma unroll 1
                for (int h = 0; h < D / 16; ++h) {
                    uint32_t ou[16];
                    tmem_ld_x16(cx.tO + 16 * h, ou);
                    tmem_ld_wait();
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = pack2<BF16>(__uint_as_float(ou[2 * i]) * inv,
                                            __uint_as_float(ou[2 * i + 1]) * inv);
                    // 16-byte chunk c of row r sits at chunk c ^ (r mod 8) of the row's 128 bytes.
                    const uint32_t rowb = sO + static_cast<uint32_t>(((2 * h) >> 3) * kBlockBytes + r * 128);
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int c = (2 * h + c2) & 7;
                        st_shared_v4(rowb + static_cast<uint32_t>((c ^ (r & 7)) * 16), pk[4 * c2], pk[4 * c2 + 1],
                                     pk[4 * c2 + 2], pk[4 * c2 + 3]);
                    }
                }
                if (p.lse != nullptr && row < N) p.lse[static_cast<int64_t>(bh) * N + row] = m + log2f(l);
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_elect(bar(L::kBarEpi + X));
                if ((warp & 3) == 0) {
                    ok = warp_wait(bar(L::kBarEpi + X), 0, abort_flag);
                    if (ok && lane == 0) {
#pragma unroll
                        for (int c = 0; c < L::kBlocks; ++c)
                            tma_store_3d(&tmap_o, sO + c * kBlockBytes, 64 * c, X ? rowB : rowA, bh);
                        bulk_commit_group();
                        bulk_wait_group_read0();  // the box has left shared memory before the CTA exits
                    }
                    __syncwarp();
                }
            } else {
                ok = false;
            }
        }
        if (!ok) raise_abort(abort_flag);
    } else {
        regs_decrease<kRegsOther>();
        if (warp == kProducerWarp && lane == 0) {
            // =============================== TMA producer ===============================
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(bar(L::kBarQFull), (nB > 0 ? 2 : 1) * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kBlocks; ++c) {
                tma_load_3d(sQ + c * kBlockBytes, &tmap_q, 64 * c, rowA, bh, bar(L::kBarQFull));
                if (nB > 0) tma_load_3d(sQ + L::kTileBytes + c * kBlockBytes, &tmap_q, 64 * c, rowB, bh, bar(L::kBarQFull));
            }
            // K runs ahead of V: K_j is needed by S(j) a step before V_j is needed by PV(j).
            int kissued = 0, vissued = 0;
            bool ok = true;
            for (int j = 0; ok && j < nmax; ++j) {
                const int sk = j % L::kKStages;
                if (!(ok = mbar_wait(bar(L::kBarKEmpty + sk), ((j / L::kKStages) & 1) ^ 1, abort_flag, kWaitTimeoutNs)))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarKFull + sk), L::kKVTileBytes);
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c)
                    tma_load_3d(sK + sk * L::kKVTileBytes + c * L::kKVBlockBytes, &tmap_k, 64 * c, j * kBN, bh,
                                bar(L::kBarKFull + sk));
                kissued = j + 1;
                for (; vissued < j; ++vissued) {  // V_{j-1} after K_j
                    const int sv = vissued % L::kVStages;
                    if (!(ok = mbar_wait(bar(L::kBarVEmpty + sv), ((vissued / L::kVStages) & 1) ^ 1, abort_flag,
                                         kWaitTimeoutNs)))
                        break;
                    mbar_arrive_expect_tx(bar(L::kBarVFull + sv), L::kKVTileBytes);
#pragma unroll
                    for (int c = 0; c < L::kBlocks; ++c)
                        tma_load_3d(sV + sv * L::kKVTileBytes + c * L::kKVBlockBytes, &tmap_v, 64 * c, vissued * kBN, bh,
                                    bar(L::kBarVFull + sv));
                }
            }
            for (; ok && vissued < nmax; ++vissued) {
                const int sv = vissued % L::kVStages;
                if (!(ok = mbar_wait(bar(L::kBarVEmpty + sv), ((vissued / L::kVStages) & 1) ^ 1, abort_flag,
                                     kWaitTimeoutNs)))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarVFull + sv), L::kKVTileBytes);
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c)
                    tma_load_3d(sV + sv * L::kKVTileBytes + c * L::kKVBlockBytes, &tmap_v, 64 * c, vissued * kBN, bh,
                                bar(L::kBarVFull + sv));
            }
            if (!ok) raise_abort(abort_flag);
            // Every copy issued must have landed before the CTA may exit. In normal operation
            // they were all consumed already and these waits return at once.
            mbar_wait(bar(L::kBarQFull), 0, nullptr, kDrainTimeoutNs);
            for (int j = max(0, kissued - L::kKStages); j < kissued; ++j)
                mbar_wait(bar(L::kBarKFull + j % L::kKStages), (j / L::kKStages) & 1, nullptr, kDrainTimeoutNs);
            for (int j = max(0, vissued - L::kVStages); j < vissued; ++j)
                mbar_wait(bar(L::kBarVFull + j % L::kVStages), (j / L::kVStages) & 1, nullptr, kDrainTimeoutNs);
        } else if (warp == kSIssuerWarp && (kWarpS || lane == 0)) {
            // ============================ S issuer: QK^T ============================
            // S_X(j) goes out as soon as K_j has landed and (j > 0) softmax X has copied
            // S_X(j-1) out of tensor memory; the two tiles progress independently. K_j's stage
            // is released by the later of the two tiles' products (the only one when the other
            // tile does not read K_j). At D = 128 (kWarpS) the whole warp runs this loop and
            // elect.sync issues: every decision is a warp vote, so the warp never splits.
            bool ok = warp_vote<kWarpS>(mbar_wait(bar(L::kBarQFull), 0, abort_flag, kWaitTimeoutNs));
            int ns0 = 0, ns1 = 0;
            uint64_t idle_since = 0;
            uint32_t polls = 0;
            while (ok && (ns0 < nA || ns1 < nB)) {
                bool progressed = false;
                // Tile B is tested first here and tile A first in the PV issuer: a fixed order
                // keeps the two tiles' steps interleaved (alternating it each pass cost 16 %),
                // and this one measured best of the four fixed ones.
#pragma unroll
                for (int XX = 0; XX < 2; ++XX) {
                    const int X = XX ^ 1;
                    int& j = X ? ns1 : ns0;
                    const int nX = X ? nB : nA, nO = X ? nA : nB, other = X ? ns0 : ns1;
                    // The usually-late condition first: barrier tests are slow while products
                    // stream their operands out of shared memory.
                    if (j < nX && warp_vote<kWarpS>((j == 0 || mbar_test(bar(L::kBarSFree + X), (j - 1) & 1)) &&
                                                    mbar_test(bar(L::kBarKFull + j % L::kKStages), (j / L::kKStages) & 1))) {
                        tc_fence_after();
                        issue_s<BF16, D, kWarpS>(tmem, sQ + X * L::kTileBytes, sK + (j % L::kKStages) * L::kKVTileBytes,
                                                 X, bar(L::kBarSFull + X));
                        // K_j is released once, after the last product that reads it (a commit
                        // covers every earlier product of this thread).
                        if (other > j || j >= nO) {
                            if constexpr (kWarpS)
                                umma_commit_elect(bar(L::kBarKEmpty + j % L::kKStages));
                            else
                                umma_commit(bar(L::kBarKEmpty + j % L::kKStages));
                        }
                        ++j;
                        progressed = true;
                    }
                }
                if (progressed) {
                    idle_since = 0;
                } else {
                    // Nothing ready: yield the issue slots to the softmax warps for a moment.
                    __nanosleep(kPollSleepNs);
                    if ((++polls & 15u) == 0) {
                        const uint64_t now = global_timer_ns();
                        if (idle_since == 0) idle_since = now;
                        if (warp_vote_any<kWarpS>(*abort_flag != 0 || now - idle_since > kWaitTimeoutNs)) ok = false;
                    }
                }
            }
            if (!ok && lane == 0) raise_abort(abort_flag);
            if constexpr (kWarpS)
                umma_commit_elect(bar(L::kBarDrain + 0));  // no S product may still run at teardown
            else
                umma_commit(bar(L::kBarDrain + 0));
            mbar_wait(bar(L::kBarDrain + 0), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        } else if (warp == kPVIssuerWarp && lane == 0) {
            // ============================== PV issuer ==============================
            // PV_X(j) goes out as soon as V_j has landed and softmax X has written P_X(j); the
            // two tiles progress independently and V_j's stage is released as K_j's is.
            bool ok = true;
            int np0 = 0, np1 = 0;
            uint64_t idle_since = 0;
            uint32_t polls = 0;
            while (ok && (np0 < nA || np1 < nB)) {
                bool progressed = false;
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    int& j = X ? np1 : np0;
                    const int nX = X ? nB : nA, nO = X ? nA : nB, other = X ? np0 : np1;
                    if (j < nX && mbar_test(bar(L::kBarPFull + X), j & 1) &&
                        mbar_test(bar(L::kBarVFull + j % L::kVStages), (j / L::kVStages) & 1)) {
                        tc_fence_after();
                        issue_pv<BF16, D>(tmem, sV + (j % L::kVStages) * L::kKVTileBytes, X, j > 0, bar(L::kBarOReady + X));
                        if (other > j || j >= nO) umma_commit(bar(L::kBarVEmpty + j % L::kVStages));
                        ++j;
                        progressed = true;
                    }
                }
                if (progressed) {
                    idle_since = 0;
                } else {
                    // Nothing ready: yield the issue slots to the softmax warps for a moment.
                    __nanosleep(kPollSleepNs);
                    if ((++polls & 15u) == 0) {
                        const uint64_t now = global_timer_ns();
                        if (idle_since == 0) idle_since = now;
                        if (*abort_flag || now - idle_since > kWaitTimeoutNs) ok = false;
                    }
                }
            }
            if (!ok) raise_abort(abort_flag);
            umma_commit(bar(L::kBarDrain + 1));  // no PV product may still run at teardown
            mbar_wait(bar(L::kBarDrain + 1), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kSIssuerWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [BH][N][D] 16-bit tensor; boxes of 128 rows x 64 values (128 bytes, the swizzle span), one
// per 64-dim column block.
bool make_map(CUtensorMap* map, const void* ptr, int64_t BH, int64_t N, int64_t D, int rows, bool bf16) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(N) * D * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Causal work items differ in length (pair p of query tiles sees about 2p key tiles), and one
// CTA runs per SM at a time, so the order of the blocks decides the makespan. The blocks are
// ordered by a best-fit-decreasing packing of the items into one bin per SM: each item weighs
// its key-tile steps plus kFixedSteps (the per-CTA fill and drain, about five steps), the
// capacity is the smallest that packs, and the blocks go out in order of their start times in
// that packing, so that the hardware, which gives the next block to the first SM that frees
// up, follows it. (Heaviest-first leaves SMs that took a long item with nothing that fits:
// at B1 H12 N8192 it finishes about 107 steps in, the packing about 98.)
constexpr int kFixedSteps = 5;

// The three tensor maps of a call depend only on the pointers and the shape, so the last few
// calls' maps are kept (a small cache shared by all threads, behind a lock).
struct FwdMaps {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    int64_t BH, N;
    int D;
    bool bf16;
    CUtensorMap mq, mk, mv, mo;
};

bool fwd_maps(const void* q, const void* k, const void* v, const void* o, int64_t BH, int64_t N, int D, int kv_rows,
              bool bf16, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv, CUtensorMap* mo) {
    constexpr int kSlots = 8;
    static std::mutex mu;
    static FwdMaps slots[kSlots];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        const FwdMaps& e = slots[i];
        if (e.q == q && e.k == k && e.v == v && e.o == o && e.BH == BH && e.N == N && e.D == D && e.bf16 == bf16) {
            *mq = e.mq;
            *mk = e.mk;
            *mv = e.mv;
            *mo = e.mo;
            return true;
        }
    }
    FwdMaps e{q, k, v, o, BH, N, D, bf16, {}, {}, {}, {}};
    if (!make_map(&e.mq, q, BH, N, D, kBM, bf16) || !make_map(&e.mk, k, BH, N, D, kv_rows, bf16) ||
        !make_map(&e.mv, v, BH, N, D, kv_rows, bf16) || !make_map(&e.mo, o, BH, N, D, kBM, bf16))
        return false;
    slots[next] = e;
    next = (next + 1) % kSlots;
    used = used < kSlots ? used + 1 : kSlots;
    *mq = e.mq;
    *mk = e.mk;
    *mv = e.mv;
    *mo = e.mo;
    return true;
}

template <bool BF16, int D>
int launch_impl(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH,
                int64_t N, bool causal, int num_sms, cudaStream_t stream) {
    constexpr int kSmemBytes = Lay<D>::kSmemBytes;
    // Once per device: the register split assumes the launch allocation (a smaller one could
    // leave the softmax groups waiting for registers forever, so it is refused instead), and the
    // shared-memory grant.
    static uint64_t ready = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    const bool ok = once_per_device(&ready, dev, [] {
        cudaFuncAttributes fattr;
        if (cudaFuncGetAttributes(&fattr, attn_fwd_tc_kernel<BF16, D>) != cudaSuccess || fattr.numRegs < kRegsLaunch) {
            if (std::getenv("ATTN_DEBUG"))
                std::fprintf(stderr, "attn: kernel has %d registers per thread, the register split needs %d\n",
                             fattr.numRegs, kRegsLaunch);
            return false;
        }
        const cudaError_t aerr = cudaFuncSetAttribute(attn_fwd_tc_kernel<BF16, D>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (aerr != cudaSuccess && std::getenv("ATTN_DEBUG"))
            std::fprintf(stderr, "attn: cannot grant %d bytes of shared memory: %s\n", kSmemBytes,
                         cudaGetErrorString(aerr));
        return aerr == cudaSuccess;
    });
    if (!ok) return ATTN_ERR_LAUNCH;
    CUtensorMap mq, mk, mv, mo;
    if (!fwd_maps(q, k, v, o, BH, N, D, Lay<D>::kBN, BF16, &mq, &mk, &mv, &mo)) return ATTN_ERR_DEVICE;
    TcParams prm;
    prm.o = o;
    prm.lse = lse;
    prm.N = static_cast<int>(N);
    prm.BH = static_cast<int>(BH);
    prm.num_pairs = static_cast<int>((N + 2 * kBM - 1) / (2 * kBM));
    prm.causal = causal ? 1 : 0;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    const int64_t blocks = static_cast<int64_t>(prm.num_pairs) * BH;
    if (blocks > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    prm.order_len = 0;
    if (causal && blocks <= kOrderMax && num_sms > 0) {
        // Item pair * BH + head weighs its key-tile steps, max(nA, nB) as the kernel counts them.
        constexpr int BN = Lay<D>::kBN;
        const PlanKey key{0, N, BH, BN, 0};
        const int num_pairs = prm.num_pairs;
        prm.order_len = plan_launch_order(key, kFixedSteps, num_sms, [&] {
            const int nkv = static_cast<int>((N + BN - 1) / BN);
            std::vector<int> w(static_cast<size_t>(blocks));
            for (int pr = 0; pr < num_pairs; ++pr) {
                const int rowA = pr * 2 * kBM, rowB = rowA + kBM;
                const int nA = std::min(nkv, (rowA + kBM - 1) / BN + 1);
                const int nB = rowB < N ? std::min(nkv, (rowB + kBM - 1) / BN + 1) : 0;
                for (int64_t h = 0; h < BH; ++h) w[static_cast<size_t>(pr) * BH + h] = std::max(nA, nB);
            }
            return w;
        }, prm.order);
    }
    attn_fwd_tc_kernel<BF16, D><<<static_cast<unsigned>(blocks), kThreads, kSmemBytes, stream>>>(
        mq, mk, mv, mo, prm);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess && std::getenv("ATTN_DEBUG"))
        std::fprintf(stderr, "attn: tensor-core kernel launch failed: %s\n", cudaGetErrorString(err));
    return err == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH,
                  int64_t N, int64_t d, bool causal, bool bf16, int num_sms, cudaStream_t stream) {
    if (N > 0x7FFFFFFFll - 2 * kBM || BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    if (d == 64)
        return bf16 ? launch_impl<true, 64>(q, k, v, o, lse, BH, N, causal, num_sms, stream)
                    : launch_impl<false, 64>(q, k, v, o, lse, BH, N, causal, num_sms, stream);
    if (d == 128)
        return bf16 ? launch_impl<true, 128>(q, k, v, o, lse, BH, N, causal, num_sms, stream)
                    : launch_impl<false, 128>(q, k, v, o, lse, BH, N, causal, num_sms, stream);
    return ATTN_ERR_UNSUPPORTED;
}

int tc_device_error(cudaStream_t stream, bool clear, unsigned* err) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_DEVICE;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (clear && v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_DEVICE;
    }
    *err = v;
    return ATTN_OK;
}

}  // namespace attn
