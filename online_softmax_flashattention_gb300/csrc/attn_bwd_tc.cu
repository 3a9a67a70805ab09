// Backward pass of exact attention for bf16 / fp16 on GB300 (sm_103a) tensor cores.
//
// The gradients follow the "Flash attention in PyTorch, then in Triton" page, section
// "Backwards, and training with it": P is made again from the scores and each row's base-2
// log-sum-exp (lse2 = m + log2 l, kept by the forward), then
//   dV = P^T dO,  dP = dO V^T,  delta_i = sum_e dO[i,e] O[i,e],  dS = P (dP - delta),
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d).
// As on the page the work is split into two kernels so that no program adds into another's
// rows: one CTA per block of 128 keys keeps dK and dV while the blocks of 128 queries that see
// those keys go past; one CTA per block of 128 queries keeps dQ while its key blocks go past.
// Both recompute the scores and dP (the page's trade: no atomics, that work done twice). The
// dQ grid is launched with programmatic stream serialisation: its CTAs take SMs as the dK/dV
// grid's last CTAs finish and wait for that grid only before they write dq.
//
// GB300 mapping. Every product is a tcgen05.mma (bf16/fp16 operands, fp32 accumulate) with
// the forward kernel's two shapes: SS (both operands K-major tiles as TMA writes them, 128-byte
// swizzle) and TS (A from tensor memory, B an MN-major tile).
//   dK/dV kernel, per query block of BQ queries (128 at d = 64, 64 at d = 128), with the keys
//   in the 128 TMEM lanes:
//     S^T = K Q^T (SS), dP^T = V dO^T (SS)               -> TMEM, BQ columns each
//     the eight elementwise warps (thread = key; two warpgroups on the same TMEM lanes, each
//     on half of the block's query columns) make P^T and dS^T = P^T (dP^T - delta) in
//     registers and store them to TMEM as 16-bit pairs
//     dV += P^T dO (TS, B = dO tile MN-major), dK += dS^T Q (TS, B = Q tile MN-major)
//   dQ kernel, per key block, with the queries in the lanes:
//     S = Q K^T (SS), dP = dO V^T (SS); dS = P (dP - delta) -> TMEM; dQ += dS K (TS, B = K)
// Tensor memory (512 columns): dK/dV kernel S^T 0, dP^T BQ, P^T 2 BQ, dS^T 2.5 BQ, dV 3 BQ,
// dK 3 BQ + d (512 columns at d = 64, 448 at d = 128); dQ kernel S 0, dP 128, dS 256, dQ 320. The next block's S and dP products go out as soon as
// the elementwise warps have loaded the current ones into registers, before their arithmetic,
// so the products overlap it.
// delta is made once per query row by a small pre-pass (one 16-byte piece of dO and O per
// lane) and parked in the first four bytes of that row of dq, an output that the dQ kernel
// overwrites last, so the call allocates nothing; the dK/dV kernel's warp 11 copies each
// query block's lse and delta into shared memory a block ahead of their use.
//
// Roles: warps 0-7 elementwise (thread = TMEM lane; warps w and w + 4 share lanes and split the
// columns), warp 8 TMA producer, warp 9 issuer of the S and dP products and tensor-memory
// owner, warp 10 issuer of the products that take P and dS, warp 11 the dK/dV kernel's lse/delta
// loader (idle in the dQ kernel). Every mbarrier wait is bounded; on expiry the kernel sets
// the shared device error word (reported by attn_device_status), drains and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBlk = 128;                   // queries or keys per block = TMEM lanes
constexpr int kBlockBytes = kBlk * 64 * 2;  // 16 KiB: 128 rows x 128 bytes (64 values), one TMA box
// Warps 0-7: elementwise (two warpgroups on the same TMEM lanes, each on half the columns);
// warpgroup 2: the TMA producer (warp 8), the two MMA issuers (warps 9, 10) and the lse/delta
// loader (warp 11). A whole warpgroup there also lets registers move: setmaxnreg acts on whole
// warpgroups, and twelve warps at launch get 168 a thread, so warpgroup 2 gives up to 72 and
// warps 0-7 take 216.
constexpr int kThreads = 384;
constexpr int kElemWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // S and dP products; tensor-memory owner
constexpr int kMma2Warp = 10;  // the products that take P and dS (dV and dK, or dQ)
constexpr int kLoaderWarp = 11;
constexpr int kRegsLaunch = 168;  // 65536 / 384, rounded down to the allocation granule of 8
constexpr int kRegsElem = 216;
constexpr int kRegsOther = 72;
static_assert(32 * kElemWarps * kRegsElem + (kThreads - 32 * kElemWarps) * kRegsOther <= kThreads * kRegsLaunch,
              "the register split must fit in the block's launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr uint64_t kDrainTimeoutNs = 100000000ull;

__device__ unsigned int g_bwd_error = 0;

// Causal calls with at most kOrderMax blocks carry a launch order (block -> item = block
// index * BH + head, planned on the host by plan_launch_order); otherwise the grid runs the
// heaviest blocks first.
constexpr int kOrderMax = 2048;
constexpr int kFixedSteps = 3;  // per-CTA fill and drain, in block steps, for the plan

struct BwdParams {
    void* grad0;  // dk (kv kernel) or dq (q kernel)
    void* grad1;  // dv (kv kernel)
    const uint8_t* delta_rows;  // dq: delta of query row n in the first four bytes of row n
    const float* lse;
    int N;
    int BH;
    int nblk;
    int causal;
    float c;      // log2(e) / sqrt(d)
    float scale;  // 1 / sqrt(d)
    int order_len;  // 0: no table
    uint16_t order[kOrderMax];
};

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
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

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_bwd_error, 1u);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag, kWaitTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}


template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
}

// delta_n = sum_e dO[n,e] O[n,e] (fp32) for every query row n of all heads, stored as the first
// four bytes of dq's row n: dq is an output the call may use as scratch, and the dQ kernel
// reads each row's delta in the CTA that later overwrites that row. D/8 lanes share a row, one
// 16-byte piece of dO and of O each; a warp takes kDeltaUnroll groups of 32 pieces (whole
// rows) per step, all loads issued before the arithmetic.
constexpr int kDeltaUnroll = 4;
template <bool BF16, int D>
__global__ void __launch_bounds__(256)
    attn_bwd_delta_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout, uint8_t* __restrict__ dq,
                          int64_t rows) {
    constexpr int kLanes = D / 8;
    const int64_t total = rows * kLanes;
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g0 = warp_id * 32 * kDeltaUnroll; g0 < total; g0 += nwarps * 32 * kDeltaUnroll) {
        uint4 x[kDeltaUnroll], y[kDeltaUnroll];
#pragma unroll
        for (int u = 0; u < kDeltaUnroll; ++u) {
            const int64_t gi = g0 + 32 * u + lane;  // 16-byte piece gi % kLanes of row gi / kLanes
            x[u] = gi < total ? o[gi] : make_uint4(0, 0, 0, 0);
            y[u] = gi < total ? dout[gi] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kDeltaUnroll; ++u) {
            const int64_t gi = g0 + 32 * u + lane;
            const uint32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w}, ys[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a = unpack2<BF16>(xs[i]), b = unpack2<BF16>(ys[i]);
                acc = fmaf(a.x, b.x, acc);
                acc = fmaf(a.y, b.y, acc);
            }
#pragma unroll
            for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (gi < total && gi % kLanes == 0) *reinterpret_cast<float*>(dq + (gi / kLanes) * (2 * D)) = acc;
        }
    }
}

// 128 x NB product over K = D of two K-major tiles (D/64 column blocks of 128-byte rows each,
// kABlk and kBBlk bytes apart in A and B) into TMEM columns `d`: D/16 steps of K = 16, the ones
// past 64 in the second column block.
template <bool BF16, int D, int NB, int kABlk, int kBBlk, bool kWarp = false>
__device__ __forceinline__ void mma_ss_kmajor(uint32_t d, uint32_t sA, uint32_t sB) {
    constexpr uint32_t kIdesc = idesc_f16(BF16, kBlk, NB, false, false);
    // The steps' descriptors differ only in the start address field (16-byte units).
    const uint64_t a0 = smem_desc_sw128(sA, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(sB, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a = a0 + static_cast<uint64_t>(((kk >> 2) * kABlk + 32 * (kk & 3)) >> 4);
        const uint64_t b = b0 + static_cast<uint64_t>(((kk >> 2) * kBBlk + 32 * (kk & 3)) >> 4);
        if constexpr (kWarp)
            umma_ss_elect(d, a, b, kIdesc, kk > 0 ? 1u : 0u);
        else
            umma_ss(d, a, b, kIdesc, kk > 0 ? 1u : 0u);
    }
}

// 128 x D product over K = 16 KSTEPS with A (128 lanes, K-step kk at column a + 8 kk) in TMEM
// and B an MN-major tile (rows = K, 16 rows = 2048 bytes a step; D/64 column blocks kBBlk bytes
// apart, the descriptor's leading byte offset), accumulated into TMEM columns `d`.
template <bool BF16, int D, int KSTEPS, int kBBlk, bool kWarp = false>
__device__ __forceinline__ void mma_ts_mn(uint32_t d, uint32_t a, uint32_t sB, bool accumulate) {
    constexpr uint32_t kIdesc = idesc_f16(BF16, kBlk, D, false, true);
    constexpr uint32_t kLbo = D == 64 ? 16u : static_cast<uint32_t>(kBBlk);
    const uint64_t b0 = smem_desc_sw128(sB, kLbo, 1024);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint64_t b = b0 + static_cast<uint64_t>((2048 * kk) >> 4);
        if constexpr (kWarp)
            umma_ts_elect(d, a + 8u * kk, b, kIdesc, (accumulate || kk > 0) ? 1u : 0u);
        else
            umma_ts(d, a + 8u * kk, b, kIdesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// An issuer's decision: with kWarp the whole warp runs the issuing loop (elect.sync picks the
// lane that issues), so each lane's result is combined into one and the warp never splits.
template <bool kWarp>
__device__ __forceinline__ bool issuer_vote(bool v) {
    if constexpr (kWarp) return __all_sync(0xffffffffu, v);
    return v;
}
template <bool kWarp>
__device__ __forceinline__ void issuer_commit(uint32_t bar) {
    if constexpr (kWarp)
        umma_commit_elect(bar);
    else
        umma_commit(bar);
}

// TMA copy of one tile of a [BH][N][D] tensor: D/64 boxes of 64 values (the map's box rows),
// landing kColBlk bytes apart.
template <int D, int kColBlk>
__device__ __forceinline__ void tma_tile(uint32_t dst, const void* map, int row, int bh, uint32_t bar) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * kColBlk, map, 64 * c, row, bh, bar);
}

// ================================ dK, dV: one CTA per key block ================================
// The query blocks that go past the CTA's 128 keys hold BQ queries: 128 at d = 64, 64 at
// d = 128, so that S^T, dP^T (BQ columns each), P^T, dS^T (BQ/2 each), dV and dK (d each) fit
// the 512 tensor-memory columns side by side (512 and 448) and the next block's S^T, dP^T never
// wait for this block's dV, dK products.
// Shared memory: K, V tiles, then a 4-stage ring of (Q, dO) tiles, then per-block lse and delta
// (double-buffered by block parity, filled by warp 11 from lse and from the delta pre-pass),
// then mbarriers.

template <int D>
struct KvLay {
    static constexpr int kBQ = D == 64 ? 128 : 64;     // queries per query block
    static constexpr int kChunks = kBQ / 64;           // 32-query chunks per elementwise warpgroup
    static constexpr int kTile = kBlk * D * 2;          // K or V tile
    static constexpr int kTileQ = kBQ * D * 2;          // Q or dO tile
    static constexpr int kQBlockBytes = kBQ * 128;      // one 64-value column block of a Q or dO tile
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTile;
    static constexpr int kOffStage = 2 * kTile;  // stage s: Q at +0, dO at +kTileQ
    static constexpr int kStageBytes = 2 * kTileQ;
    static constexpr int kStages = 4;
    static constexpr int kOffRow = kOffStage + kStages * kStageBytes;  // lse[2][BQ], delta[2][BQ] floats
    static constexpr int kOffBar = kOffRow + 4 * kBQ * 4;
    // Barriers: K and V landed; per stage full / empty; S^T and dP^T written (one commit after
    // both products); S^T and dP^T read out; P^T and dS^T written; dV, dK products done; the final drain; per row buffer: lse and
    // delta written / read.
    static constexpr int kKV = 0, kQFull = 1, kQEmpty = kQFull + kStages, kDPFull = kQEmpty + kStages,
                         kSdPFree = kDPFull + 1, kPdSFull = kDPFull + 2, kDone = kDPFull + 3,
                         kDrain = kDPFull + 4, kRowsFull = kDPFull + 5, kRowsEmpty = kRowsFull + 2,
                         kDrain2 = kRowsEmpty + 2, kNumBars = kDrain2 + 1;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
    static constexpr int kOffAbort = kOffSlot + 4;
    static constexpr int kSmem = kOffAbort + 4 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kColS = 0, kColDP = kBQ, kColP = 2 * kBQ, kColDS = 2 * kBQ + kBQ / 2;
    static constexpr uint32_t kColDV = 3 * kBQ, kColDK = 3 * kBQ + D;
    static_assert(kColDK + D <= kTmemCols, "tensor-memory budget");
};

// One 32-query chunk of the dK/dV kernel's elementwise step for this thread's key: P^T and
// dS^T = P^T (dP^T - delta) from this thread's row of S^T and dP^T, as 16-bit pairs. The
// queries' lse and delta come from shared memory, negated, four at a time; the arithmetic runs
// on query pairs with the f32x2 forms (each lane rounds as the scalar operation would).
template <bool BF16, bool kMasked>
__device__ __forceinline__ void kv_chunk(int ch, const uint32_t (&s)[32], const uint32_t (&dp)[32], const float* nls,
                                         const float* ndl, float c, int key, int q0, int N, int causal,
                                         uint32_t (&pp)[16], uint32_t (&ds)[16]) {
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int u4 = 0; u4 < 8; ++u4) {
        const float4 lv = *reinterpret_cast<const float4*>(nls + ch * 32 + 4 * u4);
        const float4 dv4 = *reinterpret_cast<const float4*>(ndl + ch * 32 + 4 * u4);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 4 * u4 + 2 * h;
            const float2 x = ffma2(make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), c2,
                                   h == 0 ? make_float2(lv.x, lv.y) : make_float2(lv.z, lv.w));
            float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if constexpr (kMasked) {
                const int query = q0 + ch * 32 + e;
                if (!(query < N && key < N && (!causal || key <= query))) pr.x = 0.f;
                if (!(query + 1 < N && key < N && (!causal || key <= query + 1))) pr.y = 0.f;
            }
            const float2 dd = fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                    h == 0 ? make_float2(dv4.x, dv4.y) : make_float2(dv4.z, dv4.w));
            const float2 dsv = fmul2(pr, dd);
            pp[2 * u4 + h] = pack2<BF16>(pr.x, pr.y);
            ds[2 * u4 + h] = pack2<BF16>(dsv.x, dsv.y);
        }
    }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            const BwdParams p) {
    using L = KvLay<D>;
    constexpr int kTile = L::kTile;
    // Which issuers run as a whole converged warp (elect.sync issues, operands in uniform
    // registers) rather than as one lane. Measured (B1 H12 N8192 causal, L2 flushed, outputs
    // bit-identical): the dV/dK issuer warp-wide at D = 64, 808 -> 851 TFLOP/s for the pair of
    // grids (N4096 non-causal 701 -> 742); at D = 128 no gain (882 -> 879); the S^T/dP^T issuer
    // warp-wide lost at both widths (795, 845).
    constexpr bool kWarpA = false;
    constexpr bool kWarpB = D == 64;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kOffSlot);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);
    constexpr int BQ = L::kBQ;
    float* const lse_s = reinterpret_cast<float*>(gbase + L::kOffRow);  // [2][BQ], negated
    float* const delta_s = lse_s + 2 * BQ;                                // [2][BQ], negated

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N;
    const int item = p.order_len > 0 ? p.order[blockIdx.x] : static_cast<int>(blockIdx.x);
    const int bh = item % p.BH;
    const int kblk = item / p.BH;  // without a table, block 0 (which sees most queries) goes first
    const int k0 = kblk * kBlk;
    const int qb0 = p.causal ? k0 / BQ : 0;  // the first query block that sees these keys
    const int nq = (N + BQ - 1) / BQ - qb0;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kKV), 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar(L::kQFull + s), 1);
            mbar_init(bar(L::kQEmpty + s), 1);
        }
        mbar_init(bar(L::kDPFull), 1);
        mbar_init(bar(L::kSdPFree), kElemWarps);
        mbar_init(bar(L::kPdSFull), kElemWarps);
        mbar_init(bar(L::kDone), 1);
        mbar_init(bar(L::kDrain), 1);
        mbar_init(bar(L::kDrain2), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::kRowsFull + b), 1);
            mbar_init(bar(L::kRowsEmpty + b), kElemWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The dQ kernel may take SMs as this grid's last CTAs finish; it waits for this grid before it
    // writes dq, whose rows hold the delta values read here.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kElemWarps) {
        // ===================== elementwise warps: thread = key (TMEM lane) =====================
        regs_increase<kRegsElem>();
        const int g = warp >> 2;  // warpgroup: query chunks g kChunks .. (g + 1) kChunks - 1
        const int r = ((warp & 3) << 5) + lane;  // key row within the block, = TMEM lane
        const int key = k0 + r;
        const uint32_t t = tmem + (static_cast<uint32_t>((warp & 3) << 5) << 16);
        bool ok = true;
        for (int i = 0; ok && i < nq; ++i) {
            const int rb = i & 1, q0 = (qb0 + i) * BQ;
            if (!(ok = warp_wait(bar(L::kRowsFull + rb), (i >> 1) & 1, abort_flag))) break;
            const float* ls = lse_s + rb * BQ;
            const float* dl = delta_s + rb * BQ;
            if (!(ok = warp_wait(bar(L::kDPFull), i & 1, abort_flag))) break;
            tc_fence_after();
            // This warpgroup's chunks of S^T and dP^T into registers, then they are released so
            // that the next block's products run during the arithmetic below.
            constexpr int NC = L::kChunks;
            uint32_t sv[NC][32], dpv[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                ATTN_TMEM_LD_X32(t + L::kColS + 32 * (g * NC + c), sv[c]);
                ATTN_TMEM_LD_X32(t + L::kColDP + 32 * (g * NC + c), dpv[c]);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kSdPFree));
            // Only query blocks that reach below the keys' last row (causal) and ragged edges
            // need a mask.
            const bool masked = (p.causal && q0 < k0 + kBlk) || q0 + BQ > N || k0 + kBlk > N;
            uint32_t ppv[NC][16], dsv[NC][16];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if (masked)
                    kv_chunk<BF16, true>(g * NC + c, sv[c], dpv[c], ls, dl, p.c, key, q0, N, p.causal, ppv[c], dsv[c]);
                else
                    kv_chunk<BF16, false>(g * NC + c, sv[c], dpv[c], ls, dl, p.c, key, q0, N, p.causal, ppv[c], dsv[c]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kRowsEmpty + rb));
            // The previous block's dV/dK products read P^T and dS^T: wait only now, before
            // overwriting them, so that those products run under the arithmetic above.
            if (i > 0 && !(ok = warp_wait(bar(L::kDone), (i - 1) & 1, abort_flag))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                tmem_st_x16(t + L::kColP + 16 * (g * NC + c), ppv[c]);
                tmem_st_x16(t + L::kColDS + 16 * (g * NC + c), dsv[c]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kPdSFull));
        }
        // ---- epilogue: dK * scale (warpgroup 0) and dV (warpgroup 1), rounded; keys >= N not stored ----
        if (ok && nq > 0) {
            if ((ok = warp_wait(bar(L::kDone), (nq - 1) & 1, abort_flag))) {
                tc_fence_after();
                uint16_t* const dst = reinterpret_cast<uint16_t*>(g == 0 ? p.grad0 : p.grad1) +
                                      (static_cast<int64_t>(bh) * N + key) * D;
                const float sc = g == 0 ? p.scale : 1.f;
                const uint32_t col = g == 0 ? L::kColDK : L::kColDV;
#pragma unroll 1
                for (int h = 0; h < D / 16; ++h) {
                    uint32_t a[16];
                    tmem_ld_x16(t + col + 16 * h, a);
                    tmem_ld_wait();
                    uint32_t pa[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        pa[j] = pack2<BF16>(__uint_as_float(a[2 * j]) * sc, __uint_as_float(a[2 * j + 1]) * sc);
                    if (key < N) {
                        uint4* x = reinterpret_cast<uint4*>(dst + 16 * h);
                        x[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                        x[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
                    }
                }
            }
        }
        if (!ok) raise_abort(abort_flag);
    } else {
        regs_decrease<kRegsOther>();
        if (warp == kProducerWarp && lane == 0) {
            // =============================== TMA producer ===============================
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(bar(L::kKV), 2 * kTile);
            tma_tile<D, kBlockBytes>(base + L::kOffK, &tm_k, k0, bh, bar(L::kKV));
            tma_tile<D, kBlockBytes>(base + L::kOffV, &tm_v, k0, bh, bar(L::kKV));
            bool ok = true;
            int issued = 0;
            for (int i = 0; i < nq; ++i) {
                const int st = i % L::kStages, q0 = (qb0 + i) * BQ;
                if (!(ok = mbar_wait(bar(L::kQEmpty + st), ((i / L::kStages) & 1) ^ 1, abort_flag, kWaitTimeoutNs)))
                    break;
                const uint32_t stage = base + L::kOffStage + st * L::kStageBytes;
                mbar_arrive_expect_tx(bar(L::kQFull + st), L::kStageBytes);
                tma_tile<D, L::kQBlockBytes>(stage, &tm_q, q0, bh, bar(L::kQFull + st));
                tma_tile<D, L::kQBlockBytes>(stage + L::kTileQ, &tm_do, q0, bh, bar(L::kQFull + st));
                issued = i + 1;
            }
            if (!ok) raise_abort(abort_flag);
            // Every copy must land before the CTA exits (normally they were all consumed).
            mbar_wait(bar(L::kKV), 0, nullptr, kDrainTimeoutNs);
            for (int i = (issued > L::kStages ? issued - L::kStages : 0); i < issued; ++i)
                mbar_wait(bar(L::kQFull + i % L::kStages), (i / L::kStages) & 1, nullptr, kDrainTimeoutNs);
        } else if (warp == kMmaWarp && (kWarpA || lane == 0)) {
            // ============================ MMA issuer: S^T, dP^T ============================
            // S^T(0), dP^T(0); then block i+1's once block i's were copied out (d = 128: once
            // block i's dV, dK products are done, as P^T and dS^T sit over S^T and dP^T). The
            // products that take P^T and dS^T come from another warp: a thread's barrier waits
            // queue behind the tensor-core instructions it issued before, so one issuer would
            // let the pipe drain at every hand-off.
            bool ok = issuer_vote<kWarpA>(mbar_wait(bar(L::kKV), 0, abort_flag, kWaitTimeoutNs));
            // Block i's (Q, dO) tiles are waited for before the release of block i-1's S^T and
            // dP^T, which comes last: the products then go out one barrier test after it.
            auto wait_tiles = [&](int i) {
                return issuer_vote<kWarpA>(
                    mbar_wait(bar(L::kQFull + i % L::kStages), (i / L::kStages) & 1, abort_flag, kWaitTimeoutNs));
            };
            auto issue_sdp = [&](int i) {
                const uint32_t stage = base + L::kOffStage + (i % L::kStages) * L::kStageBytes;
                tc_fence_after();
                mma_ss_kmajor<BF16, D, BQ, kBlockBytes, L::kQBlockBytes, kWarpA>(tmem + L::kColS, base + L::kOffK,
                                                                                 stage);  // S^T = K Q^T
                mma_ss_kmajor<BF16, D, BQ, kBlockBytes, L::kQBlockBytes, kWarpA>(tmem + L::kColDP, base + L::kOffV,
                                                                                 stage + L::kTileQ);  // dP^T = V dO^T
                issuer_commit<kWarpA>(bar(L::kDPFull));
            };
            if (ok && nq > 0 && (ok = wait_tiles(0))) issue_sdp(0);
            for (int i = 0; ok && i + 1 < nq; ++i) {
                if (!(ok = wait_tiles(i + 1))) break;
                if (!(ok = issuer_vote<kWarpA>(mbar_wait(bar(L::kSdPFree), i & 1, abort_flag, kWaitTimeoutNs)))) break;
                issue_sdp(i + 1);
            }
            if (!ok && lane == 0) raise_abort(abort_flag);
            issuer_commit<kWarpA>(bar(L::kDrain));
            mbar_wait(bar(L::kDrain), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        } else if (warp == kMma2Warp && (kWarpB || lane == 0)) {
            // ============================ MMA issuer: dV, dK ============================
            // dV, dK += block i's P^T dO, dS^T Q once P^T and dS^T are in TMEM (block i's
            // S^T, dP^T products are then done, so the stage's tiles have landed).
            bool ok = true;
            for (int i = 0; ok && i < nq; ++i) {
                if (!(ok = issuer_vote<kWarpB>(mbar_wait(bar(L::kPdSFull), i & 1, abort_flag, kWaitTimeoutNs)))) break;
                tc_fence_after();
                const uint32_t stage = base + L::kOffStage + (i % L::kStages) * L::kStageBytes;
                mma_ts_mn<BF16, D, BQ / 16, L::kQBlockBytes, kWarpB>(tmem + L::kColDV, tmem + L::kColP, stage + L::kTileQ,
                                                                     i > 0);  // dV += P^T dO
                mma_ts_mn<BF16, D, BQ / 16, L::kQBlockBytes, kWarpB>(tmem + L::kColDK, tmem + L::kColDS, stage,
                                                                     i > 0);  // dK += dS^T Q
                issuer_commit<kWarpB>(bar(L::kDone));
                issuer_commit<kWarpB>(bar(L::kQEmpty + i % L::kStages));
            }
            if (!ok && lane == 0) raise_abort(abort_flag);
            issuer_commit<kWarpB>(bar(L::kDrain2));
            mbar_wait(bar(L::kDrain2), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        } else if (warp == kLoaderWarp) {
            // ==================== warp 11: each query block's lse and delta ====================
            // into the row buffer the elementwise warps released two blocks ago, so the global
            // loads run a block ahead of their use.
            bool ok = true;
            for (int i = 0; i < nq; ++i) {
                const int rb = i & 1, q0 = (qb0 + i) * BQ;
                if (!(ok = warp_wait(bar(L::kRowsEmpty + rb), ((i >> 1) & 1) ^ 1, abort_flag))) break;
#pragma unroll
                for (int u = lane; u < BQ; u += 32) {
                    const int q = q0 + u;
                    float l2 = 0.f, dl = 0.f;
                    if (q < N) {
                        const int64_t row = static_cast<int64_t>(bh) * N + q;
                        l2 = p.lse[row];
                        dl = *reinterpret_cast<const float*>(p.delta_rows + row * (2 * D));
                    }
                    lse_s[rb * BQ + u] = -l2;
                    delta_s[rb * BQ + u] = -dl;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kRowsFull + rb));
            }
            if (!ok) raise_abort(abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ================================== dQ: one CTA per query block ==================================
// Shared memory: Q and dO tiles, then a ring of (K, V) stages (three at d = 64, two at d = 128).
// Tensor memory: S 0, dP 128, dS 256 (64 columns), dQ 320 (d columns).
enum { qQ = 0, qKVFull = 1 };

template <int D>
struct QLay {
    static constexpr int kTile = kBlk * D * 2;
    static constexpr int kStages = D == 64 ? 3 : 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kTile;
    static constexpr int kOffKV = 2 * kTile;  // stage s: K at +0, V at +kTile
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kOffBar = kOffKV + kStages * kStageBytes;
    static constexpr int kKVEmpty = qKVFull + kStages;
    // kDPFull: S and dP written (one commit after both products).
    static constexpr int kDPFull = kKVEmpty + kStages;
    static constexpr int kSdPFree = kDPFull + 1, kDSFull = kDPFull + 2, kDone = kDPFull + 3, kDrain = kDPFull + 4,
                         kDrain2 = kDPFull + 5, kNumBars = kDPFull + 6;
    static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
    static constexpr int kOffAbort = kOffSlot + 4;
    static constexpr int kSmem = kOffAbort + 4 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 320;
};

// One 32-key chunk of the dQ kernel's elementwise step for this thread's query: dS = P (dP -
// delta) from this thread's row of S and dP, as 16-bit pairs.
template <bool BF16, bool kMasked>
__device__ __forceinline__ void q_chunk(int ch, const uint32_t (&s)[32], const uint32_t (&dp)[32], float l2, float delta,
                                        float c, int query, int k0, int N, int causal, uint32_t (&ds)[16]) {
    const float2 c2 = make_float2(c, c), nl2 = make_float2(-l2, -l2), nd2 = make_float2(-delta, -delta);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const float2 x = ffma2(make_float2(__uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1])), c2, nl2);
        float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if constexpr (kMasked) {
            const int key = k0 + ch * 32 + 2 * u;
            if (!(query < N && key < N && (!causal || key <= query))) pr.x = 0.f;
            if (!(query < N && key + 1 < N && (!causal || key + 1 <= query))) pr.y = 0.f;
        }
        const float2 dsv =
            fmul2(pr, fadd2(make_float2(__uint_as_float(dp[2 * u]), __uint_as_float(dp[2 * u + 1])), nd2));
        ds[u] = pack2<BF16>(dsv.x, dsv.y);
    }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const BwdParams p) {
    using L = QLay<D>;
    constexpr int kTile = L::kTile;
    constexpr int S = L::kStages;
    // As in the dK/dV kernel: the dQ issuer warp-wide at D = 64, the S/dP issuer one lane.
    constexpr bool kWarpA = false;
    constexpr bool kWarpB = D == 64;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    auto bar = [&](int i) -> uint32_t { return base + L::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kOffSlot);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N;
    const int item = p.order_len > 0 ? p.order[blockIdx.x] : static_cast<int>(blockIdx.x);
    const int bh = item % p.BH;
    const int slot = item / p.BH;
    const int qblk = p.causal ? (p.nblk - 1 - slot) : slot;  // without a table, heaviest causal blocks first
    const int q0 = qblk * kBlk;
    const int nk = p.causal ? qblk + 1 : p.nblk;  // keys up to the block's last query

    if (threadIdx.x == 0) {
        mbar_init(bar(qQ), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(qKVFull + s), 1);
            mbar_init(bar(L::kKVEmpty + s), 1);
        }
        mbar_init(bar(L::kDPFull), 1);
        mbar_init(bar(L::kSdPFree), kElemWarps);
        mbar_init(bar(L::kDSFull), kElemWarps);
        mbar_init(bar(L::kDone), 1);
        mbar_init(bar(L::kDrain), 1);
        mbar_init(bar(L::kDrain2), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kElemWarps) {
        // ==================== elementwise warps: thread = query (TMEM lane) ====================
        regs_increase<kRegsElem>();
        const int g = warp >> 2;  // warpgroup: key columns 64g .. 64g + 63
        const int r = ((warp & 3) << 5) + lane;
        const int query = q0 + r;
        const bool qin = query < N;
        const uint32_t t = tmem + (static_cast<uint32_t>((warp & 3) << 5) << 16);
        bool ok = true;
        // This row's delta (from the pre-pass, in the row's own dq bytes, which only this CTA's
        // epilogue overwrites, after every elementwise warp has passed this point) and lse.
        float delta = 0.f, l2 = 0.f;
        if (qin) {
            const int64_t row = static_cast<int64_t>(bh) * N + query;
            delta = *reinterpret_cast<const float*>(p.delta_rows + row * (2 * D));
            l2 = p.lse[row];
        }
        for (int j = 0; ok && j < nk; ++j) {
            const int k0 = j * kBlk;
            if (!(ok = warp_wait(bar(L::kDPFull), j & 1, abort_flag))) break;
            tc_fence_after();
            // This warpgroup's two chunks of S and dP into registers, released before the
            // arithmetic so the next block's products overlap it.
            uint32_t s0[32], dp0[32], s1[32], dp1[32];
            ATTN_TMEM_LD_X32(t + L::kColS + 64 * g, s0);
            ATTN_TMEM_LD_X32(t + L::kColDP + 64 * g, dp0);
            ATTN_TMEM_LD_X32(t + L::kColS + 64 * g + 32, s1);
            ATTN_TMEM_LD_X32(t + L::kColDP + 64 * g + 32, dp1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kSdPFree));
            const bool masked = (p.causal && j == qblk) || q0 + kBlk > N || k0 + kBlk > N;
            uint32_t ds0[16], ds1[16];
            if (masked) {
                q_chunk<BF16, true>(2 * g, s0, dp0, l2, delta, p.c, query, k0, N, p.causal, ds0);
                q_chunk<BF16, true>(2 * g + 1, s1, dp1, l2, delta, p.c, query, k0, N, p.causal, ds1);
            } else {
                q_chunk<BF16, false>(2 * g, s0, dp0, l2, delta, p.c, query, k0, N, p.causal, ds0);
                q_chunk<BF16, false>(2 * g + 1, s1, dp1, l2, delta, p.c, query, k0, N, p.causal, ds1);
            }
            // The previous block's dQ product reads dS: wait only now, before overwriting it.
            if (j > 0 && !(ok = warp_wait(bar(L::kDone), (j - 1) & 1, abort_flag))) break;
            tc_fence_after();
            tmem_st_x16(t + L::kColDS + 32 * g, ds0);
            tmem_st_x16(t + L::kColDS + 32 * g + 16, ds1);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kDSFull));
        }
        // ---- epilogue: dQ * scale (warpgroup g: dims D/2 g .. D/2 (g + 1) - 1), rounded; rows >= N not stored ----
        if (ok && nk > 0) {
            if ((ok = warp_wait(bar(L::kDone), (nk - 1) & 1, abort_flag))) {
                tc_fence_after();
                // dq's rows hold the delta values the dK/dV grid reads: wait for that grid to
                // complete (launched with programmatic serialisation, this grid may start before).
                asm volatile("griddepcontrol.wait;" ::: "memory");
                uint16_t* const dq = reinterpret_cast<uint16_t*>(p.grad0) + (static_cast<int64_t>(bh) * N + query) * D;
#pragma unroll 1
                for (int h = g * (D / 32); h < (g + 1) * (D / 32); ++h) {
                    uint32_t a[16];
                    tmem_ld_x16(t + L::kColDQ + 16 * h, a);
                    tmem_ld_wait();
                    uint32_t pa[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pa[i] = pack2<BF16>(__uint_as_float(a[2 * i]) * p.scale, __uint_as_float(a[2 * i + 1]) * p.scale);
                    if (qin) {
                        uint4* x = reinterpret_cast<uint4*>(dq + 16 * h);
                        x[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                        x[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
                    }
                }
            }
        }
        if (!ok) raise_abort(abort_flag);
    } else {
        regs_decrease<kRegsOther>();
        if (warp == kProducerWarp && lane == 0) {
            // =============================== TMA producer ===============================
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(bar(qQ), 2 * kTile);
            tma_tile<D, kBlockBytes>(base + L::kOffQ, &tm_q, q0, bh, bar(qQ));
            tma_tile<D, kBlockBytes>(base + L::kOffDO, &tm_do, q0, bh, bar(qQ));
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < nk; ++j) {
                const int st = j % S;
                if (!(ok = mbar_wait(bar(L::kKVEmpty + st), ((j / S) & 1) ^ 1, abort_flag, kWaitTimeoutNs))) break;
                const uint32_t stage = base + L::kOffKV + st * L::kStageBytes;
                mbar_arrive_expect_tx(bar(qKVFull + st), 2 * kTile);
                tma_tile<D, kBlockBytes>(stage, &tm_k, j * kBlk, bh, bar(qKVFull + st));
                tma_tile<D, kBlockBytes>(stage + kTile, &tm_v, j * kBlk, bh, bar(qKVFull + st));
                issued = j + 1;
            }
            if (!ok) raise_abort(abort_flag);
            mbar_wait(bar(qQ), 0, nullptr, kDrainTimeoutNs);
            for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
                mbar_wait(bar(qKVFull + j % S), (j / S) & 1, nullptr, kDrainTimeoutNs);
        } else if (warp == kMmaWarp && (kWarpA || lane == 0)) {
            // ============================= MMA issuer: S, dP =============================
            // S(0), dP(0); then key block j+1's once block j's were copied out. dQ comes from
            // another warp (see the dK/dV kernel).
            bool ok = issuer_vote<kWarpA>(mbar_wait(bar(qQ), 0, abort_flag, kWaitTimeoutNs));
            // Key block j's tiles are waited for before the release of block j-1's S and dP (as
            // in the dK/dV kernel).
            auto wait_tiles = [&](int j) {
                return issuer_vote<kWarpA>(mbar_wait(bar(qKVFull + j % S), (j / S) & 1, abort_flag, kWaitTimeoutNs));
            };
            auto issue_sdp = [&](int j) {
                const uint32_t stage = base + L::kOffKV + (j % S) * L::kStageBytes;
                tc_fence_after();
                mma_ss_kmajor<BF16, D, kBlk, kBlockBytes, kBlockBytes, kWarpA>(tmem + L::kColS, base + L::kOffQ,
                                                                               stage);  // S = Q K^T
                mma_ss_kmajor<BF16, D, kBlk, kBlockBytes, kBlockBytes, kWarpA>(tmem + L::kColDP, base + L::kOffDO,
                                                                               stage + kTile);  // dP = dO V^T
                issuer_commit<kWarpA>(bar(L::kDPFull));
            };
            if (ok && nk > 0 && (ok = wait_tiles(0))) issue_sdp(0);
            for (int j = 0; ok && j + 1 < nk; ++j) {
                if (!(ok = wait_tiles(j + 1))) break;
                if (!(ok = issuer_vote<kWarpA>(mbar_wait(bar(L::kSdPFree), j & 1, abort_flag, kWaitTimeoutNs)))) break;
                issue_sdp(j + 1);
            }
            if (!ok && lane == 0) raise_abort(abort_flag);
            issuer_commit<kWarpA>(bar(L::kDrain));
            mbar_wait(bar(L::kDrain), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        } else if (warp == kMma2Warp && (kWarpB || lane == 0)) {
            // ============================== MMA issuer: dQ ==============================
            // dQ += dS K once block j's dS is in TMEM (its S, dP products are then done).
            bool ok = true;
            for (int j = 0; ok && j < nk; ++j) {
                if (!(ok = issuer_vote<kWarpB>(mbar_wait(bar(L::kDSFull), j & 1, abort_flag, kWaitTimeoutNs)))) break;
                tc_fence_after();
                const uint32_t stage = base + L::kOffKV + (j % S) * L::kStageBytes;
                mma_ts_mn<BF16, D, kBlk / 16, kBlockBytes, kWarpB>(tmem + L::kColDQ, tmem + L::kColDS, stage,
                                                                   j > 0);  // dQ += dS K
                issuer_commit<kWarpB>(bar(L::kDone));
                issuer_commit<kWarpB>(bar(L::kKVEmpty + j % S));
            }
            if (!ok && lane == 0) raise_abort(abort_flag);
            issuer_commit<kWarpB>(bar(L::kDrain2));
            mbar_wait(bar(L::kDrain2), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------ host side ------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// [BH][N][D] 16-bit tensor; boxes of 128 rows x 64 values (128 bytes, the swizzle span), one per
// 64-value column block; rows past N of a head are out of bounds (zero-filled), never the next
// head's.
bool make_map(CUtensorMap* map, const void* ptr, int64_t BH, int64_t N, int64_t D, bool bf16, int rows = kBlk) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(N) * D * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BF16, int D>
int launch_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int64_t BH, int64_t N, bool causal, int num_sms, cudaStream_t stream) {
    // The dQ kernel takes 128-row tiles of everything; the dK/dV kernel takes its Q and dO tiles
    // in query blocks of KvLay<D>::kBQ rows.
    constexpr int kBQ = KvLay<D>::kBQ;
    CUtensorMap mq, mk, mv, mdo, mqb, mdob;
    if (!make_map(&mq, q, BH, N, D, BF16) || !make_map(&mk, k, BH, N, D, BF16) || !make_map(&mv, v, BH, N, D, BF16) ||
        !make_map(&mdo, dout, BH, N, D, BF16) || !make_map(&mqb, q, BH, N, D, BF16, kBQ) ||
        !make_map(&mdob, dout, BH, N, D, BF16, kBQ))
        return ATTN_ERR_DEVICE;
    static uint64_t ready = 0;  // shared-memory grants, once per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (!once_per_device(&ready, dev, [] {
            return cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        KvLay<D>::kSmem) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        QLay<D>::kSmem) == cudaSuccess;
        }))
        return ATTN_ERR_LAUNCH;
    BwdParams prm;
    prm.delta_rows = static_cast<const uint8_t*>(dq);
    prm.lse = lse;
    prm.N = static_cast<int>(N);
    prm.BH = static_cast<int>(BH);
    prm.nblk = static_cast<int>((N + kBlk - 1) / kBlk);
    prm.causal = causal ? 1 : 0;
    prm.c = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    prm.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    const int64_t blocks = static_cast<int64_t>(prm.nblk) * BH;
    if (blocks > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    // delta of every query row into dq's rows, then dK/dV, then dQ (which overwrites them).
    const int64_t rows = BH * N;
    const int64_t pieces = rows * (D / 8);
    const unsigned dblocks =
        static_cast<unsigned>(std::min<int64_t>((pieces + 256 * kDeltaUnroll - 1) / (256 * kDeltaUnroll), 2048));
    attn_bwd_delta_kernel<BF16, D><<<dblocks, 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dout), static_cast<uint8_t*>(dq), rows);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    // Launch orders (causal calls up to kOrderMax blocks): dK/dV item kblk * BH + head weighs its
    // query blocks, dQ item slot * BH + head its key blocks.
    const bool plan = causal && blocks <= kOrderMax && num_sms > 0;
    prm.order_len = 0;
    const int nblk = prm.nblk;
    if (plan) {
        prm.order_len = plan_launch_order(PlanKey{1, N, BH, D, 0}, kFixedSteps, num_sms, [&] {
            const int nqb = static_cast<int>((N + kBQ - 1) / kBQ);
            std::vector<int> w(static_cast<size_t>(blocks));
            for (int kb = 0; kb < nblk; ++kb)
                for (int64_t h = 0; h < BH; ++h) w[static_cast<size_t>(kb) * BH + h] = nqb - kb * kBlk / kBQ;
            return w;
        }, prm.order);
    }
    prm.grad0 = dk;
    prm.grad1 = dv;
    attn_bwd_dkdv_tc_kernel<BF16, D><<<static_cast<unsigned>(blocks), kThreads, KvLay<D>::kSmem, stream>>>(
        mqb, mk, mv, mdob, prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    prm.grad0 = dq;
    prm.grad1 = nullptr;
    if (plan) {
        prm.order_len = plan_launch_order(PlanKey{2, N, BH, D, 0}, kFixedSteps, num_sms, [&] {
            std::vector<int> w(static_cast<size_t>(blocks));
            for (int sl = 0; sl < nblk; ++sl)
                for (int64_t h = 0; h < BH; ++h) w[static_cast<size_t>(sl) * BH + h] = nblk - sl;
            return w;
        }, prm.order);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = QLay<D>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_bwd_dq_tc_kernel<BF16, D>, mq, mk, mv, mdo, prm) == cudaSuccess ? ATTN_OK
                                                                                                : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, int64_t BH, int64_t N, int64_t d, bool causal, bool bf16,
                  int num_sms, cudaStream_t stream) {
    if (N > 0x7FFFFFFFll - kBlk || BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    if (d == 64)
        return bf16 ? launch_impl<true, 64>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, num_sms, stream)
                    : launch_impl<false, 64>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, num_sms, stream);
    if (d == 128)
        return bf16 ? launch_impl<true, 128>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, num_sms, stream)
                    : launch_impl<false, 128>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, num_sms, stream);
    return ATTN_ERR_UNSUPPORTED;
}

int bwd_tc_device_error(bool clear, unsigned* err) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof(v)) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (clear && v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_DEVICE;
    }
    *err = v;
    return ATTN_OK;
}

}  // namespace attn
