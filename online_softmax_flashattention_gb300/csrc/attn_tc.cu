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
// ("A kernel in Triton": the kernel keeps its scores times log two e), and the
// probabilities are rounded to the input type before they weigh v so the tensor cores can
// take them (same section). Causal tiles past a query tile's last row are skipped
// (section "The online softmax, in PyTorch"); ragged N is masked on keys and clipped on
// stores.
//
// GB300 mapping (a fresh design; the pages' kernels target sm_75 CUDA cores and a Triton
// kernel on sm_89):
//   * One CTA owns two query tiles A and B of 128 rows (rows 256c .. 256c+255 of one head)
//     and streams K/V tiles of 128 keys past both, so each K/V tile is fetched once for
//     256 queries.
//   * Warp 8 issues TMA loads (128-byte swizzle) into a 3-stage K/V ring guarded by
//     full/empty mbarriers. Warp 9 owns the tensor memory and issues every tcgen05.mma from
//     one thread. Warps 0-3 (tile A) and 4-7 (tile B) are the softmax warpgroups: thread t
//     of a group owns query row t, which is TMEM lane t, so row reductions need no shuffles.
//   * Tensor memory (512 columns x 128 lanes x 32 bit): S_A, S_B fp32 scores (128 columns
//     each), O_A, O_B fp32 outputs (64 each), P_A, P_B probabilities as 16-bit pairs (64
//     each). S = Q K^T runs with both operands in shared memory; O += P V takes P from
//     tensor memory and V (dims contiguous, "MN-major") from shared memory.
//   * The MMA thread issues S_X(j+1) as soon as softmax X has copied S_X(j) into registers,
//     so the next QK^T overlaps the exponentials; while one group is in its softmax the
//     tensor core works on the other group's products.
//   * Every mbarrier wait is bounded. A wait that exceeds its deadline sets the device
//     error word and an abort flag; all roles then leave their loops, drain copies and MMAs
//     still in flight (with a deadline of their own), free tensor memory and return.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kD = 64;
constexpr int kBM = 128;  // query rows per tile = TMEM lanes
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kStages = 3;
constexpr int kTileBytes = kBM * kD * 2;  // 16 KiB per 128 x 64 tile of 16-bit values
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // + 128 * tile
constexpr uint32_t kColO = 256;  // + 64 * tile
constexpr uint32_t kColP = 384;  // + 64 * tile
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s for any single wait
constexpr uint64_t kDrainTimeoutNs = 100000000ull;  // 100 ms to drain after an abort

// Shared-memory layout (byte offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;                                   // 2 tiles
constexpr int kOffK = kOffQ + 2 * kTileBytes;              // kStages tiles
constexpr int kOffV = kOffK + kStages * kTileBytes;        // kStages tiles
constexpr int kOffBar = kOffV + kStages * kTileBytes;      // mbarriers, 8 bytes each
// barrier indices
constexpr int kBarQFull = 0;
constexpr int kBarKFull = 1;
constexpr int kBarVFull = kBarKFull + kStages;
constexpr int kBarKvEmpty = kBarVFull + kStages;
constexpr int kBarSFull = kBarKvEmpty + kStages;  // 2
constexpr int kBarSFree = kBarSFull + 2;          // 2
constexpr int kBarPFull = kBarSFree + 2;          // 2
constexpr int kBarOReady = kBarPFull + 2;         // 2
constexpr int kBarMmaDone = kBarOReady + 2;
constexpr int kNumBars = kBarMmaDone + 1;
constexpr int kOffSlot = kOffBar + 8 * kNumBars;  // TMEM base address written by tcgen05.alloc
constexpr int kOffAbort = kOffSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms need 1024-byte alignment");

__device__ unsigned int g_tc_error = 0;

struct TcParams {
    void* o;
    int N;
    int BH;
    int num_pairs;
    int causal;
    float scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_tc_error, 1u);
}

// All lanes of a warp wait; the result is the same in every lane, so a warp never splits
// in front of a warp-collective tcgen05.ld / tcgen05.st.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag, kWaitTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);

    const uint32_t sQ = base + kOffQ;
    const uint32_t sK = base + kOffK;
    const uint32_t sV = base + kOffV;
    auto bar = [&](int i) -> uint32_t { return base + kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffSlot);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + kOffAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: pair of query tiles (A, B) of head bh; heaviest causal pairs first ----
    const int N = p.N;
    const int bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.BH));
    const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.BH));
    const int pair = p.causal ? (p.num_pairs - 1 - slot) : slot;
    const int rowA = pair * 2 * kBM;
    const int rowB = rowA + kBM;
    const int nkv = (N + kBN - 1) / kBN;
    const int nA = p.causal ? min(nkv, rowA / kBN + 1) : nkv;
    const int nB = (rowB < N) ? (p.causal ? min(nkv, rowB / kBN + 1) : nkv) : 0;
    const int nmax = max(nA, nB);

    // ---- setup: barriers (thread 0), tensor memory (MMA warp) ----
    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQFull), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarKvEmpty + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(kBarSFull + x), 1);
            mbar_init(bar(kBarSFree + x), 4);
            mbar_init(bar(kBarPFull + x), 4);
            mbar_init(bar(kBarOReady + x), 1);
        }
        mbar_init(bar(kBarMmaDone), 1);
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

    if (warp < 8) {
        // =========================== softmax warpgroups ===========================
        const int X = warp >> 2;
        const int nX = X ? nB : nA;
        const int r0 = X ? rowB : rowA;
        const int trow = ((warp & 3) << 5) + lane;
        const int row = r0 + trow;
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) << 5) << 16;
        const uint32_t tS = tmem + lane_addr + kColS + 128u * X;
        const uint32_t tO = tmem + lane_addr + kColO + 64u * X;
        const uint32_t tP = tmem + lane_addr + kColP + 64u * X;
        const float c = p.scale_log2;
        const int limit = p.causal ? min(row + 1, N) : N;  // keys >= limit are masked

        float m = -INFINITY;  // running max of scaled scores (base-2 units)
        float l = 0.f;        // running denominator, relative to m
        bool ok = true;
        for (int j = 0; j < nX; ++j) {
            if (!warp_wait(bar(kBarSFull + X), j & 1, abort_flag)) {
                raise_abort(abort_flag);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t su[kBN];
            ATTN_TMEM_LD_X32(tS + 0, (su + 0));
            ATTN_TMEM_LD_X32(tS + 32, (su + 32));
            ATTN_TMEM_LD_X32(tS + 64, (su + 64));
            ATTN_TMEM_LD_X32(tS + 96, (su + 96));
            tmem_ld_wait();
            float s[kBN];
#pragma unroll
            for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(su[i]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + X));

            const int kbase = j * kBN;
            if (kbase + kBN > limit || kbase + kBN > N) {
#pragma unroll
                for (int i = 0; i < kBN; ++i)
                    if (kbase + i >= limit) s[i] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int i = 1; i + 1 < kBN; i += 2) mx = fmax3(mx, s[i], s[i + 1]);
            mx = fmaxf(mx, s[kBN - 1]);
            const float m_new = fmaxf(m, mx * c);
            // A row with every key masked so far keeps a zero reference so no inf - inf occurs.
            const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2_approx(m - m_ref);
            const float neg = -m_ref;

            bool rescale = false;
            if (j > 0) {
                // O and P are still in use by the previous PV product until it completes.
                if (!warp_wait(bar(kBarOReady + X), (j - 1) & 1, abort_flag)) {
                    raise_abort(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                rescale = __any_sync(0xffffffffu, alpha != 1.f);
            }
            float rs = 0.f;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2_approx(fmaf(s[32 * h + 2 * i], c, neg));
                    const float p1 = ex2_approx(fmaf(s[32 * h + 2 * i + 1], c, neg));
                    rs += p0 + p1;
                    pk[i] = pack2<BF16>(p0, p1);
                }
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,"
                    "%10,%11,%12,%13,%14,%15,%16};" ::"r"(tP + 16 * h),
                    "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]),
                    "r"(pk[6]), "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]),
                    "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
                    : "memory");
            }
            if (rescale) {
                // O <- alpha * O, after the scores are spent so both never occupy registers.
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ou[32];
                    ATTN_TMEM_LD_X32(tO + 32 * h, ou);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ou[i] = __float_as_uint(__uint_as_float(ou[i]) * alpha);
                    ATTN_TMEM_ST_X32(tO + 32 * h, ou);
                }
            }
            l = l * alpha + rs;
            m = m_ref;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPFull + X));
        }

        // ---- epilogue: O / l, rounded to the output type, rows >= N not stored ----
        if (ok && nX > 0) {
            if (warp_wait(bar(kBarOReady + X), (nX - 1) & 1, abort_flag)) {
                tc_fence_after();
                const float inv = 1.f / l;
                using elem = uint16_t;
                elem* const orow = reinterpret_cast<elem*>(p.o) +
                                   (static_cast<int64_t>(bh) * N + row) * kD;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ou[32];
                    ATTN_TMEM_LD_X32(tO + 32 * h, ou);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack2<BF16>(__uint_as_float(ou[2 * i]) * inv,
                                            __uint_as_float(ou[2 * i + 1]) * inv);
                    if (row < N) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * h);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            } else {
                raise_abort(abort_flag);
            }
        }
    } else if (warp == kProducerWarp) {
        // =============================== TMA producer ===============================
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(bar(kBarQFull), (nB > 0 ? 2 : 1) * kTileBytes);
            tma_load_3d(sQ, &tmap_q, 0, rowA, bh, bar(kBarQFull));
            if (nB > 0) tma_load_3d(sQ + kTileBytes, &tmap_q, 0, rowB, bh, bar(kBarQFull));
            int issued = 0;
            for (int j = 0; j < nmax; ++j) {
                const int s = j % kStages;
                if (!mbar_wait(bar(kBarKvEmpty + s), ((j / kStages) & 1) ^ 1, abort_flag,
                               kWaitTimeoutNs)) {
                    raise_abort(abort_flag);
                    break;
                }
                mbar_arrive_expect_tx(bar(kBarKFull + s), kTileBytes);
                tma_load_3d(sK + s * kTileBytes, &tmap_k, 0, j * kBN, bh, bar(kBarKFull + s));
                mbar_arrive_expect_tx(bar(kBarVFull + s), kTileBytes);
                tma_load_3d(sV + s * kTileBytes, &tmap_v, 0, j * kBN, bh, bar(kBarVFull + s));
                issued = j + 1;
            }
            // Every copy issued must have landed before the CTA may exit. In normal operation
            // they were all consumed already and these waits return at once.
            mbar_wait(bar(kBarQFull), 0, nullptr, kDrainTimeoutNs);
            for (int j = max(0, issued - kStages); j < issued; ++j) {
                const int s = j % kStages;
                mbar_wait(bar(kBarKFull + s), (j / kStages) & 1, nullptr, kDrainTimeoutNs);
                mbar_wait(bar(kBarVFull + s), (j / kStages) & 1, nullptr, kDrainTimeoutNs);
            }
        }
    } else {
        // ================================ MMA issuer ================================
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_f16(BF16, kBM, kBN, false, false);
            constexpr uint32_t kIdescPV = idesc_f16(BF16, kBM, kD, false, true);
            bool ok = mbar_wait(bar(kBarQFull), 0, abort_flag, kWaitTimeoutNs);
            bool issued_any = false;

            // S_X(j) = Q_X K_j^T : M=128, N=128, K=64 as four K=16 steps (32 bytes each)
            auto issue_s = [&](int X, int j) {
                const int s = j % kStages;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(sQ + X * kTileBytes + 32 * kk, 16, 1024);
                    const uint64_t b = smem_desc_sw128(sK + s * kTileBytes + 32 * kk, 16, 1024);
                    umma_ss(tmem + kColS + 128u * X, a, b, kIdescQK, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(kBarSFull + X));
                issued_any = true;
            };
            // O_X += P_X V_j : M=128, N=64, K=128 as eight K=16 steps (16 keys = 2048 bytes of V)
            auto issue_pv = [&](int X, int j) {
                const int s = j % kStages;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(sV + s * kTileBytes + 2048 * kk, 16, 1024);
                    umma_ts(tmem + kColO + 64u * X, tmem + kColP + 64u * X + 8u * kk, b, kIdescPV,
                            (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(kBarOReady + X));
                issued_any = true;
            };

            if (ok && nmax > 0) {
                ok = mbar_wait(bar(kBarKFull + 0), 0, abort_flag, kWaitTimeoutNs);
                if (ok) {
                    tc_fence_after();
                    if (nA > 0) issue_s(0, 0);
                    if (nB > 0) issue_s(1, 0);
                }
            }
            for (int j = 0; ok && j < nmax; ++j) {
                const int s = j % kStages;
                const int s1 = (j + 1) % kStages;
                for (int X = 0; X < 2 && ok; ++X) {
                    if (j + 1 < (X ? nB : nA)) {
                        ok = mbar_wait(bar(kBarKFull + s1), ((j + 1) / kStages) & 1, abort_flag,
                                       kWaitTimeoutNs) &&
                             mbar_wait(bar(kBarSFree + X), j & 1, abort_flag, kWaitTimeoutNs);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(X, j + 1);
                    }
                    if (j < (X ? nB : nA)) {
                        ok = mbar_wait(bar(kBarVFull + s), (j / kStages) & 1, abort_flag,
                                       kWaitTimeoutNs) &&
                             mbar_wait(bar(kBarPFull + X), j & 1, abort_flag, kWaitTimeoutNs);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(X, j);
                    }
                }
                if (ok) umma_commit(bar(kBarKvEmpty + s));
            }
            if (!ok) raise_abort(abort_flag);
            // No MMA may still be running when the tensor memory is released.
            if (issued_any) {
                umma_commit(bar(kBarMmaDone));
                mbar_wait(bar(kBarMmaDone), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
            }
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

// [BH][N][64] 16-bit tensor; boxes of 128 rows x 64 values (128 bytes, the swizzle span).
bool make_map(CUtensorMap* map, const void* ptr, int64_t BH, int64_t N, bool bf16) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                   static_cast<cuuint64_t>(N) * kD * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kBM), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BF16>
int launch_impl(const void* q, const void* k, const void* v, void* o, int64_t BH, int64_t N,
                bool causal, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, BH, N, BF16) || !make_map(&mk, k, BH, N, BF16) ||
        !make_map(&mv, v, BH, N, BF16))
        return ATTN_ERR_DEVICE;
    // The attribute is per device; setting it on every call is cheap and thread-safe.
    if (cudaFuncSetAttribute(attn_fwd_tc_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
        return ATTN_ERR_LAUNCH;
    TcParams prm;
    prm.o = o;
    prm.N = static_cast<int>(N);
    prm.BH = static_cast<int>(BH);
    prm.num_pairs = static_cast<int>((N + 2 * kBM - 1) / (2 * kBM));
    prm.causal = causal ? 1 : 0;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
    const int64_t blocks = static_cast<int64_t>(prm.num_pairs) * BH;
    if (blocks > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    attn_fwd_tc_kernel<BF16><<<static_cast<unsigned>(blocks), kThreads, kSmemBytes, stream>>>(
        mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, int64_t BH, int64_t N,
                  bool causal, bool bf16, int /*num_sms*/, cudaStream_t stream) {
    if (N > 0x7FFFFFFFll - 2 * kBM || BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    return bf16 ? launch_impl<true>(q, k, v, o, BH, N, causal, stream)
                : launch_impl<false>(q, k, v, o, BH, N, causal, stream);
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
