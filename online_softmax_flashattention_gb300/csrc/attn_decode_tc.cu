// Key-value cache attention on tcgen05 tensor cores, for 2 or more new queries (bf16 / fp16,
// head width 64 or 128): the same operation and work split as attn_decode.cu (query i at position
// Nk - Nq + i; the keys of a head cut into pieces on different CTAs, merged by their
// log-sum-exps; the "Backwards, and training with it" section of "Flash attention in PyTorch,
// then in Triton" names this generation case and leaves it out of its kernel), with the products
// on tensor cores instead of CUDA cores.
//
// A head's group of up to 128 new queries is one 128-row Q tile (rows past the group zero-filled
// by the tensor map), so S = Q K^T and O += P V are M128 products like the forward's, with every
// padded row wasted; the arithmetic has room for that: a K and V tile pair (32 KB: 128 keys at
// d = 64, 64 at d = 128) takes the SM about 1500 cycles to receive at the HBM rate, the products
// about 600. Softmax warps whose 32 rows are all padding skip the exponentials and write zero
// probabilities.
//
// Pipeline (one CTA per SM, persistent over the pieces of its run): the TMA producer streams the
// pieces' K and V tiles through 4-stage rings and the group's Q tile into one of two buffers; S(g)
// and P(g) are double-buffered in tensor memory by step parity e = g & 1, and softmax warps q and
// q + 4 (the same 32 rows) take the even and the odd steps, each with an online softmax of its own
// (running max, total and output O_e over the key tiles of its parity) that the two merge once per
// piece. With two S and two P buffers the softmax never waits for the products of its own step:
// S(g+2) is computed while step g runs and P(g) is written while PV(g-1) still reads the other
// buffer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_decode_common.cuh"
#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr uint64_t kDrainTimeoutNs = 100000000ull;
constexpr float kLazyLog2 = 8.f;  // keep a stale max until a tile exceeds it by 2^8

__device__ unsigned int g_dtc_error = 0;

constexpr int kThreads = 384;  // warps 0-7 softmax, 8 TMA producer, 9 S issuer (owns TMEM), 10 PV issuer, 11 idle
constexpr int kProducerWarp = 8;
constexpr int kSIssuerWarp = 9;
constexpr int kPVIssuerWarp = 10;
// Register split: launched at 168 a thread (384 x 168 = 64512); the softmax warpgroups rise to
// 216 and the third (TMA, MMA issuers) drops to 72.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSm = 216;
constexpr int kRegsOt = 72;
static_assert(256 * kRegsSm + 128 * kRegsOt <= kThreads * kRegsLaunch, "register split must fit the launch");
constexpr int kQRows = 128;            // queries per group (one Q tile)
constexpr int kBlkQ = 128 * 128;       // one 64-value column block of a Q tile: 128 rows x 128 bytes
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 2;
constexpr int kBarKFull = 4;
constexpr int kBarKEmpty = kBarKFull + kStages;
constexpr int kBarVFull = kBarKEmpty + kStages;
constexpr int kBarVEmpty = kBarVFull + kStages;
constexpr int kBarSFull = kBarVEmpty + kStages;  // [2]
constexpr int kBarSFree = kBarSFull + 2;          // [2] count 4 (the softmax warps of that parity)
constexpr int kBarPFull = kBarSFree + 2;          // [2] count 4
constexpr int kBarPVDone = kBarPFull + 2;         // [2]
constexpr int kBarDrain = kBarPVDone + 2;         // [2] S issuer, PV issuer
constexpr int kBarX = kBarDrain + 2;              // [4] per row quarter: both parities' m, l posted (64 threads)
constexpr int kNumBars = kBarX + 4;

// What depends on the head width D. Keys per tile BN: 128 at d = 64, 64 at d = 128, so that
// S_e (BN fp32 columns), P_e (BN/2) and O_e (D) of both parities fit the 512 TMEM columns
// (512 and 448). Tiles are D/64 column blocks of rows x 128 bytes, one TMA box each. Tensor
// memory: S_e at BN e, P_e at 2 BN + BN/2 e, O_e at 512 - 2 D + D e.
template <int D>
struct DLay {
    static_assert(D == 64 || D == 128, "head width 64 or 128");
    static constexpr int kBN = D == 64 ? 128 : 64;
    static constexpr int kBlocks = D / 64;
    static constexpr int kQTile = kBlocks * kBlkQ;      // 16 or 32 KB
    static constexpr int kKVBlock = kBN * 128;          // one column block of a K or V tile
    static constexpr int kKVTile = kBlocks * kKVBlock;  // 16 KB
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColP = 2 * kBN;
    static constexpr uint32_t kColO = kTmemCols - 2 * D;
    static_assert(kColP + kBN <= kColO, "tensor-memory budget");
    static constexpr int kOffQ = 0;  // two Q buffers
    static constexpr int kOffK = kOffQ + 2 * kQTile;
    static constexpr int kOffV = kOffK + kStages * kKVTile;
    static constexpr int kOffBar = kOffV + kStages * kKVTile;
    // Per-piece exchange of m and l, [piece parity][m | l][step parity][row]: double-buffered by
    // piece so that one barrier a piece suffices (a warp writes a buffer again two pieces later,
    // after its partner's arrival for the piece between, which follows the partner's reads).
    static constexpr int kOffX = kOffBar + 8 * kNumBars;
    static constexpr int kOffSlot = kOffX + 4 * 2 * 2 * 2 * 128;
    static constexpr int kOffAbort = kOffSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // slack to align the base to 1024
    static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
    static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_dtc_error, 1u);
}

// Bounded wait that sleeps inside mbarrier.try_wait (woken when the phase completes).
__device__ __forceinline__ bool wait_s(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// All lanes of a warp wait; the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = wait_s(bar, parity, abort_flag, kWaitTimeoutNs);
    return __all_sync(0xffffffffu, ok);
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

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Row maximum of BN (64 or 128) scores: eight independent chains of 3-input max, then a tree.
template <int BN>
__device__ __forceinline__ float row_max_t(const uint32_t (&su)[BN]) {
    float mx[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
        mx[g] = fmax3(__uint_as_float(su[g]), __uint_as_float(su[g + 8]), __uint_as_float(su[g + 16]));
#pragma unroll
    for (int t = 3; t < BN / 8 - 1; t += 2)
#pragma unroll
        for (int g = 0; g < 8; ++g) mx[g] = fmax3(mx[g], __uint_as_float(su[g + 8 * t]), __uint_as_float(su[g + 8 * t + 8]));
#pragma unroll
    for (int g = 0; g < 8; ++g) mx[g] = fmaxf(mx[g], __uint_as_float(su[g + BN - 8]));
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
}

// One key tile of the online softmax of this thread's query row, for the warps of step parity
// e = g & 1 (global step g of this CTA): waits for S(g), copies it out and (with the other three
// warps of its parity) frees the buffer; once PV(g-2) has finished with P_e and O_e, takes the row
// maximum, moves this parity's reference m when the tile exceeds it by more than 2^8 (rescaling
// O_e; any reference common to l and O gives the same O / l), and writes P(g) = 2^(s c - m) into
// P_e in 32-key pieces. A warp whose rows are all padding (active = false) writes zeros.
template <bool BF16, int D>
__device__ __forceinline__ bool dtc_step(uint32_t tmem_lane, uint32_t bar0, uint32_t g, bool first, bool masked,
                                         bool active, int key0, int limit, float c, float& m, float& l,
                                         volatile int* abort_flag) {
    using L = DLay<D>;
    constexpr int kBN = L::kBN;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    const uint32_t e = g & 1u;
    if (!warp_wait(bar(kBarSFull + static_cast<int>(e)), (g >> 1) & 1u, abort_flag)) return false;
    tc_fence_after();
    uint32_t su[kBN];
    if (active) {
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc)
            ATTN_TMEM_LD_X32(tmem_lane + L::kColS + kBN * e + 32u * cc, (su + 32 * cc));
        tmem_ld_wait();
    }
    tc_fence_before();
    __syncwarp();
    mbar_arrive_elect(bar(kBarSFree + static_cast<int>(e)));
    // P_e and O_e were last used by PV(g-2).
    if (g >= 2 && !warp_wait(bar(kBarPVDone + static_cast<int>(e)), ((g - 2) >> 1) & 1u, abort_flag)) return false;
    tc_fence_after();
    float tile_sum = 0.f;
    if (active) {
        if (masked) {  // warp-uniform
            const int nvalid = limit - key0;
#pragma unroll
            for (int i = 0; i < kBN; ++i) su[i] = (i < nvalid) ? su[i] : 0xFF800000u;
        }
        const float mt = row_max_t<kBN>(su) * c;
        float alpha = 1.f;
        if (mt > m + kLazyLog2) {
            alpha = ex2_approx(m - mt);  // 0 on the first tile (m = -inf)
            m = mt;
            l *= alpha;
        }
        const float m_use = (m == -INFINITY) ? 0.f : m;  // no inf - inf while every key is masked
        const float2 c2 = make_float2(c, c), nm = make_float2(-m_use, -m_use);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < kBN / 32; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k2 = 32 * ch + 2 * i;
                const float2 t = ffma2(make_float2(__uint_as_float(su[k2]), __uint_as_float(su[k2 + 1])), c2, nm);
                const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                acc = fadd2(acc, pp);
                pk[i] = pack2<BF16>(pp.x, pp.y);
            }
            tmem_st_x16(tmem_lane + L::kColP + (kBN / 2) * e + 16u * ch, pk);
        }
        tile_sum = acc.x + acc.y;
        if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O_e <- alpha O_e (rare); PV(g-2), the last product into O_e, is complete.
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
            for (int qq = 0; qq < D / 16; ++qq) {
                uint32_t ou[16];
                tmem_ld_x16(tmem_lane + L::kColO + D * e + 16u * qq, ou);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 v = fmul2(make_float2(__uint_as_float(ou[i]), __uint_as_float(ou[i + 1])), a2);
                    ou[i] = __float_as_uint(v.x);
                    ou[i + 1] = __float_as_uint(v.y);
                }
                tmem_st_x16(tmem_lane + L::kColO + D * e + 16u * qq, ou);
            }
        }
    } else {
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int ch = 0; ch < kBN / 32; ++ch) tmem_st_x16(tmem_lane + L::kColP + (kBN / 2) * e + 16u * ch, z);
    }
    l += tile_sum;
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    mbar_arrive_elect(bar(kBarPFull + static_cast<int>(e)));
    return true;
}

// S = Q K^T: M=128 (queries), N=BN (keys), K=D as D/16 steps of K=16 (32 bytes of a 128-byte
// row; steps 4..7 at D = 128 read the second column block), both operands in shared memory;
// warp-wide (one elected lane issues).
template <bool BF16, int D>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t sQ, uint32_t sK) {
    using L = DLay<D>;
    constexpr uint32_t kIdesc = idesc_f16(BF16, 128, L::kBN, false, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t a_off = static_cast<uint32_t>((kk >> 2) * kBlkQ + 32 * (kk & 3));
        const uint32_t b_off = static_cast<uint32_t>((kk >> 2) * L::kKVBlock + 32 * (kk & 3));
        umma_ss_elect(d_tmem, smem_desc_sw128(sQ + a_off, 16, 1024), smem_desc_sw128(sK + b_off, 16, 1024), kIdesc,
                      kk > 0 ? 1u : 0u);
    }
}

// O_e += P_e V: M=128, N=D, K=BN as BN/16 steps of K=16 (16 keys = 2048 bytes of each column
// block), P from tensor memory, V MN-major (dims contiguous; at D = 128 its two 64-dim column
// blocks are one block apart, the descriptor's leading byte offset).
template <bool BF16, int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t sV, bool accumulate) {
    using L = DLay<D>;
    constexpr uint32_t kIdesc = idesc_f16(BF16, 128, D, false, true);
    constexpr uint32_t kLbo = D == 64 ? 16u : static_cast<uint32_t>(L::kKVBlock);
#pragma unroll
    for (int kk = 0; kk < L::kBN / 16; ++kk)
        umma_ts_elect(o_tmem, p_tmem + 8u * kk, smem_desc_sw128(sV + 2048 * kk, kLbo, 1024), kIdesc,
                      (accumulate || kk > 0) ? 1u : 0u);
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    using L = DLay<D>;
    constexpr int kBN = L::kBN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kOffQ, sK = base + L::kOffK, sV = base + L::kOffV;
    const uint32_t bar0 = base + L::kOffBar;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    float* const xch = reinterpret_cast<float*>(gbase + L::kOffX);  // [piece parity][m | l][step parity][row]
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kOffSlot);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarQFull + i), 1);
            mbar_init(bar(kBarQEmpty + i), 1);
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarSFree + i), 4);
            mbar_init(bar(kBarPFull + i), 4);
            mbar_init(bar(kBarPVDone + i), 1);
            mbar_init(bar(kBarDrain + i), 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarKEmpty + s), 1);
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(kBarX + i), 64);
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
    // Let the merge kernel (launched with programmatic stream serialisation) get onto the GPU
    // now; it waits for this grid to finish before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < 8) {
        // =============================== softmax ===============================
        regs_increase<kRegsSm>();
        const uint32_t q = static_cast<uint32_t>(warp & 3), e = static_cast<uint32_t>(warp >> 2);
        const uint32_t tmem_lane = tmem + ((q * 32u) << 16);
        const int r = static_cast<int>(q) * 32 + lane;  // row of the Q tile
        uint32_t g0 = 0;  // steps of this CTA before the piece
        uint32_t xk = 0;  // exchanges of this row quarter so far
        bool ok = true;
        Piece pc;
        for (int k = 0; ok && get_piece<kQRows, kBN>(p, cta, k, pc); ++k) {
            const int n = pc.t1 - pc.t0;
            const int qi = pc.g0 + r;  // query index within the head
            const int limit = p.causal ? min(p.Nk - p.Nq + qi + 1, p.Nk) : p.Nk;
            // The first row of the group sees the fewest keys: key tiles past its limit hold
            // masked keys for some row and take the masked path.
            const int lim0 = p.causal ? min(p.Nk - p.Nq + pc.g0 + 1, p.Nk) : p.Nk;
            const bool active = static_cast<int>(q) * 32 < pc.ng;
            float m = -INFINITY, l = 0.f;
            const int j0 = static_cast<int>((g0 & 1u) ^ e);  // this parity's first step of the piece
            for (int j = j0; ok && j < n; j += 2) {
                const int key0 = (pc.t0 + j) * kBN;
                ok = dtc_step<BF16, D>(tmem_lane, bar0, g0 + static_cast<uint32_t>(j), j < 2, key0 + kBN > lim0, active,
                                    key0, limit, p.c, m, l, abort_flag);
            }
            if (!ok) break;
            if (active) {
                // ---- merge the two parities, O = (2^(m0-M) O_0 + 2^(m1-M) O_1) / (2^(m0-M) l0 +
                // 2^(m1-M) l1); this thread writes columns D/2 e .. D/2 e + D/2 - 1 of its row. Both
                // warps wait for the piece's last products before the exchange. ----
                if (n >= 1) {
                    const uint32_t gl = g0 + static_cast<uint32_t>(n) - 1;
                    if (!(ok = warp_wait(bar(kBarPVDone + static_cast<int>(gl & 1u)), (gl >> 1) & 1u, abort_flag))) break;
                    if (n >= 2 && !(ok = warp_wait(bar(kBarPVDone + static_cast<int>((gl - 1) & 1u)), ((gl - 1) >> 1) & 1u,
                                                   abort_flag)))
                        break;
                }
                tc_fence_after();
                float* const xb = xch + 512u * (xk & 1u);
                xb[e * 128 + r] = m;
                xb[256 + e * 128 + r] = l;
                mbar_arrive(bar(kBarX + static_cast<int>(q)));
                if (!(ok = warp_wait(bar(kBarX + static_cast<int>(q)), xk & 1u, abort_flag))) break;
                ++xk;
                const float m_o = xb[(e ^ 1u) * 128 + r], l_o = xb[256 + (e ^ 1u) * 128 + r];
                const float M = fmaxf(m, m_o);
                // A parity with no key tile in this piece, or none visible yet, has m = -inf and
                // l = 0; its O buffer holds another piece's values and is not read.
                const bool use_s = m != -INFINITY, use_o = m_o != -INFINITY;
                const float a_s = use_s ? ex2_approx(m - M) : 0.f;
                const float a_o = use_o ? ex2_approx(m_o - M) : 0.f;
                const float lt = l * a_s + l_o * a_o;
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                const float lse2 = lt > 0.f ? M + log2f(lt) : -INFINITY;  // -inf: no visible key in the piece
                const bool use0 = e ? use_o : use_s, use1 = e ? use_s : use_o;
                const float a0 = (e ? a_o : a_s) * inv, a1 = (e ? a_s : a_o) * inv;
                const float2 w0 = make_float2(a0, a0), w1 = make_float2(a1, a1);
                const int64_t row = static_cast<int64_t>(pc.bh) * p.Nq + qi;
                const bool real = r < pc.ng;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t u0[16], u1[16];
                    tmem_ld_x16(tmem_lane + L::kColO + (D / 2) * e + 16u * cc, u0);
                    tmem_ld_x16(tmem_lane + L::kColO + D + (D / 2) * e + 16u * cc, u1);
                    tmem_ld_wait();
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const float2 x0 = use0 ? fmul2(make_float2(__uint_as_float(u0[i]), __uint_as_float(u0[i + 1])), w0)
                                               : make_float2(0.f, 0.f);
                        const float2 xx = use1 ? ffma2(make_float2(__uint_as_float(u1[i]), __uint_as_float(u1[i + 1])), w1, x0)
                                               : x0;
                        x[i] = xx.x;
                        x[i + 1] = xx.y;
                    }
                    if (!real) continue;
                    const int c0 = static_cast<int>((D / 2) * e) + 16 * cc;
                    if (pc.nslots == 1) {
                        uint32_t pk[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) pk[i] = pack2<BF16>(x[2 * i], x[2 * i + 1]);
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row * D + c0);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.part_o + (row * p.P + pc.slot) * D + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                    }
                }
                if (real && e == 0) {
                    if (pc.nslots == 1) {
                        if (p.lse != nullptr) p.lse[row] = lse2;
                    } else {
                        p.part_lse[row * p.P + pc.slot] = lse2;
                    }
                }
                tc_fence_before();
            }
            g0 += static_cast<uint32_t>(n);
        }
        if (!ok) raise_abort(abort_flag);
    } else {
        regs_decrease<kRegsOt>();
    }
    if (warp == kProducerWarp && lane == 0) {
        // ============================ TMA producer ============================
        // Pieces in order: the group's Q tile (pieces with key tiles only) into one of two
        // buffers, then the K tiles into the K ring and, one tile behind, the V tiles.
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        uint32_t kv = 0, vq = 0, qi = 0;
        int pend_bh = -1, pend_t = 0;
        bool ok = true;
        auto issue_v = [&](int bh, int t) -> bool {
            const int s = static_cast<int>(vq % kStages);
            if (!wait_s(bar(kBarVEmpty + s), ((vq / kStages) & 1u) ^ 1u, abort_flag, kWaitTimeoutNs)) return false;
            mbar_arrive_expect_tx(bar(kBarVFull + s), L::kKVTile);
#pragma unroll
            for (int c = 0; c < L::kBlocks; ++c)
                tma_load_3d(sV + s * L::kKVTile + c * L::kKVBlock, &tmap_v, 64 * c, t * kBN, bh, bar(kBarVFull + s));
            ++vq;
            return true;
        };
        Piece pc;
        for (int k = 0; ok && get_piece<kQRows, kBN>(p, cta, k, pc); ++k) {
            if (pc.t1 <= pc.t0) continue;
            const int qb = static_cast<int>(qi & 1u);
            if (!(ok = wait_s(bar(kBarQEmpty + qb), ((qi >> 1) & 1u) ^ 1u, abort_flag, kWaitTimeoutNs))) break;
            mbar_arrive_expect_tx(bar(kBarQFull + qb), L::kQTile);
#pragma unroll
            for (int c = 0; c < L::kBlocks; ++c)
                tma_load_3d(sQ + qb * L::kQTile + c * kBlkQ, &tmap_q, 64 * c, pc.g0, pc.bh, bar(kBarQFull + qb));
            ++qi;
            for (int t = pc.t0; ok && t < pc.t1; ++t) {
                const int s = static_cast<int>(kv % kStages);
                if (!(ok = wait_s(bar(kBarKEmpty + s), ((kv / kStages) & 1u) ^ 1u, abort_flag, kWaitTimeoutNs))) break;
                mbar_arrive_expect_tx(bar(kBarKFull + s), L::kKVTile);
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c)
                    tma_load_3d(sK + s * L::kKVTile + c * L::kKVBlock, &tmap_k, 64 * c, t * kBN, pc.bh,
                                bar(kBarKFull + s));
                ++kv;
                if (pend_bh >= 0 && !(ok = issue_v(pend_bh, pend_t))) break;
                pend_bh = pc.bh;
                pend_t = t;
            }
        }
        if (ok && pend_bh >= 0) ok = issue_v(pend_bh, pend_t);
        if (!ok) raise_abort(abort_flag);
        // Every copy into this CTA must have landed before it may exit; in normal operation the
        // issuers consumed them all already and these waits return at once.
        for (uint32_t i = qi > 2 ? qi - 2 : 0; i < qi; ++i)
            wait_s(bar(kBarQFull + static_cast<int>(i & 1u)), (i >> 1) & 1u, nullptr, kDrainTimeoutNs);
        for (uint32_t i = kv > kStages ? kv - kStages : 0; i < kv; ++i)
            wait_s(bar(kBarKFull + static_cast<int>(i % kStages)), (i / kStages) & 1u, nullptr, kDrainTimeoutNs);
        for (uint32_t i = vq > kStages ? vq - kStages : 0; i < vq; ++i)
            wait_s(bar(kBarVFull + static_cast<int>(i % kStages)), (i / kStages) & 1u, nullptr, kDrainTimeoutNs);
    } else if (warp == kSIssuerWarp) {
        // ============================ S issuer (whole warp) ============================
        // S(g) = Q K^T into the S buffer of parity g & 1 once the key tile has landed and the
        // softmax has copied out S(g-2); each K stage and each Q buffer is released by a commit
        // after the products that read it.
        uint32_t gs = 0, kvs = 0, qs = 0;
        bool ok = true;
        Piece pc;
        for (int k = 0; ok && get_piece<kQRows, kBN>(p, cta, k, pc); ++k) {
            const int n = pc.t1 - pc.t0;
            for (int j = 0; j < n; ++j) {
                const int s = static_cast<int>(kvs % kStages);
                const int qb = static_cast<int>(qs & 1u);
                if (!(ok = warp_wait(bar(kBarKFull + s), (kvs / kStages) & 1u, abort_flag))) break;
                if (j == 0 && !(ok = warp_wait(bar(kBarQFull + qb), (qs >> 1) & 1u, abort_flag))) break;
                if (gs >= 2 &&
                    !(ok = warp_wait(bar(kBarSFree + static_cast<int>(gs & 1u)), ((gs - 2) >> 1) & 1u, abort_flag)))
                    break;
                tc_fence_after();
                issue_s<BF16, D>(tmem + L::kColS + kBN * (gs & 1u), sQ + qb * L::kQTile, sK + s * L::kKVTile);
                umma_commit_elect(bar(kBarSFull + static_cast<int>(gs & 1u)));
                umma_commit_elect(bar(kBarKEmpty + s));
                if (j == n - 1) {
                    umma_commit_elect(bar(kBarQEmpty + qb));
                    ++qs;
                }
                ++gs;
                ++kvs;
            }
        }
        if (!ok) raise_abort(abort_flag);
        umma_commit_elect(bar(kBarDrain + 0));  // no product may still run at teardown
        wait_s(bar(kBarDrain + 0), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
    } else if (warp == kPVIssuerWarp) {
        // ============================ PV issuer (whole warp) ============================
        // O_e += P_e V once the softmax has written P(g) and the value tile has landed; the first
        // product into each O_e of a piece (its step 0 or 1) starts it from zero.
        uint32_t gp = 0, kvp = 0;
        bool ok = true;
        Piece pc;
        for (int k = 0; ok && get_piece<kQRows, kBN>(p, cta, k, pc); ++k) {
            const int n = pc.t1 - pc.t0;
            for (int j = 0; j < n; ++j) {
                const int s = static_cast<int>(kvp % kStages);
                if (!(ok = warp_wait(bar(kBarVFull + s), (kvp / kStages) & 1u, abort_flag))) break;
                if (!(ok = warp_wait(bar(kBarPFull + static_cast<int>(gp & 1u)), (gp >> 1) & 1u, abort_flag))) break;
                tc_fence_after();
                issue_pv<BF16, D>(tmem + L::kColO + D * (gp & 1u), tmem + L::kColP + (kBN / 2) * (gp & 1u),
                                  sV + s * L::kKVTile, j >= 2);
                umma_commit_elect(bar(kBarPVDone + static_cast<int>(gp & 1u)));
                umma_commit_elect(bar(kBarVEmpty + s));
                ++gp;
                ++kvp;
            }
        }
        if (!ok) raise_abort(abort_flag);
        umma_commit_elect(bar(kBarDrain + 1));
        wait_s(bar(kBarDrain + 1), 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kSIssuerWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

namespace {
template <bool BF16, int D>
int launch_tc(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& prm,
              cudaStream_t stream) {
    static uint64_t ready = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (!once_per_device(&ready, dev, [] {
            return cudaFuncSetAttribute(attn_decode_tc_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        DLay<D>::kSmemBytes) == cudaSuccess;
        }))
        return ATTN_ERR_LAUNCH;
    attn_decode_tc_kernel<BF16, D><<<static_cast<unsigned>(prm.C), kThreads, DLay<D>::kSmemBytes, stream>>>(mq, mk, mv,
                                                                                                            prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}
}  // namespace

int launch_decode_tc_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& prm,
                          bool bf16, int d, cudaStream_t stream) {
    if (d == 64)
        return bf16 ? launch_tc<true, 64>(mq, mk, mv, prm, stream) : launch_tc<false, 64>(mq, mk, mv, prm, stream);
    if (d == 128)
        return bf16 ? launch_tc<true, 128>(mq, mk, mv, prm, stream) : launch_tc<false, 128>(mq, mk, mv, prm, stream);
    return ATTN_ERR_UNSUPPORTED;
}

int decode_tc_device_error(bool clear, unsigned* err) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dtc_error, sizeof(v)) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (clear && v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_dtc_error, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_DEVICE;
    }
    *err = v;
    return ATTN_OK;
}

}  // namespace attn
