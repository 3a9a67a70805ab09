// Key-value cache attention (decode): Nq new queries, the last Nq positions of a sequence,
// against Nk >= Nq cached keys and values, with the key range cut into pieces that run on
// different CTAs and are merged by their log-sum-exps.
//
// The "Flash attention in PyTorch, then in Triton" page names this case and leaves it out of
// its kernel (section "Backwards, and training with it": generation with a cache, where a few
// new tokens attend to every cached key). Query i sits at position Nk - Nq + i; when causal it
// sees keys 0 .. Nk - Nq + i. Each piece runs the page's online softmax (section "Flash
// attention": a running maximum, denominator and output per query, rescaled when a tile raises
// the maximum) over its keys and leaves (O_p / l_p, lse2_p = m_p + log2 l_p); the merge kernel
// combines the pieces the way the online softmax combines tiles:
//     lse2 = log2 sum_p 2^lse2_p,   O = sum_p 2^(lse2_p - lse2) O_p.
// A query does one product of d terms per cached row of 2d values, so the work is bound by
// reading the cache from HBM. This file's kernel streams K and V once per group of up to eight
// queries through a ring of shared-memory stages filled by TMA, with the arithmetic on CUDA
// cores; it serves one new query, fp32, and everything the tensor-core kernel does not take.
// Two or more 16-bit queries go to attn_decode_tc.cu (groups of up to 128 queries as M128
// tensor-core tiles) under the same work split and the same merge kernel.
//
// Work split. The queries are cut into groups of QG (1, 2, 4 or 8 here, 128 on tensor cores);
// a segment is one (head, query group) with Tn tiles of ROWS keys (128 here; 128 or 64 on
// tensor cores). Two ways to cut segments into pieces:
//   balanced (num_splits == 0): the grid is persistent (as many CTAs as fit on the GPU, or
//     fewer when there is less work) and CTA c takes the contiguous run of tiles
//     [c G / C, (c+1) G / C) of all G = segments * Tn tiles, cut at segment boundaries, so
//     every CTA streams the same number of tiles (within one) whatever B*H is;
//   explicit (num_splits = S >= 1): every segment is cut into S equal shares, handed out to
//     the CTAs round robin.
// A piece that covers a whole segment writes o and lse directly; the others write fp32
// partials to the workspace for the merge kernel.
//
// CTA layout: four consumer warps and one producer warp. The producer's first lane walks the
// same pieces as the consumers and, per tile, waits for a free stage and issues the K and V
// tile loads (128 rows x 64 values, 128-byte swizzle; fp32 rows are two 32-value halves).
// Consumer warp w takes rows 32w .. 32w+31 of each tile, one key per lane: scores against the
// group's queries (pre-scaled by log2(e)/sqrt(d), in warp-private shared memory), a warp-wide
// online update per query, then the weighted values with lane L owning dims 2L, 2L+1 and the
// probabilities read back from shared memory. At the end of a piece the four warps' states
// merge through shared memory. Every wait is bounded: on a timeout the kernel records an
// error, stops, and the producer waits for its loads in flight before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "attn_decode_common.cuh"
#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr uint64_t kDrainTimeoutNs = 100000000ull;

__device__ unsigned int g_decode_error = 0;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Per element type and head width D (64 or 128): consumer warps (32 keys each, so a tile holds
// 32 * kCW keys), ring depth, and how many 128-byte boxes make one row. Every configuration
// keeps about 192 KB of loads in flight per SM (two CTAs of 96 KB, or one of 192 KB).
template <typename T, int D>
struct Cfg {
    static constexpr int kEsz = static_cast<int>(sizeof(T));
    static constexpr int kCW = (kEsz == 4 && D == 128) ? 2 : 4;
    static constexpr int kStages = 3;
    static constexpr int kRows = 32 * kCW;
    static constexpr int kThreads = 32 * (kCW + 1);
    static constexpr int kBoxes = D * kEsz / 128;   // boxes per row (128 bytes each)
    static constexpr int kBoxElems = 128 / kEsz;    // elements in a box row
    static constexpr int kChunkElems = 16 / kEsz;   // elements in a 16-byte chunk
    static constexpr int kDL = D / 32;              // output dims per lane
    static constexpr int kBoxBytes = kRows * 128;   // one box of a tile
    static constexpr int kTileBytes = kRows * D * kEsz;  // one of K, V
    static constexpr int kStageBytes = 2 * kTileBytes;
};

// N consecutive values (N * sizeof(T) bytes: 4, 8 or 16, naturally aligned) as fp32.
template <typename T, int N>
__device__ __forceinline__ void to_f32(const uint8_t* p, float (&f)[N]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (N == 2) {
            const float2 x = *reinterpret_cast<const float2*>(p);
            f[0] = x.x; f[1] = x.y;
        } else {
            static_assert(N == 4, "2 or 4 fp32 values");
            const float4 x = *reinterpret_cast<const float4*>(p);
            f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
        }
    } else {
        uint32_t w[N / 2];
        if constexpr (N == 2) {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        } else if constexpr (N == 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(p);
            w[0] = x.x; w[1] = x.y;
        } else {
            static_assert(N == 8, "2, 4 or 8 16-bit values");
            const uint4 x = *reinterpret_cast<const uint4*>(p);
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        }
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                f[2 * i] = h.x;
                f[2 * i + 1] = h.y;
            }
        }
    }
}

// Two consecutive values from global memory as fp32, and two fp32 stored as T.
template <typename T>
__device__ __forceinline__ float2 load2(const T* p);
template <>
__device__ __forceinline__ float2 load2<float>(const float* p) { return *reinterpret_cast<const float2*>(p); }
template <>
__device__ __forceinline__ float2 load2<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <>
__device__ __forceinline__ float2 load2<__half>(const __half* p) {
    return __half22float2(*reinterpret_cast<const __half2*>(p));
}

template <typename T>
__device__ __forceinline__ void store2(T* p, float a, float b);
template <>
__device__ __forceinline__ void store2<float>(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
template <>
__device__ __forceinline__ void store2<__half>(__half* p, float a, float b) {
    *reinterpret_cast<__half2*>(p) = __floats2half2_rn(a, b);
}

template <typename T, int QG, int D>
struct Smem {
    using C = Cfg<T, D>;
    static constexpr int kRing = C::kStages * C::kStageBytes;
    static constexpr int kQs = kRing;                      // [kCW][QG][D] f32
    static constexpr int kPs = kQs + C::kCW * QG * D * 4;  // [kCW][QG][32] f32
    static constexpr int kMl = kPs + C::kCW * QG * 32 * 4; // [kCW][QG] m, then [kCW][QG] l
    static constexpr int kBars = kMl + 2 * C::kCW * QG * 4;  // full[S], empty[S], mFull, mFree
    static constexpr int kAbort = kBars + (2 * C::kStages + 2) * 8;
    static constexpr int kBytes = kAbort + 16;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
    static_assert(kAlloc <= 227 * 1024, "shared memory budget of one CTA");
};

__device__ __forceinline__ void raise_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_decode_error, 1u);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag, kWaitTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

// Byte offset of the 16-byte chunk `ch` of row r in a box of 128-byte rows written with the
// 128-byte swizzle (the chunks of a row are permuted by row % 8).
__device__ __forceinline__ uint32_t sw_chunk(int r, int ch) {
    return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
}

template <typename T, int QG, int D>
__global__ void __launch_bounds__(Cfg<T, D>::kThreads)
    attn_decode_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                       const DecodeParams p) {
    using C = Cfg<T, D>;
    using L = Smem<T, QG, D>;
    constexpr int S = C::kStages;
    constexpr int kCW = C::kCW;
    constexpr int kRows = C::kRows;
    constexpr int DL = C::kDL;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    auto full = [&](int s) { return base + L::kBars + 8 * s; };
    auto empty = [&](int s) { return base + L::kBars + 8 * (S + s); };
    const uint32_t mFull = base + L::kBars + 8 * (2 * S), mFree = mFull + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCW);
        }
        mbar_init(mFull, kCW);
        mbar_init(mFree, kCW);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32 * kCW) {
        prefetch_tmap(&mk);
        prefetch_tmap(&mv);
    }
    __syncthreads();
    // Let the merge kernel (launched with programmatic stream serialisation) get onto the GPU
    // now; it waits for this grid to finish before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int cta = blockIdx.x;

    if (warp == kCW) {
        // ------------------------------------ producer ------------------------------------
        if (lane != 0) return;
        int nt = 0;  // tiles issued by this CTA
        bool ok = true;
        Piece pc;
        for (int k = 0; ok && get_piece<QG, kRows>(p, cta, k, pc); ++k) {
            for (int t = pc.t0; t < pc.t1; ++t, ++nt) {
                const int s = nt % S;
                if (!(ok = mbar_wait(empty(s), ((nt / S) & 1) ^ 1, abort_flag, kWaitTimeoutNs))) break;
                const uint32_t dst = base + s * C::kStageBytes;
                mbar_arrive_expect_tx(full(s), C::kStageBytes);
#pragma unroll
                for (int h = 0; h < C::kBoxes; ++h) {
                    tma_load_3d(dst + h * C::kBoxBytes, &mk, h * C::kBoxElems, t * kRows, pc.bh, full(s));
                    tma_load_3d(dst + C::kTileBytes + h * C::kBoxBytes, &mv, h * C::kBoxElems, t * kRows, pc.bh,
                                full(s));
                }
            }
        }
        if (!ok) raise_abort(abort_flag);
        // Wait for the loads still in flight so that none lands after the CTA has exited.
        for (int u = max(0, nt - S); u < nt; ++u)
            mbar_wait(full(u % S), (u / S) & 1, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        return;
    }

    // ------------------------------------ consumers ------------------------------------
    float* qs = reinterpret_cast<float*>(smem + L::kQs) + warp * QG * D;  // this warp's queries, scaled
    float* ps = reinterpret_cast<float*>(smem + L::kPs) + warp * QG * 32;  // this warp's probabilities
    float* ml = reinterpret_cast<float*>(smem + L::kMl);                    // m [kCW][QG], l [kCW][QG]
    const int tid = threadIdx.x;  // 0 .. 32*kCW - 1
    // Lane L owns output dims e0 .. e0 + DL - 1, inside box vb at element ve of its row.
    const int e0 = DL * lane;
    const int vb = e0 / C::kBoxElems, ve = e0 % C::kBoxElems;
    const int vch = ve / C::kChunkElems, vbyte = (ve % C::kChunkElems) * C::kEsz;
    int nt = 0;  // tiles consumed by this CTA
    bool ok = true;
    Piece pc;
    for (int k = 0; get_piece<QG, kRows>(p, cta, k, pc); ++k) {
        // The previous piece's merge read every warp's qs; wait until all are done with it.
        if (k > 0 && !(ok = warp_wait(mFree, (k - 1) & 1, abort_flag))) break;
        {
            const T* qh = static_cast<const T*>(p.q) + (static_cast<int64_t>(pc.bh) * p.Nq + pc.g0) * D;
#pragma unroll
            for (int i = 0; i < QG; ++i) {
#pragma unroll
                for (int h = 0; h < DL; h += 2) {
                    float2 x = make_float2(0.f, 0.f);
                    if (i < pc.ng) x = load2<T>(qh + i * D + e0 + h);
                    *reinterpret_cast<float2*>(qs + i * D + e0 + h) = make_float2(x.x * p.c, x.y * p.c);
                }
            }
            __syncwarp();
        }
        float m[QG], l[QG], acc[QG][DL];
#pragma unroll
        for (int i = 0; i < QG; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
#pragma unroll
            for (int h = 0; h < DL; ++h) acc[i][h] = 0.f;
        }
        const int qpos0 = p.Nk - p.Nq + pc.g0;  // position of the group's first query
        for (int t = pc.t0; t < pc.t1; ++t, ++nt) {
            const int s = nt % S;
            if (!(ok = warp_wait(full(s), (nt / S) & 1, abort_flag))) break;
            const uint8_t* kt = smem + s * C::kStageBytes;
            const uint8_t* vt = kt + C::kTileBytes;
            const int r = 32 * warp + lane;
            const int j = t * kRows + r;
            // ---- scores of key j against the group's queries ----
            // Pairs of dims on the f32x2 FMA, q read four dims at a time; NA2 pairs of
            // independent partial sums per query.
            constexpr int NA2 = QG == 1 ? 2 : 1;
            float2 sa[QG][NA2];
#pragma unroll
            for (int i = 0; i < QG; ++i)
#pragma unroll
                for (int a = 0; a < NA2; ++a) sa[i][a] = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < C::kBoxes; ++h) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float kf[C::kChunkElems];
                    to_f32<T, C::kChunkElems>(kt + h * C::kBoxBytes + sw_chunk(r, ch), kf);
                    const int e = h * C::kBoxElems + ch * C::kChunkElems;  // first dim of the chunk
#pragma unroll
                    for (int i = 0; i < QG; ++i) {
#pragma unroll
                        for (int u = 0; u < C::kChunkElems; u += 4) {
                            const float4 qv = *reinterpret_cast<const float4*>(qs + i * D + e + u);
                            float2& a0 = sa[i][(u / 4) % NA2];
                            a0 = ffma2(make_float2(qv.x, qv.y), make_float2(kf[u], kf[u + 1]), a0);
                            a0 = ffma2(make_float2(qv.z, qv.w), make_float2(kf[u + 2], kf[u + 3]), a0);
                        }
                    }
                }
            }
            // ---- online update per query, probabilities to shared memory ----
#pragma unroll
            for (int i = 0; i < QG; ++i) {
                float sc = 0.f;
#pragma unroll
                for (int a = 0; a < NA2; ++a) sc += sa[i][a].x + sa[i][a].y;
                const bool vis = j < pc.ke && i < pc.ng && (!p.causal || j <= qpos0 + i);
                sc = vis ? sc : -INFINITY;
                float mx = sc;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(m[i], mx);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no inf - inf on empty rows
                const float alpha = ex2f(m[i] - m_use);
                const float pr = ex2f(sc - m_use);
                l[i] = fmaf(l[i], alpha, pr);  // this lane's share of the row total
#pragma unroll
                for (int h = 0; h < DL; h += 2) {
                    const float2 v = fmul2(make_float2(acc[i][h], acc[i][h + 1]), make_float2(alpha, alpha));
                    acc[i][h] = v.x;
                    acc[i][h + 1] = v.y;
                }
                m[i] = m_new;
                ps[i * 32 + lane] = pr;
            }
            __syncwarp();
            // ---- weighted values: lane L owns dims e0 .. e0 + DL - 1 ----
            const int nk = min(32, pc.ke - (t * kRows + 32 * warp));  // rows of this warp with a visible key
#pragma unroll
            for (int k4 = 0; k4 < 32; k4 += 4) {
                if (k4 >= nk) break;
                float4 pp[QG];
#pragma unroll
                for (int i = 0; i < QG; ++i) pp[i] = *reinterpret_cast<const float4*>(ps + i * 32 + k4);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int rr = 32 * warp + k4 + u;
                    float vv[DL];
                    to_f32<T, DL>(vt + vb * C::kBoxBytes + sw_chunk(rr, vch) + vbyte, vv);
#pragma unroll
                    for (int i = 0; i < QG; ++i) {
                        const float w = u == 0 ? pp[i].x : u == 1 ? pp[i].y : u == 2 ? pp[i].z : pp[i].w;
#pragma unroll
                        for (int h = 0; h < DL; h += 2) {
                            const float2 v = ffma2(make_float2(w, w), make_float2(vv[h], vv[h + 1]),
                                                   make_float2(acc[i][h], acc[i][h + 1]));
                            acc[i][h] = v.x;
                            acc[i][h + 1] = v.y;
                        }
                    }
                }
            }
            __syncwarp();
            mbar_arrive_elect(empty(s));
        }
        if (!ok) break;
        // ---- merge the warps' states: this warp's O into its qs, m and l beside ----
#pragma unroll
        for (int i = 0; i < QG; ++i) {
            float tl = l[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tl += __shfl_xor_sync(0xffffffffu, tl, off);
#pragma unroll
            for (int h = 0; h < DL; h += 2)
                *reinterpret_cast<float2*>(qs + i * D + e0 + h) = make_float2(acc[i][h], acc[i][h + 1]);
            if (lane == 0) {
                ml[warp * QG + i] = m[i];
                ml[kCW * QG + warp * QG + i] = tl;
            }
        }
        __syncwarp();
        mbar_arrive_elect(mFull);
        if (!(ok = warp_wait(mFull, k & 1, abort_flag))) break;
        const float* qall = reinterpret_cast<const float*>(smem + L::kQs);
        for (int it = tid; it < QG * (D / 2); it += 32 * kCW) {
            const int i = it / (D / 2), d2 = 2 * (it % (D / 2));
            if (i >= pc.ng) continue;
            float mm = -INFINITY;
#pragma unroll
            for (int w = 0; w < kCW; ++w) mm = fmaxf(mm, ml[w * QG + i]);
            const float m_use = (mm == -INFINITY) ? 0.f : mm;
            float lt = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) {
                const float f = ex2f(ml[w * QG + i] - m_use);
                const float2 ow = *reinterpret_cast<const float2*>(qall + (w * QG + i) * D + d2);
                lt = fmaf(ml[kCW * QG + w * QG + i], f, lt);
                o0 = fmaf(ow.x, f, o0);
                o1 = fmaf(ow.y, f, o1);
            }
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const float lse2 = lt > 0.f ? mm + log2f(lt) : -INFINITY;  // -inf: no visible key here
            const int64_t row = static_cast<int64_t>(pc.bh) * p.Nq + pc.g0 + i;
            if (pc.nslots == 1) {
                store2<T>(static_cast<T*>(p.o) + row * D + d2, o0 * inv, o1 * inv);
                if (p.lse != nullptr && d2 == 0) p.lse[row] = lse2;
            } else {
                float* po = p.part_o + (row * p.P + pc.slot) * D;
                *reinterpret_cast<float2*>(po + d2) = make_float2(o0 * inv, o1 * inv);
                if (d2 == 0) p.part_lse[row * p.P + pc.slot] = lse2;
            }
        }
        __syncwarp();
        mbar_arrive_elect(mFree);
    }
    if (!ok) raise_abort(abort_flag);
}

// One warp per query row: merge the row's pieces by their log-sum-exps. Rows whose segment is
// a single piece were written by the main kernel and are skipped. Lane s holds piece s's
// log-sum-exp and weight (pieces in rounds of 32), so the loads of a round are independent;
// lane L owns output dims 2L, 2L+1 (+ 64 for D = 128).
template <typename T, int QG, int D>
__global__ void __launch_bounds__(128) attn_decode_merge_kernel(const DecodeParams p, int64_t rows) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the main kernel's writes are visible
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int bh = static_cast<int>(row / p.Nq), qi = static_cast<int>(row % p.Nq);
    int n;
    if (p.explicit_splits > 0) {
        n = p.explicit_splits;
    } else {
        const int64_t s0 = (static_cast<int64_t>(bh) * p.groups + qi / QG) * p.Tn;
        n = static_cast<int>(owner_of(s0 + p.Tn - 1, p.C, p.G) - owner_of(s0, p.C, p.G) + 1);
    }
    if (n == 1) return;
    constexpr int G = D / 64;
    const float* pl = p.part_lse + row * p.P;
    const float* po = p.part_o + row * p.P * D + 2 * lane;
    float mx = -INFINITY;
    for (int s0 = 0; s0 < n; s0 += 32) mx = fmaxf(mx, s0 + lane < n ? pl[s0 + lane] : -INFINITY);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float w_tot = 0.f, o[G][2];
#pragma unroll
    for (int g = 0; g < G; ++g) o[g][0] = o[g][1] = 0.f;
    for (int s0 = 0; s0 < n; s0 += 32) {
        const float ls = s0 + lane < n ? pl[s0 + lane] : -INFINITY;
        const float w = ls == -INFINITY ? 0.f : ex2f(ls - mx);  // a piece with no visible key weighs 0
        w_tot += w;
        const int m = min(32, n - s0);
#pragma unroll 8
        for (int u = 0; u < m; ++u) {
            const float wu = __shfl_sync(0xffffffffu, w, u);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float2 ov = *reinterpret_cast<const float2*>(po + (s0 + u) * D + 64 * g);
                o[g][0] = fmaf(wu, ov.x, o[g][0]);
                o[g][1] = fmaf(wu, ov.y, o[g][1]);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) w_tot += __shfl_xor_sync(0xffffffffu, w_tot, off);
    const float inv = 1.f / w_tot;  // every row sees at least one key, so w_tot >= 1
#pragma unroll
    for (int g = 0; g < G; ++g)
        store2<T>(static_cast<T*>(p.o) + row * D + 64 * g + 2 * lane, o[g][0] * inv, o[g][1] * inv);
    if (p.lse != nullptr && lane == 0) p.lse[row] = mx + log2f(w_tot);
}

// A kernel whose one wait can never complete: a warp waits on the first phase of an mbarrier
// nobody arrives on, with the caller's limit. When the limit runs out the warp takes the same
// path as any kernel of this library (abort flag, device error word) and returns.
__global__ void __launch_bounds__(32) attn_wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_word = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const bool ok = mbar_wait(smem_u32(&bar), 0, nullptr, timeout_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) raise_abort(&abort_word);
}

// ------------------------------------------ host side ------------------------------------------
int queries_per_group(int64_t Nq) { return Nq <= 1 ? 1 : Nq <= 2 ? 2 : Nq <= 4 ? 4 : 8; }

template <typename X>
struct Tag {
    using type = X;
};
template <int V>
using IC = std::integral_constant<int, V>;

// Calls f(Tag<T>, IC<QG>, IC<D>) for the element type, query group and head width of a call.
template <typename F>
int visit_cfg(int dtype, int64_t d, int qg, F&& f) {
    auto by_qg = [&](auto t, auto dd) -> int {
        switch (qg) {
            case 1: return f(t, IC<1>{}, dd);
            case 2: return f(t, IC<2>{}, dd);
            case 4: return f(t, IC<4>{}, dd);
            default: return f(t, IC<8>{}, dd);
        }
    };
    auto by_d = [&](auto t) -> int { return d == 128 ? by_qg(t, IC<128>{}) : by_qg(t, IC<64>{}); };
    switch (dtype) {
        case ATTN_F32: return by_d(Tag<float>{});
        case ATTN_BF16: return by_d(Tag<__nv_bfloat16>{});
        default: return by_d(Tag<__half>{});
    }
}

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

// [BH][Nk][D] tensor; boxes of `rows` rows x 128 bytes (64 16-bit values or 32 fp32 values, so
// a row takes D * esz / 128 boxes), 128-byte swizzle; rows past Nk of a head are out of bounds
// (zero-filled), never the next head's.
bool make_map(CUtensorMap* map, const void* ptr, int64_t BH, int64_t Nk, int64_t D, int dtype, int rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t esz = dtype == ATTN_F32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz, static_cast<cuuint64_t>(Nk) * D * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUtensorMapDataType dt = dtype == ATTN_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of the main kernel that fit on one SM (0 if the query fails; only success is cached).
template <typename T, int QG, int D>
int ctas_per_sm() {
    static int cached = 0;
    if (cached > 0) return cached;
    int v = 0;
    if (cudaFuncSetAttribute(attn_decode_kernel<T, QG, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<T, QG, D>::kAlloc) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, attn_decode_kernel<T, QG, D>, Cfg<T, D>::kThreads,
                                                      Smem<T, QG, D>::kAlloc) != cudaSuccess)
        return 0;
    cached = v;
    return v;
}

// The grid and slot layout of one call. The workspace query and the launch both build it, so
// they agree on P.
struct Plan {
    int qg, groups, rows, Tn, C, P, tps;
    int64_t G;
    bool merge;  // some segment has more than one piece
};

bool make_plan(int64_t BH, int64_t Nq, int64_t Nk, int rows, int splits, int num_sms, int per_sm, int qg, Plan* pl) {
    pl->qg = qg;
    pl->groups = static_cast<int>((Nq + pl->qg - 1) / pl->qg);
    pl->rows = rows;
    pl->Tn = static_cast<int>((Nk + rows - 1) / rows);
    const int64_t segs = BH * pl->groups;
    const int64_t slots = static_cast<int64_t>(std::max(1, num_sms)) * std::max(1, per_sm);
    if (splits > 0) {
        pl->tps = (pl->Tn + splits - 1) / splits;
        pl->P = splits;
        pl->G = 0;
        pl->C = static_cast<int>(std::min<int64_t>(slots, segs * splits));
        pl->merge = splits > 1;
    } else {
        pl->tps = 0;
        pl->G = segs * pl->Tn;
        pl->C = static_cast<int>(std::min<int64_t>(slots, pl->G));
        // Every CTA run holds at least floor(G / C) tiles, so a segment of Tn tiles meets at
        // most ceil((Tn - 1) / run) + 1 runs.
        const int64_t run = pl->G / pl->C;
        pl->P = static_cast<int>(std::min<int64_t>(pl->C, (pl->Tn - 1 + run - 1) / run + 1));
        pl->merge = pl->P > 1;
    }
    return pl->C >= 1;
}

size_t partial_bytes(int64_t BH, int64_t Nq, int64_t D, int64_t P) {
    const double need = static_cast<double>(BH) * static_cast<double>(Nq) * static_cast<double>(P) * (D + 1) * 4.0;
    if (need > 9.0e18) return 0;
    const size_t r = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * static_cast<size_t>(P);
    return (r * static_cast<size_t>(D) * sizeof(float) + 255) / 256 * 256 + (r * sizeof(float) + 255) / 256 * 256;
}

// Two or more new queries in bf16/fp16 may run on the tensor-core kernel (attn_decode_tc.cu):
// groups of up to 128 queries as one M128 tile, key tiles of 128 (d = 64) or 64 (d = 128), one CTA
// per SM. It costs more per piece (a Q tile, the exchange of the two step parities) and its
// floor per call is a couple of microseconds higher, while the CUDA-core kernel slows with every
// query of a group (3 queries run as a group of 4). Measured on GB300 (bf16, causal): at d = 128
// the tensor-core kernel is never slower; at d = 64 it wins from 8 queries on (B64 H12 Nk256: 35
// against 41 us), for 3 to 7 once the cache holds 1024 keys and the call 2^18 cached rows in all
// (B64 H12 Nk1024 Nq4: 55 against 67 us; B16 H12 Nk8192 Nq3: 73 against 102; B4 H8 Nk2048 Nq4:
// 19 against 16), and for 2 only on long caches (B1 H1 Nk100000: 35 against 52 us; B16 H12
// Nk8192: 72.5 against 69.3).
bool use_tc(int dtype, int64_t d, int64_t BH, int64_t Nq, int64_t Nk) {
    if (dtype == ATTN_F32 || Nq < 2 || (d != 64 && d != 128)) return false;
    if (d == 128 || Nq >= 8 || Nk >= 32768) return true;
    return Nq >= 3 && Nk >= 1024 && BH * Nk >= (int64_t{1} << 18);
}

// Builds the plan of a call: the kernel's tile rows and occupancy come from its configuration.
bool plan_for(int64_t BH, int64_t Nq, int64_t Nk, int64_t D, int splits, int dtype, int num_sms, Plan* pl) {
    if (use_tc(dtype, D, BH, Nq, Nk)) return make_plan(BH, Nq, Nk, D == 64 ? 128 : 64, splits, num_sms, 1, 128, pl);
    int rows = 0, per_sm = 0;
    visit_cfg(dtype, D, queries_per_group(Nq), [&](auto t, auto qg, auto dd) -> int {
        using T = typename decltype(t)::type;
        rows = Cfg<T, decltype(dd)::value>::kRows;
        per_sm = ctas_per_sm<T, decltype(qg)::value, decltype(dd)::value>();
        return 0;
    });
    if (per_sm <= 0) return false;
    return make_plan(BH, Nq, Nk, rows, splits, num_sms, per_sm, queries_per_group(Nq), pl);
}

// Programmatic stream serialisation: the merge grid may start while the main grid runs (it is
// released by the main kernel's launch_dependents) and waits in griddepcontrol.wait until that
// grid has completed and its memory is visible.
template <typename T, int QG, int D>
int launch_merge(const DecodeParams& prm, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(prm.BH) * prm.Nq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_merge_kernel<T, QG, D>, prm, rows) == cudaSuccess ? ATTN_OK
                                                                                                  : ATTN_ERR_LAUNCH;
}

}  // namespace

size_t decode_workspace_bytes(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int splits, int dtype, int num_sms) {
    if (BH <= 0 || Nq <= 0 || Nk <= 0 || splits < 0 || splits > ATTN_KV_MAX_SPLITS) return 0;
    if (BH > 0x7FFFFFFFll || Nq > ATTN_MAX_N || Nk > ATTN_MAX_N || (d != 64 && d != 128)) return 0;
    if (splits == 1) return 0;
    if (splits > 1) return partial_bytes(BH, Nq, d, splits);
    Plan pl;
    if (!plan_for(BH, Nq, Nk, d, 0, dtype, num_sms, &pl)) return 0;
    return pl.merge ? partial_bytes(BH, Nq, d, pl.P) : 0;
}

int launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream) {
    attn_wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int decode_device_error(bool clear, unsigned* err) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (clear && v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_DEVICE;
    }
    *err = v;
    return ATTN_OK;
}

int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                  size_t workspace_bytes, int64_t BH, int64_t Nq, int64_t Nk, int64_t d, bool causal, int dtype,
                  int splits, int num_sms, cudaStream_t stream) {
    if (Nk > ATTN_MAX_N || BH > 0x7FFFFFFFll || splits < 0 || splits > ATTN_KV_MAX_SPLITS) return ATTN_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    Plan pl;
    if (!plan_for(BH, Nq, Nk, d, splits, dtype, num_sms, &pl)) return ATTN_ERR_LAUNCH;
    if (BH * pl.groups > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    DecodeParams prm;
    prm.q = q;
    prm.o = o;
    prm.lse = lse;
    prm.Nq = static_cast<int>(Nq);
    prm.Nk = static_cast<int>(Nk);
    prm.BH = static_cast<int>(BH);
    prm.groups = pl.groups;
    prm.Tn = pl.Tn;
    prm.causal = causal ? 1 : 0;
    prm.explicit_splits = splits;
    prm.tps = pl.tps;
    prm.P = pl.P;
    prm.C = pl.C;
    prm.G = pl.G;
    prm.c = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    prm.part_o = nullptr;
    prm.part_lse = nullptr;
    if (pl.merge) {
        const size_t need = partial_bytes(BH, Nq, d, pl.P);
        if (need == 0) return ATTN_ERR_UNSUPPORTED;
        if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        const size_t r = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * static_cast<size_t>(pl.P);
        prm.part_o = static_cast<float*>(workspace);
        prm.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                (r * static_cast<size_t>(d) * sizeof(float) + 255) / 256 * 256);
    }
    CUtensorMap mk, mv;
    if (!make_map(&mk, k, BH, Nk, d, dtype, pl.rows) || !make_map(&mv, v, BH, Nk, d, dtype, pl.rows))
        return ATTN_ERR_DEVICE;
    if (use_tc(dtype, d, BH, Nq, Nk)) {
        CUtensorMap mq;
        if (!make_map(&mq, q, BH, Nq, d, dtype, 128)) return ATTN_ERR_DEVICE;
        const int st = launch_decode_tc_main(mq, mk, mv, prm, dtype == ATTN_BF16, static_cast<int>(d), stream);
        if (st != ATTN_OK || !pl.merge) return st;
        if (d == 64)
            return dtype == ATTN_BF16 ? launch_merge<__nv_bfloat16, 128, 64>(prm, stream)
                                      : launch_merge<__half, 128, 64>(prm, stream);
        return dtype == ATTN_BF16 ? launch_merge<__nv_bfloat16, 128, 128>(prm, stream)
                                  : launch_merge<__half, 128, 128>(prm, stream);
    }
    return visit_cfg(dtype, d, pl.qg, [&](auto t, auto qg, auto dd) -> int {
        using T = typename decltype(t)::type;
        constexpr int QG = decltype(qg)::value, D = decltype(dd)::value;
        // ctas_per_sm (called by the plan of a balanced call) has set the shared-memory limit;
        // an explicit plan sets it here.
        if (cudaFuncSetAttribute(attn_decode_kernel<T, QG, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Smem<T, QG, D>::kAlloc) != cudaSuccess)
            return ATTN_ERR_LAUNCH;
        attn_decode_kernel<T, QG, D><<<static_cast<unsigned>(prm.C), Cfg<T, D>::kThreads, Smem<T, QG, D>::kAlloc,
                                       stream>>>(mk, mv, prm);
        if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
        if (!pl.merge) return ATTN_OK;
        return launch_merge<T, QG, D>(prm, stream);
    });
}

}  // namespace attn
