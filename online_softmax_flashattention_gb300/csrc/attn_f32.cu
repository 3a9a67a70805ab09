// Online-softmax attention forward for float32 on CUDA cores (FFMA).
//
// Same operation and recurrence as the tensor-core kernel: per query row a running max m,
// a running denominator l and a running output, rescaled by exp(m_old - m_new) when a key
// tile raises the max (attention.cu, attentionOnline and its "online-update" step; "Flash
// attention in PyTorch, then in Triton", section "Flash attention"). Scores are kept in
// base-2 units, s * log2(e) / sqrt(d), so every exponential is an exp2 ("A kernel in
// Triton"). Causal key tiles past a block's last query are skipped and ragged N is guarded
// on every load and store (the page's kernel masks rows and keys past T).
//
// Layout per CTA: BM query rows (64; 32 when the grid would not fill the GPU; 16 for causal
// grids that split the keys, below) against key tiles of 64, head width D = 64 or 128, BM/4 x 16
// threads. Thread (ty, tx) holds a 4 x 4 score micro-tile — rows ty*4 + i, keys tx + 16 j — and a
// 4 x D/16 output micro-tile — rows ty*4 + i, dims 64 g + tx*4 + j. Rows of shared tiles are
// padded to D + 4 floats so that every float4 read of a key row, every P store and every V read
// is free of bank conflicts. The 16 threads that share a row sit in one half-warp, so row max
// and row sum are 4-step xor shuffles.
// With an `lse` pointer each row's log-sum-exp is stored too, in base 2 as the page's
// forward kernel keeps it for the backward pass (m + log2 l, "Backwards, and training with
// it").
//
// Small grids (fewer blocks than the GPU has SMs to fill, e.g. one head of 4096 queries) split
// the keys inside the CTA: G groups of BM*4 threads share the Q tile and each takes the key tiles
// t = g, g + G, ... with a running max, total and output of its own (the online softmax over a
// subset of the keys), synchronising on a named barrier of its own; at the end the groups'
// partial results merge as the online softmax merges tiles: M = max m_g, o = sum 2^(m_g - M)
// O_g / sum 2^(m_g - M) l_g.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

// Padded row stride (floats) of every shared tile.
template <int D>
__host__ __device__ constexpr int ld_of() { return D + 4; }

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte asynchronous copy global -> shared (cp.async, cached in L2 only); with `valid` false
// nothing is read and the 16 bytes are filled with zeros.
__device__ __forceinline__ void cp_async16(float* smem_dst, const float* gsrc, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's most recent copy groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One 64-key tile of K or V (rows kbase .. kbase + kBN - 1 of a head, rows >= N as zeros) into a
// padded shared tile, kBN * D / 4 16-byte copies spread over the group's threads.
template <int kBN, int D, int kThreads>
__device__ __forceinline__ void load_tile_async(float* dst, const float* src, int kbase, int N, int tid) {
    constexpr int kD4 = D / 4;
    constexpr int kLd = D + 4;
    static_assert(kBN * kD4 % kThreads == 0, "whole 16-byte copies per thread");
#pragma unroll
    for (int u = 0; u < kBN * kD4 / kThreads; ++u) {
        const int idx = tid + u * kThreads;
        const int r = idx / kD4, e4 = idx % kD4;
        const bool ok = kbase + r < N;
        cp_async16(dst + r * kLd + 4 * e4, ok ? src + static_cast<int64_t>(kbase + r) * D + 4 * e4 : src, ok);
    }
}

// Group-local barrier (G > 1) or the whole CTA (G = 1).
template <int G, int kThreads>
__device__ __forceinline__ void group_sync(int grp) {
    if constexpr (G == 1) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kThreads) : "memory");
    }
}

template <int BM, int D, int G, int kBN>
__global__ void __launch_bounds__(BM * 4 * G)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                        int N, int BH, int nblk, int causal, float c) {
    constexpr int kThreads = BM * 4;  // one group
    constexpr int kLd = ld_of<D>();
    constexpr int kD4 = D / 4;   // float4 per row
    constexpr int kG = D / 64;   // 64-dim groups of this thread's output columns
    constexpr int kJ = kBN / 16;  // keys of this thread's score micro-tile
    extern __shared__ float4 smem4[];
    const int grp = static_cast<int>(threadIdx.x) / kThreads;
    float* const Qs = reinterpret_cast<float*>(smem4);
    float* const Ks = Qs + BM * kLd + grp * (2 * kBN + BM) * kLd;
    float* const Vs = Ks + kBN * kLd;
    float* const Ps = Vs + kBN * kLd;

    const int tid = static_cast<int>(threadIdx.x) % kThreads;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(BH));
    const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(BH));
    const int blk = causal ? (nblk - 1 - slot) : slot;
    const int row0 = blk * BM;
    const int64_t head = static_cast<int64_t>(bh) * N * D;
    const float* qh = q + head;
    const float* kh = k + head;
    const float* vh = v + head;

    // Q tile, rows >= N read as zero (all groups load it together).
    for (int idx = static_cast<int>(threadIdx.x); idx < BM * kD4; idx += kThreads * G) {
        const int r = idx / kD4, e4 = idx % kD4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < N) val = *reinterpret_cast<const float4*>(qh + static_cast<int64_t>(row0 + r) * D + 4 * e4);
        *reinterpret_cast<float4*>(Qs + r * kLd + 4 * e4) = val;
    }

    float m[4], l[4], acc[4][4 * kG];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < 4 * kG; ++j) acc[i][j] = 0.f;
    }

    if constexpr (G > 1) __syncthreads();  // Q is in
    const int kend = causal ? min(N, row0 + BM) : N;
    const int ntiles = (kend + kBN - 1) / kBN;
    // K and V stream through one shared tile each, software-pipelined with asynchronous copies:
    // tile t + G's keys load while tile t's softmax and P V run, its values while tile t + G's
    // scores are formed. Copy groups are committed K, V, K, V, ... so that "all but the newest
    // group" is always the tile about to be read.
    if (grp < ntiles) {
        load_tile_async<kBN, D, kThreads>(Ks, kh, grp * kBN, N, tid);
        cp_async_commit();
        load_tile_async<kBN, D, kThreads>(Vs, vh, grp * kBN, N, tid);
        cp_async_commit();
    }
    for (int t = grp; t < ntiles; t += G) {
        const int kbase = t * kBN;
        const bool next = t + G < ntiles;
        cp_async_wait<1>();            // this thread's copies of K(t) have landed
        group_sync<G, kThreads>(grp);  // everyone's have

        // S micro-tile: rows ty*4+i, keys tx+16j.
        float s[4][kJ];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < kJ; ++j) s[i][j] = 0.f;
#pragma unroll 4
        for (int e = 0; e < D; e += 4) {
            float4 qa[4], kb[kJ];
#pragma unroll
            for (int i = 0; i < 4; ++i) qa[i] = *reinterpret_cast<const float4*>(Qs + (ty * 4 + i) * kLd + e);
#pragma unroll
            for (int j = 0; j < kJ; ++j) kb[j] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * j) * kLd + e);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    s[i][j] = fmaf(qa[i].x, kb[j].x, s[i][j]);
                    s[i][j] = fmaf(qa[i].y, kb[j].y, s[i][j]);
                    s[i][j] = fmaf(qa[i].z, kb[j].z, s[i][j]);
                    s[i][j] = fmaf(qa[i].w, kb[j].w, s[i][j]);
                }
        }

        group_sync<G, kThreads>(grp);  // K(t) is read: the next tile's keys may overwrite it
        if (next) load_tile_async<kBN, D, kThreads>(Ks, kh, kbase + G * kBN, N, tid);
        cp_async_commit();

        // Mask keys past N and, when causal, keys after the query.
        if (kbase + kBN > N || (causal && kbase + kBN - 1 > row0)) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = row0 + ty * 4 + i;
                const int lim = causal ? min(row + 1, N) : N;
#pragma unroll
                for (int j = 0; j < kJ; ++j)
                    if (kbase + tx + 16 * j >= lim) s[i][j] = -INFINITY;
            }
        }

        // Online update per row.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = s[i][0];
#pragma unroll
            for (int j = 1; j < kJ; ++j) mx = fmaxf(mx, s[i][j]);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx * c);
            const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2f(m[i] - m_ref);
            float ps = 0.f;
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const float pv = ex2f(fmaf(s[i][j], c, -m_ref));
                ps += pv;
                Ps[(ty * 4 + i) * kLd + tx + 16 * j] = pv;
            }
            l[i] = l[i] * alpha + ps;  // this thread's share of the row total
            m[i] = m_ref;
#pragma unroll
            for (int j = 0; j < 4 * kG; ++j) acc[i][j] *= alpha;
        }
        cp_async_wait<1>();            // V(t) has landed (K(t + G) may still be in flight)
        group_sync<G, kThreads>(grp);  // V(t) and P are visible to the group

        // O micro-tile += P V: rows ty*4+i, dims 64g + tx*4+j.
#pragma unroll 4
        for (int kk = 0; kk < kBN; kk += 4) {
            float4 pa[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pa[i] = *reinterpret_cast<const float4*>(Ps + (ty * 4 + i) * kLd + kk);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                float4 vb[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    vb[u] = *reinterpret_cast<const float4*>(Vs + (kk + u) * kLd + 64 * g + 4 * tx);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float pw[4] = {pa[i].x, pa[i].y, pa[i].z, pa[i].w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc[i][4 * g + 0] = fmaf(pw[u], vb[u].x, acc[i][4 * g + 0]);
                        acc[i][4 * g + 1] = fmaf(pw[u], vb[u].y, acc[i][4 * g + 1]);
                        acc[i][4 * g + 2] = fmaf(pw[u], vb[u].z, acc[i][4 * g + 2]);
                        acc[i][4 * g + 3] = fmaf(pw[u], vb[u].w, acc[i][4 * g + 3]);
                    }
                }
            }
        }
        group_sync<G, kThreads>(grp);  // V(t) and P are read
        if (next) load_tile_async<kBN, D, kThreads>(Vs, vh, kbase + G * kBN, N, tid);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // Row totals across the 16 threads of the row.
    float tot[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        tot[i] = l[i];
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) tot[i] += __shfl_xor_sync(0xffffffffu, tot[i], off);
    }
    if constexpr (G > 1) {
        // Merge the groups' partial results into group 0 through shared memory (the K/V/P tiles
        // are free once every group is past its last tile). A group with no key tile, or whose
        // rows saw no key yet, has m = -inf and l = 0 and contributes nothing.
        __syncthreads();
        float* const X = reinterpret_cast<float*>(smem4) + BM * kLd;  // [G][kThreads][4 * (4 kG + 2)]
        constexpr int kRec = 4 * (4 * kG + 2);
        float* const mine = X + (grp * kThreads + tid) * kRec;
        if (grp > 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mine[i * (4 * kG + 2)] = m[i];
                mine[i * (4 * kG + 2) + 1] = tot[i];
#pragma unroll
                for (int j = 0; j < 4 * kG; ++j) mine[i * (4 * kG + 2) + 2 + j] = acc[i][j];
            }
        }
        __syncthreads();
        if (grp > 0) return;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float M = m[i];
#pragma unroll
            for (int h = 1; h < G; ++h) M = fmaxf(M, X[(h * kThreads + tid) * kRec + i * (4 * kG + 2)]);
            const float a0 = (m[i] == -INFINITY) ? 0.f : ex2f(m[i] - M);
            tot[i] *= a0;
#pragma unroll
            for (int j = 0; j < 4 * kG; ++j) acc[i][j] *= a0;
#pragma unroll
            for (int h = 1; h < G; ++h) {
                const float* r = X + (h * kThreads + tid) * kRec + i * (4 * kG + 2);
                const float a = (r[0] == -INFINITY) ? 0.f : ex2f(r[0] - M);
                tot[i] = fmaf(r[1], a, tot[i]);
#pragma unroll
                for (int j = 0; j < 4 * kG; ++j) acc[i][j] = fmaf(r[2 + j], a, acc[i][j]);
            }
            m[i] = M;
        }
    }
    // O / l.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = row0 + ty * 4 + i;
        if (row < N) {
            const float inv = 1.f / tot[i];
#pragma unroll
            for (int g = 0; g < kG; ++g)
                *reinterpret_cast<float4*>(o + head + static_cast<int64_t>(row) * D + 64 * g + 4 * tx) =
                    make_float4(acc[i][4 * g] * inv, acc[i][4 * g + 1] * inv, acc[i][4 * g + 2] * inv,
                                acc[i][4 * g + 3] * inv);
            if (lse != nullptr && tx == 0) lse[static_cast<int64_t>(bh) * N + row] = m[i] + log2f(tot[i]);
        }
    }
}

template <int BM, int D, int G, int kBN = 64>
int launch_bm(const float* q, const float* k, const float* v, float* o, float* lse, int64_t BH,
              int64_t N, bool causal, cudaStream_t stream) {
    // Q, then per group K, V and P tiles; the groups' merge records reuse the K/V/P space.
    constexpr int kLd = ld_of<D>();
    constexpr int kTiles = (BM + G * (2 * kBN + BM)) * kLd * static_cast<int>(sizeof(float));
    constexpr int kMerge = (BM * kLd + G * BM * 4 * 4 * (4 * (D / 64) + 2)) * static_cast<int>(sizeof(float));
    constexpr int smem = kTiles > kMerge ? kTiles : kMerge;
    static_assert(smem <= 227 * 1024, "shared memory of one CTA");
    static uint64_t ready = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    if (!once_per_device(&ready, dev, [] {
            return cudaFuncSetAttribute(attn_fwd_f32_kernel<BM, D, G, kBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem) == cudaSuccess;
        }))
        return ATTN_ERR_LAUNCH;
    const int64_t nblk = (N + BM - 1) / BM;
    const int64_t blocks = nblk * BH;
    if (blocks > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    const float c = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    attn_fwd_f32_kernel<BM, D, G, kBN><<<static_cast<unsigned>(blocks), BM * 4 * G, smem, stream>>>(
        q, k, v, o, lse, static_cast<int>(N), static_cast<int>(BH), static_cast<int>(nblk), causal ? 1 : 0, c);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int64_t BH,
                   int64_t N, int64_t d, bool causal, int num_sms, cudaStream_t stream) {
    if (N > 0x7FFFFFFFll - 64 || BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    constexpr int kBN = 64;
    // Grids that fill the GPU run 64-row blocks; smaller ones 32-row blocks, and when even those
    // leave most SMs with a single block, the keys are split over G groups inside each block.
    const int64_t blocks64 = ((N + 63) / 64) * BH;
    const int64_t blocks32 = ((N + 31) / 32) * BH;
    const bool small = blocks64 < 2 * static_cast<int64_t>(num_sms);
    const bool split = blocks32 < 2 * static_cast<int64_t>(num_sms) && N > 2 * kBN;
    // Causal small grids take 16-row blocks: the heaviest block (the last rows, which see every
    // key) bounds the call, and it runs on one SM, so halving its rows halves the critical path.
    if (d == 64)
        return split ? (causal ? launch_bm<16, 64, 4>(q, k, v, o, lse, BH, N, causal, stream)
                               : launch_bm<32, 64, 4>(q, k, v, o, lse, BH, N, causal, stream))
               : small ? launch_bm<32, 64, 1>(q, k, v, o, lse, BH, N, causal, stream)
                       : launch_bm<64, 64, 1>(q, k, v, o, lse, BH, N, causal, stream);
    if (d == 128)
        return split ? launch_bm<32, 128, 2>(q, k, v, o, lse, BH, N, causal, stream)
               : small ? launch_bm<32, 128, 1>(q, k, v, o, lse, BH, N, causal, stream)
                       : launch_bm<64, 128, 1>(q, k, v, o, lse, BH, N, causal, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
