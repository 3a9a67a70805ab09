// Key-value cache attention (decode): Nq new queries, the last Nq positions of a sequence,
// against Nk >= Nq cached keys and values, with the key range split across CTAs and the
// partial results merged by their log-sum-exps.
//
// The "Flash attention in PyTorch, then in Triton" page names this case and leaves it out of
// its kernel (section "Backwards, and training with it": generation with a cache, where a few
// new tokens attend to every cached key). Query i sits at position Nk - Nq + i; when causal it
// sees keys 0 .. Nk - Nq + i. Each split runs the page's online softmax ("Flash attention": a running
// maximum, denominator and output per query, rescaled when a tile raises the maximum) over
// its share of the keys and leaves (O_s / l_s, lse2_s = m_s + log2 l_s); the combine step
// merges the splits the way the online softmax merges tiles:
//     lse2 = log2 sum_s 2^lse2_s,   O = sum_s 2^(lse2_s - lse2) O_s.
// A query sees few keys per byte it reads (one product of d terms per cached row of 2d
// values), so the work is bound by reading the cache from HBM; the kernel streams each K and
// V row once per query group with 16-byte loads and keeps the arithmetic on CUDA cores.
//
// Layout per CTA (bh, split, query group of QG queries): 4 warps, each taking 32 keys at a
// time, one key per lane. Scores: the lane forms q_i . k_j for its key and the group's QG
// queries (queries pre-scaled by log2(e)/sqrt(d) in shared memory). Online update per query
// over the warp's 32 keys (shuffle max), then the weighted values: lane L accumulates O_i for
// dims 2L, 2L+1, reading each value row coalesced and taking p_ij from lane j by shuffle. The
// four warps' states merge in shared memory at the end.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kD = 64;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight consecutive elements as fp32.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

// Two consecutive elements as fp32 (for the value rows, lane L reads dims 2L, 2L+1).
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
__device__ __forceinline__ void store2<float>(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
template <>
__device__ __forceinline__ void store2<__half>(__half* p, float a, float b) {
    *reinterpret_cast<__half2*>(p) = __floats2half2_rn(a, b);
}

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;          // written directly when splits == 1
    float* lse;       // null, or [BH, Nq] (direct mode)
    float* part_o;    // [BH][Nq][splits][64] when splits > 1
    float* part_lse;  // [BH][Nq][splits]
    int Nq, Nk, BH, splits, chunk, causal;
    float c;  // log2(e) / sqrt(d)
};

template <typename T, int QG>
__global__ void __launch_bounds__(kThreads)
    attn_decode_split_kernel(const DecodeParams p) {
    __shared__ float qs[QG][kD];
    __shared__ float wm[kWarps][QG], wl[kWarps][QG];
    __shared__ float wo[kWarps][QG][kD];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int split = blockIdx.y;
    const int g0 = blockIdx.z * QG;  // first query of the group
    const int ng = min(QG, p.Nq - g0);
    const T* const qh = static_cast<const T*>(p.q) + static_cast<int64_t>(bh) * p.Nq * kD;
    const T* const kh = static_cast<const T*>(p.k) + static_cast<int64_t>(bh) * p.Nk * kD;
    const T* const vh = static_cast<const T*>(p.v) + static_cast<int64_t>(bh) * p.Nk * kD;

    // The group's queries, scaled so that scores come out in base-2 units.
    for (int idx = threadIdx.x; idx < QG * kD; idx += kThreads) {
        const int i = idx / kD, e = idx % kD;
        float val = 0.f;
        if (i < ng) {
            float f[8];
            load8<T>(qh + static_cast<int64_t>(g0 + i) * kD + (e & ~7), f);
            val = f[e & 7] * p.c;
        }
        qs[i][e] = val;
    }
    __syncthreads();

    // Keys of this split, and the last key any query of the group may see.
    const int ks = split * p.chunk;
    int ke = min(p.Nk, ks + p.chunk);
    if (p.causal) ke = min(ke, p.Nk - p.Nq + g0 + ng);
    float m[QG], l[QG], acc[QG][2];
#pragma unroll
    for (int i = 0; i < QG; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
        acc[i][0] = acc[i][1] = 0.f;
    }
    for (int base = ks + 32 * warp; base < ke; base += 32 * kWarps) {
        const int j = base + lane;
        // scores of key j against the group's queries
        float s[QG];
#pragma unroll
        for (int i = 0; i < QG; ++i) s[i] = 0.f;
        if (j < ke) {
            const T* krow = kh + static_cast<int64_t>(j) * kD;
#pragma unroll
            for (int c8 = 0; c8 < kD; c8 += 8) {
                float f[8];
                load8<T>(krow + c8, f);
#pragma unroll
                for (int i = 0; i < QG; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(&qs[i][c8]);
                    const float4 b = *reinterpret_cast<const float4*>(&qs[i][c8 + 4]);
                    s[i] = fmaf(a.x, f[0], s[i]);
                    s[i] = fmaf(a.y, f[1], s[i]);
                    s[i] = fmaf(a.z, f[2], s[i]);
                    s[i] = fmaf(a.w, f[3], s[i]);
                    s[i] = fmaf(b.x, f[4], s[i]);
                    s[i] = fmaf(b.y, f[5], s[i]);
                    s[i] = fmaf(b.z, f[6], s[i]);
                    s[i] = fmaf(b.w, f[7], s[i]);
                }
            }
        }
        float pr[QG];
#pragma unroll
        for (int i = 0; i < QG; ++i) {
            const bool vis = j < ke && i < ng && (!p.causal || j <= p.Nk - p.Nq + g0 + i);
            const float sc = vis ? s[i] : -INFINITY;
            float mx = sc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no inf - inf on empty rows
            const float alpha = ex2f(m[i] - m_use);
            pr[i] = ex2f(sc - m_use);
            l[i] = l[i] * alpha + pr[i];  // this lane's share of the row total
            acc[i][0] *= alpha;
            acc[i][1] *= alpha;
            m[i] = m_new;
        }
        // weighted values: lane L owns dims 2L, 2L+1
        const int nk = min(32, ke - base);
#pragma unroll 8
        for (int kk = 0; kk < nk; ++kk) {
            const float2 vv = load2<T>(vh + static_cast<int64_t>(base + kk) * kD + 2 * lane);
#pragma unroll
            for (int i = 0; i < QG; ++i) {
                const float w = __shfl_sync(0xffffffffu, pr[i], kk);
                acc[i][0] = fmaf(w, vv.x, acc[i][0]);
                acc[i][1] = fmaf(w, vv.y, acc[i][1]);
            }
        }
    }
    // The warp's totals, then the four warps' states merged in shared memory.
#pragma unroll
    for (int i = 0; i < QG; ++i) {
        float t = l[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (lane == 0) {
            wm[warp][i] = m[i];
            wl[warp][i] = t;
        }
        *reinterpret_cast<float2*>(&wo[warp][i][2 * lane]) = make_float2(acc[i][0], acc[i][1]);
    }
    __syncthreads();
    // Thread t of the first QG*32 threads finishes query t/32, dims 2(t%32), 2(t%32)+1.
    for (int item = threadIdx.x; item < QG * 32; item += kThreads) {
        const int i = item >> 5, d2 = 2 * (item & 31);
        if (i >= ng) continue;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, wm[w][i]);
        const float m_use = (mm == -INFINITY) ? 0.f : mm;
        float lt = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = ex2f(wm[w][i] - m_use);
            lt = fmaf(wl[w][i], f, lt);
            o0 = fmaf(wo[w][i][d2], f, o0);
            o1 = fmaf(wo[w][i][d2 + 1], f, o1);
        }
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float lse2 = lt > 0.f ? mm + log2f(lt) : -INFINITY;  // -inf: no key of this split visible
        const int64_t row = static_cast<int64_t>(bh) * p.Nq + g0 + i;
        if (p.splits == 1) {
            store2<T>(static_cast<T*>(p.o) + row * kD + d2, o0 * inv, o1 * inv);
            if (p.lse != nullptr && d2 == 0) p.lse[row] = lse2;
        } else {
            float* po = p.part_o + (row * p.splits + split) * kD;
            po[d2] = o0 * inv;
            po[d2 + 1] = o1 * inv;
            if (d2 == 0) p.part_lse[row * p.splits + split] = lse2;
        }
    }
}

// One warp per query row: merge the splits by their log-sum-exps.
template <typename T>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const DecodeParams p, int64_t rows) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* pl = p.part_lse + row * p.splits;
    float mx = -INFINITY;
    for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, pl[s]);
    float w_tot = 0.f, o0 = 0.f, o1 = 0.f;
    for (int s = 0; s < p.splits; ++s) {
        if (pl[s] == -INFINITY) continue;  // a split with no visible key
        const float w = ex2f(pl[s] - mx);
        const float2 ov = *reinterpret_cast<const float2*>(p.part_o + (row * p.splits + s) * kD + 2 * lane);
        w_tot += w;
        o0 = fmaf(w, ov.x, o0);
        o1 = fmaf(w, ov.y, o1);
    }
    const float inv = 1.f / w_tot;  // every row sees at least one key, so w_tot >= 1
    store2<T>(static_cast<T*>(p.o) + row * kD + 2 * lane, o0 * inv, o1 * inv);
    if (p.lse != nullptr && lane == 0) p.lse[row] = mx + log2f(w_tot);
}

template <typename T>
int launch_t(DecodeParams prm, int64_t groups, int qg, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(prm.BH), static_cast<unsigned>(prm.splits), static_cast<unsigned>(groups));
    switch (qg) {
        case 1: attn_decode_split_kernel<T, 1><<<grid, kThreads, 0, stream>>>(prm); break;
        case 2: attn_decode_split_kernel<T, 2><<<grid, kThreads, 0, stream>>>(prm); break;
        case 4: attn_decode_split_kernel<T, 4><<<grid, kThreads, 0, stream>>>(prm); break;
        default: attn_decode_split_kernel<T, 8><<<grid, kThreads, 0, stream>>>(prm); break;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    if (prm.splits > 1) {
        const int64_t rows = static_cast<int64_t>(prm.BH) * prm.Nq;
        attn_decode_combine_kernel<T><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(prm, rows);
        if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    }
    return ATTN_OK;
}

}  // namespace

namespace {

int queries_per_group(int64_t Nq) { return Nq <= 1 ? 1 : Nq <= 2 ? 2 : Nq <= 4 ? 4 : 8; }

}  // namespace

size_t decode_workspace_bytes(int64_t BH, int64_t Nq, int64_t splits) {
    if (BH <= 0 || Nq <= 0 || splits <= 1 || splits > ATTN_KV_MAX_SPLITS) return 0;
    if (BH > 0x7FFFFFFFll || Nq > ATTN_MAX_N) return 0;
    // rows * splits * 65 floats stays below 2^31 * 2^30 * 2^10 * 2^7 < 2^64 only for sizes the
    // launcher accepts; check in double first.
    const double need = static_cast<double>(BH) * static_cast<double>(Nq) * static_cast<double>(splits) * (kD + 1) * 4.0;
    if (need > 9.0e18) return 0;
    const size_t r = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * static_cast<size_t>(splits);
    const size_t o_bytes = (r * kD * sizeof(float) + 255) / 256 * 256;
    const size_t l_bytes = (r * sizeof(float) + 255) / 256 * 256;
    return o_bytes + l_bytes;
}

int decode_auto_splits(int64_t BH, int64_t Nq, int64_t Nk, int num_sms) {
    if (BH <= 0 || Nq <= 0 || Nk <= 0) return 1;
    const int64_t groups = (Nq + queries_per_group(Nq) - 1) / queries_per_group(Nq);
    const int64_t ctas = BH * groups;
    const int64_t target = 8 * static_cast<int64_t>(num_sms);  // about eight CTAs of four warps per SM
    int64_t want = (target + ctas - 1) / ctas;
    want = std::min<int64_t>(want, std::max<int64_t>(1, Nk / 256));  // at least 256 keys per split
    want = std::min<int64_t>(want, ATTN_KV_MAX_SPLITS);
    return static_cast<int>(std::max<int64_t>(want, 1));
}

int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, int64_t BH,
                  int64_t Nq, int64_t Nk, bool causal, int dtype, int splits, cudaStream_t stream) {
    if (Nk > ATTN_MAX_N || BH > 0x7FFFFFFFll || splits < 1 || splits > ATTN_KV_MAX_SPLITS) return ATTN_ERR_UNSUPPORTED;
    const int qg = queries_per_group(Nq);
    const int64_t groups = (Nq + qg - 1) / qg;
    if (groups > 65535) return ATTN_ERR_UNSUPPORTED;
    DecodeParams prm;
    prm.q = q;
    prm.k = k;
    prm.v = v;
    prm.o = o;
    prm.lse = lse;
    prm.Nq = static_cast<int>(Nq);
    prm.Nk = static_cast<int>(Nk);
    prm.BH = static_cast<int>(BH);
    prm.splits = splits;
    prm.chunk = static_cast<int>(((Nk + splits - 1) / splits + 31) / 32 * 32);
    prm.causal = causal ? 1 : 0;
    prm.c = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
    if (splits > 1) {
        const size_t r = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * static_cast<size_t>(splits);
        prm.part_o = static_cast<float*>(workspace);
        prm.part_lse =
            reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + (r * kD * sizeof(float) + 255) / 256 * 256);
    } else {
        prm.part_o = nullptr;
        prm.part_lse = nullptr;
    }
    switch (dtype) {
        case ATTN_F32: return launch_t<float>(prm, groups, qg, stream);
        case ATTN_BF16: return launch_t<__nv_bfloat16>(prm, groups, qg, stream);
        default: return launch_t<__half>(prm, groups, qg, stream);
    }
}

}  // namespace attn
