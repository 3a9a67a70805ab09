// Backward pass of exact attention for float32 tensors on CUDA cores (FFMA). The bf16/fp16
// backward runs on tensor cores (attn_bwd_tc.cu) with the same two-kernel structure.
//
// Given the output gradient dO, the forward's output O and each row's base-2 log-sum-exp
// (lse2 = m + log2 l, kept by attn_fwd_lse), the gradients follow the "Flash attention in
// PyTorch, then in Triton" page, section "Backwards, and training with it":
//   P = 2^(S log2(e) - lse2) with S = Q K^T / sqrt(d)  (the probabilities made again from the
//                                                       scores, a block at a time)
//   dV = P^T dO,  dP = dO V^T,  delta_i = sum_e dO[i,e] O[i,e],  dS = P (dP - delta),
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d).
// As on the page the work is split into two kernels so that every program writes only its own
// rows and nothing is added up across programs: bwd_kv has a program per block of 64 keys
// that keeps dK and dV while the blocks of queries that see those keys go past; bwd_q has a
// program per block of 64 queries that keeps dQ while the blocks of keys it sees go past.
// Both recompute S and dP (the page's trade: no atomics, that work done twice). delta is
// recomputed per query block from dO and O (64 products per row) rather than kept in a
// buffer, so the call allocates nothing.
//
// Layout per program: 256 threads as 16 x 16 (ty, tx). A score micro-tile of 4 x 4 is rows
// (queries) ty*4+i, keys tx+16j; a gradient micro-tile is rows ty*4+i (keys in bwd_kv, queries
// in bwd_q), dims 64g + tx*4+j for the D/64 groups g (head width D = 64 or 128). Shared tiles
// are 64 rows padded to D + 4 floats (the P/dS tile to 68), so float4 row reads and the scalar
// P/dS stores are free of bank conflicts (the forward fp32 kernel's layout).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kB = 64;   // rows per block (queries and keys)
constexpr int kLdP = 68;  // padded row stride (floats) of the 64 x 64 P / dS tile
constexpr int kThreads = 256;

// Padded row stride (floats) of a 64 x D tile.
template <int D>
__host__ __device__ constexpr int ld_of() { return D + 4; }

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static __device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
    static __device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};
// Rows row0 .. row0+63 of a [N, D] head into a padded shared tile as fp32; rows >= N are 0.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int row0, int N) {
    constexpr int kLd = ld_of<D>();
    for (int idx = threadIdx.x; idx < kB * (D / 4); idx += kThreads) {
        const int r = idx / (D / 4), e4 = idx % (D / 4);
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < N) val = Elem<T>::load4(src + static_cast<int64_t>(row0 + r) * D + 4 * e4);
        *reinterpret_cast<float4*>(dst + r * kLd + 4 * e4) = val;
    }
}

// delta[r] = sum_e dO[r,e] O[r,e] for the 64 rows of a block (4 threads per row), and the
// rows' log-sum-exps; padded rows get delta 0, lse 0 (their probabilities are masked).
template <typename T, int D>
__device__ __forceinline__ void load_row_terms(float* delta, float* lse_s, const float* dOs, const T* o,
                                               const float* lse, int row0, int N) {
    constexpr int kLd = ld_of<D>(), kPart = D / 4;
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    float acc = 0.f;
    if (row0 + r < N) {
        const T* orow = o + static_cast<int64_t>(row0 + r) * D + kPart * part;
#pragma unroll
        for (int e = 0; e < kPart; e += 4) {
            const float4 ov = Elem<T>::load4(orow + e);
            const float4 dv = *reinterpret_cast<const float4*>(dOs + r * kLd + kPart * part + e);
            acc = fmaf(ov.x, dv.x, acc);
            acc = fmaf(ov.y, dv.y, acc);
            acc = fmaf(ov.z, dv.z, acc);
            acc = fmaf(ov.w, dv.w, acc);
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (part == 0) {
        delta[r] = acc;
        lse_s[r] = (row0 + r < N) ? lse[row0 + r] : 0.f;
    }
}

// 4 x 4 micro-tile of A B^T for shared 64 x D tiles A (rows ty*4+i) and B (rows tx+16j), K = D.
template <int D>
__device__ __forceinline__ void micro_abt(float (&c)[4][4], const float* A, const float* Bm, int ty, int tx) {
    constexpr int kLd = ld_of<D>();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[i][j] = 0.f;
#pragma unroll 4
    for (int e = 0; e < D; e += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (ty * 4 + i) * kLd + e);
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(Bm + (tx + 16 * j) * kLd + e);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c[i][j] = fmaf(a[i].x, b[j].x, c[i][j]);
                c[i][j] = fmaf(a[i].y, b[j].y, c[i][j]);
                c[i][j] = fmaf(a[i].z, b[j].z, c[i][j]);
                c[i][j] = fmaf(a[i].w, b[j].w, c[i][j]);
            }
    }
}

// acc[i][4g+j] += sum_r X[r][ty*4+i] * Y[r][64g + tx*4+j] over the 64 rows r of the P/dS tile X
// and a 64 x D tile Y (X^T Y for a gradient micro-tile whose rows index X's columns).
template <int D>
__device__ __forceinline__ void micro_atb(float (&acc)[4][D / 16], const float* X, const float* Y, int ty, int tx) {
    constexpr int kLd = ld_of<D>();
#pragma unroll 4
    for (int r = 0; r < kB; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(X + r * kLdP + 4 * ty);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int g = 0; g < D / 64; ++g) {
            const float4 y = *reinterpret_cast<const float4*>(Y + r * kLd + 64 * g + 4 * tx);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[i][4 * g + 0] = fmaf(xs[i], y.x, acc[i][4 * g + 0]);
                acc[i][4 * g + 1] = fmaf(xs[i], y.y, acc[i][4 * g + 1]);
                acc[i][4 * g + 2] = fmaf(xs[i], y.z, acc[i][4 * g + 2]);
                acc[i][4 * g + 3] = fmaf(xs[i], y.w, acc[i][4 * g + 3]);
            }
        }
    }
}

// acc[i][4g+j] += sum_c X[ty*4+i][c] * Y[c][64g + tx*4+j] over the 64 columns c of the P/dS
// tile X and the rows of a 64 x D tile Y (X Y).
template <int D>
__device__ __forceinline__ void micro_ab(float (&acc)[4][D / 16], const float* X, const float* Y, int ty, int tx) {
    constexpr int kLd = ld_of<D>();
#pragma unroll 4
    for (int c = 0; c < kB; c += 4) {
        float4 x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = *reinterpret_cast<const float4*>(X + (ty * 4 + i) * kLdP + c);
#pragma unroll
        for (int g = 0; g < D / 64; ++g) {
            float4 y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) y[u] = *reinterpret_cast<const float4*>(Y + (c + u) * kLd + 64 * g + 4 * tx);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float xs[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[i][4 * g + 0] = fmaf(xs[u], y[u].x, acc[i][4 * g + 0]);
                    acc[i][4 * g + 1] = fmaf(xs[u], y[u].y, acc[i][4 * g + 1]);
                    acc[i][4 * g + 2] = fmaf(xs[u], y[u].z, acc[i][4 * g + 2]);
                    acc[i][4 * g + 3] = fmaf(xs[u], y[u].w, acc[i][4 * g + 3]);
                }
            }
        }
    }
}

// P for the score micro-tile (queries q0 + ty*4+i, keys k0 + tx+16j); masked entries 0.
__device__ __forceinline__ void probs(float (&p)[4][4], const float (&s)[4][4], const float* lse_s, int q0,
                                      int k0, int N, int causal, float c, int ty, int tx) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int qi = q0 + ty * 4 + i;
        const float l2 = lse_s[ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kj = k0 + tx + 16 * j;
            const bool vis = qi < N && kj < N && (!causal || kj <= qi);
            p[i][j] = vis ? ex2f(fmaf(s[i][j], c, -l2)) : 0.f;
        }
    }
}

// ------------------------------- dK, dV: one program per key block -------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    attn_bwd_kv_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const T* __restrict__ o, const T* __restrict__ dout, const float* __restrict__ lse,
                       T* __restrict__ dk, T* __restrict__ dv, int N, int BH, int nblk, int causal,
                       float c, float scale) {
    constexpr int kLd = ld_of<D>(), G = D / 16;
    extern __shared__ float4 smem4[];
    float* const Ks = reinterpret_cast<float*>(smem4);
    float* const Vs = Ks + kB * kLd;
    float* const Qs = Vs + kB * kLd;
    float* const dOs = Qs + kB * kLd;
    float* const Ps = dOs + kB * kLd;
    float* const delta = Ps + kB * kLdP;
    float* const lse_s = delta + kB;

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(BH));
    const int kblk = static_cast<int>(blockIdx.x / static_cast<unsigned>(BH));
    const int k0 = kblk * kB;
    const int64_t head = static_cast<int64_t>(bh) * N * D;
    load_tile<T, D>(Ks, k + head, k0, N);
    load_tile<T, D>(Vs, v + head, k0, N);

    float dK[4][G], dV[4][G];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < G; ++j) dK[i][j] = dV[i][j] = 0.f;

    // With causal attention these keys are seen by the queries from the block's first key on.
    for (int qb = causal ? kblk : 0; qb < nblk; ++qb) {
        const int q0 = qb * kB;
        __syncthreads();  // the previous block is done with Qs, dOs, Ps, delta
        load_tile<T, D>(Qs, q + head, q0, N);
        load_tile<T, D>(dOs, dout + head, q0, N);
        __syncthreads();
        load_row_terms<T, D>(delta, lse_s, dOs, o + head, lse + static_cast<int64_t>(bh) * N, q0, N);
        __syncthreads();

        float s[4][4], p[4][4], dp[4][4];
        micro_abt<D>(s, Qs, Ks, ty, tx);  // S = Q K^T: queries ty*4+i, keys tx+16j
        probs(p, s, lse_s, q0, k0, N, causal, c, ty, tx);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * kLdP + tx + 16 * j] = p[i][j];
        micro_abt<D>(dp, dOs, Vs, ty, tx);  // dP = dO V^T
        __syncthreads();
        micro_atb<D>(dV, Ps, dOs, ty, tx);  // dV[key][dim] += sum_q P[q][key] dO[q][dim]
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float dl = delta[ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * kLdP + tx + 16 * j] = p[i][j] * (dp[i][j] - dl);
        }
        __syncthreads();
        micro_atb<D>(dK, Ps, Qs, ty, tx);  // dK[key][dim] += sum_q dS[q][key] Q[q][dim]
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int key = k0 + ty * 4 + i;
        if (key < N) {
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const int64_t off = head + static_cast<int64_t>(key) * D + 64 * g + 4 * tx;
                Elem<T>::store4(dk + off, make_float4(dK[i][4 * g] * scale, dK[i][4 * g + 1] * scale,
                                                      dK[i][4 * g + 2] * scale, dK[i][4 * g + 3] * scale));
                Elem<T>::store4(dv + off, make_float4(dV[i][4 * g], dV[i][4 * g + 1], dV[i][4 * g + 2], dV[i][4 * g + 3]));
            }
        }
    }
}

// --------------------------------- dQ: one program per query block ---------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    attn_bwd_q_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const T* __restrict__ o, const T* __restrict__ dout, const float* __restrict__ lse,
                      T* __restrict__ dq, int N, int BH, int nblk, int causal, float c, float scale) {
    constexpr int kLd = ld_of<D>(), G = D / 16;
    extern __shared__ float4 smem4[];
    float* const Qs = reinterpret_cast<float*>(smem4);
    float* const dOs = Qs + kB * kLd;
    float* const Ks = dOs + kB * kLd;
    float* const Vs = Ks + kB * kLd;
    float* const Ps = Vs + kB * kLd;
    float* const delta = Ps + kB * kLdP;
    float* const lse_s = delta + kB;

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(BH));
    const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(BH));
    const int qblk = causal ? (nblk - 1 - slot) : slot;  // heaviest causal blocks first
    const int q0 = qblk * kB;
    const int64_t head = static_cast<int64_t>(bh) * N * D;
    load_tile<T, D>(Qs, q + head, q0, N);
    load_tile<T, D>(dOs, dout + head, q0, N);
    __syncthreads();
    load_row_terms<T, D>(delta, lse_s, dOs, o + head, lse + static_cast<int64_t>(bh) * N, q0, N);

    float dQ[4][G];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < G; ++j) dQ[i][j] = 0.f;

    const int kend = causal ? qblk + 1 : nblk;  // keys up to the block's last query
    for (int kb = 0; kb < kend; ++kb) {
        const int k0 = kb * kB;
        __syncthreads();  // the previous block is done with Ks, Vs, Ps
        load_tile<T, D>(Ks, k + head, k0, N);
        load_tile<T, D>(Vs, v + head, k0, N);
        __syncthreads();
        float s[4][4], p[4][4], dp[4][4];
        micro_abt<D>(s, Qs, Ks, ty, tx);
        probs(p, s, lse_s, q0, k0, N, causal, c, ty, tx);
        micro_abt<D>(dp, dOs, Vs, ty, tx);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float dl = delta[ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * kLdP + tx + 16 * j] = p[i][j] * (dp[i][j] - dl);
        }
        __syncthreads();
        micro_ab<D>(dQ, Ps, Ks, ty, tx);  // dQ[q][dim] += sum_key dS[q][key] K[key][dim]
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty * 4 + i;
        if (row < N) {
#pragma unroll
            for (int g = 0; g < D / 64; ++g)
                Elem<T>::store4(dq + head + static_cast<int64_t>(row) * D + 64 * g + 4 * tx,
                                make_float4(dQ[i][4 * g] * scale, dQ[i][4 * g + 1] * scale, dQ[i][4 * g + 2] * scale,
                                            dQ[i][4 * g + 3] * scale));
        }
    }
}

template <typename T, int D>
int launch_t(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int64_t BH, int64_t N, bool causal, cudaStream_t stream) {
    constexpr int smem = (4 * kB * ld_of<D>() + kB * kLdP + 2 * kB) * static_cast<int>(sizeof(float));
    if (cudaFuncSetAttribute(attn_bwd_kv_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_q_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return ATTN_ERR_LAUNCH;
    const int64_t nblk = (N + kB - 1) / kB;
    const int64_t blocks = nblk * BH;
    if (blocks > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    const double dd = static_cast<double>(D);
    const float c = static_cast<float>(1.4426950408889634 / std::sqrt(dd));
    const float scale = static_cast<float>(1.0 / std::sqrt(dd));
    const T* qt = static_cast<const T*>(q);
    const T* kt = static_cast<const T*>(k);
    const T* vt = static_cast<const T*>(v);
    const T* ot = static_cast<const T*>(o);
    const T* dot = static_cast<const T*>(dout);
    attn_bwd_kv_kernel<T, D><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
        qt, kt, vt, ot, dot, lse, static_cast<T*>(dk), static_cast<T*>(dv), static_cast<int>(N),
        static_cast<int>(BH), static_cast<int>(nblk), causal ? 1 : 0, c, scale);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    attn_bwd_q_kernel<T, D><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
        qt, kt, vt, ot, dot, lse, static_cast<T*>(dq), static_cast<int>(N), static_cast<int>(BH),
        static_cast<int>(nblk), causal ? 1 : 0, c, scale);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

int launch_bwd_f32(const float* q, const float* k, const float* v, const float* o, const float* dout,
                   const float* lse, float* dq, float* dk, float* dv, int64_t BH, int64_t N, int64_t d, bool causal,
                   cudaStream_t stream) {
    if (N > 0x7FFFFFFFll - kB || BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    if (d == 64) return launch_t<float, 64>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, stream);
    if (d == 128) return launch_t<float, 128>(q, k, v, o, dout, lse, dq, dk, dv, BH, N, causal, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
