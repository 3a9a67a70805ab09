// Materialised attention, kept as an ablation of the online path: it writes the whole
// N x N score matrix to device memory and reads it back, which is the traffic the flash
// kernels remove. The three stages follow attention.cu's naive path (scoresQKt,
// softmaxRows, weightedV) and the "Attention by hand" section of the "Flash attention in
// PyTorch, then in Triton" page (masked fill with minus infinity, row softmax, times v):
//   1. S = q k^T / sqrt(d), masked entries set to -inf, written in full (fp32);
//   2. per row: max over S, then P = exp(S - max) written to a second N x N buffer and the
//      row total to a vector (S read twice, P written once);
//   3. o = (P v) / total (P read once).
// That is five passes over N^2 floats per head: 5 * 4 * N^2 bytes.
// Every input type is widened to fp32; o is rounded to the input type (nearest even).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kD = 64;
constexpr int kT = 64;   // tile edge of both products
constexpr int kLd = 68;  // padded shared row stride (floats)
constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

struct Ws {
    float* S;
    float* P;
    float* total;
};

__device__ __forceinline__ Ws head_ws(void* ws, size_t head_bytes, size_t nn_bytes, int64_t h) {
    uint8_t* b = static_cast<uint8_t*>(ws) + static_cast<size_t>(h) * head_bytes;
    return {reinterpret_cast<float*>(b), reinterpret_cast<float*>(b + nn_bytes),
            reinterpret_cast<float*>(b + 2 * nn_bytes)};
}

// Stage 1. Grid (key tiles, query tiles, heads); thread (ty, tx) owns rows ty*4+i, keys tx+16j.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    scores_kernel(const T* __restrict__ q, const T* __restrict__ k, void* ws, size_t head_bytes,
                  size_t nn_bytes, int N, int causal, float scale) {
    __shared__ __align__(16) float Qs[kT * kLd];
    __shared__ __align__(16) float Ks[kT * kLd];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int kb = blockIdx.x * kT, qb = blockIdx.y * kT;
    const int64_t h = blockIdx.z;
    const T* qh = q + h * N * kD;
    const T* kh = k + h * N * kD;
    for (int idx = threadIdx.x; idx < kT * kD; idx += kThreads) {
        const int r = idx / kD, e = idx % kD;
        Qs[r * kLd + e] = (qb + r < N) ? to_f(qh[static_cast<int64_t>(qb + r) * kD + e]) : 0.f;
        Ks[r * kLd + e] = (kb + r < N) ? to_f(kh[static_cast<int64_t>(kb + r) * kD + e]) : 0.f;
    }
    __syncthreads();
    float s[4][4] = {};
    for (int e = 0; e < kD; e += 4) {
        float4 qa[4], kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qa[i] = *reinterpret_cast<const float4*>(Qs + (ty * 4 + i) * kLd + e);
#pragma unroll
        for (int j = 0; j < 4; ++j) kv[j] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * j) * kLd + e);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                s[i][j] += qa[i].x * kv[j].x + qa[i].y * kv[j].y + qa[i].z * kv[j].z + qa[i].w * kv[j].w;
    }
    Ws w = head_ws(ws, head_bytes, nn_bytes, h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = qb + ty * 4 + i;
        if (row >= N) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = kb + tx + 16 * j;
            if (col >= N) continue;
            w.S[static_cast<int64_t>(row) * N + col] = (causal && col > row) ? -INFINITY : s[i][j] * scale;
        }
    }
}

// Stage 2. One block per row (grid (N, heads)): pass 1 finds the max, pass 2 writes
// exp(S - max) to P and totals it.
__global__ void __launch_bounds__(kThreads)
    softmax_rows_kernel(void* ws, size_t head_bytes, size_t nn_bytes, int N) {
    __shared__ float red[kThreads / 32];
    const int64_t row = blockIdx.x;
    const Ws w = head_ws(ws, head_bytes, nn_bytes, blockIdx.y);
    const float* line = w.S + row * N;
    float* out = w.P + row * N;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

    float best = -INFINITY;
    for (int j = threadIdx.x; j < N; j += kThreads) best = fmaxf(best, line[j]);
    for (int off = 16; off > 0; off >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) red[wid] = best;
    __syncthreads();
    best = red[0];
    for (int i = 1; i < kThreads / 32; ++i) best = fmaxf(best, red[i]);
    __syncthreads();

    float tot = 0.f;
    for (int j = threadIdx.x; j < N; j += kThreads) {
        const float e = expf(line[j] - best);
        out[j] = e;
        tot += e;
    }
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane == 0) red[wid] = tot;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kThreads / 32; ++i) t += red[i];
        w.total[row] = t;
    }
}

// Stage 3. Grid (query tiles, heads); thread (ty, tx) owns rows ty*4+i, dims tx*4+j.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    weighted_v_kernel(const T* __restrict__ v, T* __restrict__ o, void* ws, size_t head_bytes,
                      size_t nn_bytes, int N) {
    __shared__ __align__(16) float Ps[kT * kLd];
    __shared__ __align__(16) float Vs[kT * kLd];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int qb = blockIdx.x * kT;
    const int64_t h = blockIdx.y;
    const T* vh = v + h * N * kD;
    const Ws w = head_ws(ws, head_bytes, nn_bytes, h);
    float acc[4][4] = {};
    for (int kb = 0; kb < N; kb += kT) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kT * kT; idx += kThreads) {
            const int r = idx / kT, c = idx % kT;
            Ps[r * kLd + c] = (qb + r < N && kb + c < N) ? w.P[static_cast<int64_t>(qb + r) * N + kb + c] : 0.f;
            Vs[r * kLd + c] = (kb + r < N) ? to_f(vh[static_cast<int64_t>(kb + r) * kD + c]) : 0.f;
        }
        __syncthreads();
        for (int kk = 0; kk < kT; kk += 4) {
            float4 pa[4], vb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pa[i] = *reinterpret_cast<const float4*>(Ps + (ty * 4 + i) * kLd + kk);
#pragma unroll
            for (int u = 0; u < 4; ++u) vb[u] = *reinterpret_cast<const float4*>(Vs + (kk + u) * kLd + 4 * tx);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pw[4] = {pa[i].x, pa[i].y, pa[i].z, pa[i].w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[i][0] += pw[u] * vb[u].x;
                    acc[i][1] += pw[u] * vb[u].y;
                    acc[i][2] += pw[u] * vb[u].z;
                    acc[i][3] += pw[u] * vb[u].w;
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = qb + ty * 4 + i;
        if (row >= N) continue;
        const float inv = 1.f / w.total[row];
        T* dst = o + h * N * kD + static_cast<int64_t>(row) * kD + 4 * tx;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = from_f<T>(acc[i][j] * inv);
    }
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <typename T>
int launch_t(const void* q, const void* k, const void* v, void* o, void* ws, size_t head_bytes,
             int64_t heads, int64_t N, bool causal, cudaStream_t stream) {
    const size_t nn_bytes = round256(static_cast<size_t>(N) * static_cast<size_t>(N) * sizeof(float));
    const unsigned tiles = static_cast<unsigned>((N + kT - 1) / kT);
    const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kD)));
    scores_kernel<T><<<dim3(tiles, tiles, static_cast<unsigned>(heads)), kThreads, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), ws, head_bytes, nn_bytes,
        static_cast<int>(N), causal ? 1 : 0, scale);
    softmax_rows_kernel<<<dim3(static_cast<unsigned>(N), static_cast<unsigned>(heads)), kThreads, 0, stream>>>(
        ws, head_bytes, nn_bytes, static_cast<int>(N));
    weighted_v_kernel<T><<<dim3(tiles, static_cast<unsigned>(heads)), kThreads, 0, stream>>>(
        static_cast<const T*>(v), static_cast<T*>(o), ws, head_bytes, nn_bytes, static_cast<int>(N));
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace

size_t materialized_head_bytes(int64_t N) {
    if (N < 0 || N > (static_cast<int64_t>(1) << 30)) return 0;
    const size_t nn = static_cast<size_t>(N) * static_cast<size_t>(N);
    if (N > 0 && nn / static_cast<size_t>(N) != static_cast<size_t>(N)) return 0;
    return 2 * round256(nn * sizeof(float)) + round256(static_cast<size_t>(N) * sizeof(float));
}

int launch_materialized(const void* q, const void* k, const void* v, void* o, void* ws,
                        size_t head_ws_bytes, int64_t heads, int64_t N, bool causal, int dtype,
                        cudaStream_t stream) {
    if (N > 65535 * static_cast<int64_t>(kT) || heads > 65535) return ATTN_ERR_UNSUPPORTED;
    switch (dtype) {
        case ATTN_F32: return launch_t<float>(q, k, v, o, ws, head_ws_bytes, heads, N, causal, stream);
        case ATTN_BF16: return launch_t<__nv_bfloat16>(q, k, v, o, ws, head_ws_bytes, heads, N, causal, stream);
        case ATTN_F16: return launch_t<__half>(q, k, v, o, ws, head_ws_bytes, heads, N, causal, stream);
        default: return ATTN_ERR_UNSUPPORTED;
    }
}

}  // namespace attn
