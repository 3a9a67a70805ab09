// Throughput probes for the rooflines the attention kernels are measured against.
// FFMA: every SM runs one block of 1024 threads; each thread runs kChains independent chains of
// fused multiply-adds (a * m + b, with m and b chosen so the values stay bounded), so the FMA
// pipes never wait on a dependency. The caller times the launch with CUDA events on `stream`;
// the flop count of the launch is returned on the host.
// SFU: the same grid, each thread running kChains independent chains of a = 2^(-a)
// (ex2.approx, the exponential the softmax uses; a stays in [0.5, 1]), so the special-function
// units never wait on a dependency; the count of exponentials is returned.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kThreads, 1) ffma_probe_kernel(float* sink, int64_t iters) {
    float a[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) a[c] = 0.1f * static_cast<float>(c) + 1e-4f * static_cast<float>(threadIdx.x);
    const float m = 0.999f, b = 1e-3f;
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[c]) : "f"(m), "f"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += a[c];
    sink[static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads, 1) sfu_probe_kernel(float* sink, int64_t iters) {
    float a[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) a[c] = 0.5f + 0.05f * static_cast<float>(c) + 1e-5f * static_cast<float>(threadIdx.x);
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("{\n\t.reg .f32 t;\n\tneg.f32 t, %0;\n\tex2.approx.ftz.f32 %0, t;\n\t}" : "+f"(a[c]));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += a[c];
    sink[static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x] = s;
}

// Shared argument and device checks of the probes; on success *sms holds the SM count.
int probe_checks(const float* sink, int64_t sink_floats, int64_t iters, const double* count, int* sms) {
    if (sink == nullptr || count == nullptr || iters < 1 || iters > (int64_t{1} << 24)) return ATTN_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_DEVICE;
    if (major != 10 || minor != 3) return ATTN_ERR_DEVICE;
    if (sink_floats < static_cast<int64_t>(*sms) * kThreads) return ATTN_ERR_WORKSPACE;
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_probe_sfu_ex2(float* sink, int64_t sink_floats, int64_t iters, double* ops, void* stream) {
    int sms = 0;
    const int st = probe_checks(sink, sink_floats, iters, ops, &sms);
    if (st != ATTN_OK) return st;
    sfu_probe_kernel<<<sms, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    *ops = static_cast<double>(sms) * kThreads * kChains * static_cast<double>(iters);
    return ATTN_OK;
}

extern "C" int attn_probe_fp32_fma(float* sink, int64_t sink_floats, int64_t iters, double* flop, void* stream) {
    int sms = 0;
    const int st = probe_checks(sink, sink_floats, iters, flop, &sms);
    if (st != ATTN_OK) return st;
    ffma_probe_kernel<<<sms, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    *flop = 2.0 * static_cast<double>(sms) * kThreads * kChains * static_cast<double>(iters);
    return ATTN_OK;
}
