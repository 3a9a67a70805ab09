// attn_fwd_materialized_noalloc: the materialised ablation with its scratch in a fixed array
// compiled into the library instead of a caller-supplied workspace. It has no counterpart on the
// attention pages; it reuses the three kernels of attn_materialized.cu unchanged.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"
#include "attn_internal.h"

// Materialised path without any allocation.
//
// Some callers cannot allocate device memory: code running where cudaMalloc is forbidden or
// unsafe (inside a memory-pool-restricted service, a plugin whose host owns all
// allocations, or a path that must not synchronise the device the way cudaMalloc/cudaFree
// can), or that simply has no workspace buffer to hand over. For them the scratch of the
// materialised path (S, P and row totals) lives in a fixed array compiled into this
// library, and the caller passes only q, k, v and o.
//
// The array is a file-scope __device__ variable in this translation unit alone, so its module
// (and the memory) is loaded only by the first call of this entry point on a device; from then
// on that GPU holds ATTN_NOALLOC_SCRATCH_BYTES for as long as the process lives. Host code may
// not use the array's name as a device address: every call looks the address up with
// cudaGetSymbolAddress on the current device (so a device reset, which reloads the module,
// cannot leave a stale address behind). The first call on a device loads the module and
// should therefore come before any stream capture. All calls share the array: calls whose
// kernels overlap on the GPU (for example on two streams without ordering) race on it.
// Nothing in it has to start at zero: each call writes every score, every probability and
// every row total before reading it.
// ---------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace attn {
namespace {

constexpr int64_t kD = 64;

// Device address of the scratch array on the current device.
int noalloc_scratch(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_DEVICE;
    *out = p;
    return ATTN_OK;
}

bool noalloc_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace attn

extern "C" int attn_fwd_materialized_noalloc(const void* q, const void* k, const void* v, void* o,
                                             int64_t B, int64_t H, int64_t N, int64_t d, int causal,
                                             int dtype, void* stream) {
    using namespace attn;
    if (B < 0 || H < 0 || N < 0 || d < 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
    if (d != kD) return ATTN_ERR_UNSUPPORTED;
    if (B > 0x7FFFFFFFll || H > 0x7FFFFFFFll || B * H > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    // One head's scratch must fit the fixed array (N <= ATTN_NOALLOC_MAX_N).
    if (N > ATTN_NOALLOC_MAX_N) return ATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH == 0 || N == 0) return ATTN_OK;
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if (mis & 15u) return ATTN_ERR_ALIGN;
    const size_t esz = dtype == ATTN_F32 ? 4 : 2;
    const size_t bytes = static_cast<size_t>(BH) * static_cast<size_t>(N) * kD * esz;
    if (noalloc_overlap(o, bytes, q, bytes) || noalloc_overlap(o, bytes, k, bytes) ||
        noalloc_overlap(o, bytes, v, bytes))
        return ATTN_ERR_ALIAS;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_DEVICE;
    if (major != 10 || minor != 3) return ATTN_ERR_DEVICE;
    const size_t per = materialized_head_bytes(N);
    if (per == 0 || per > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    int st = noalloc_scratch(&scratch);
    if (st != ATTN_OK) return st;
    int64_t group = static_cast<int64_t>(ATTN_NOALLOC_SCRATCH_BYTES / per);
    if (group > BH) group = BH;
    if (group > 65535) group = 65535;
    const size_t head_elems = static_cast<size_t>(N) * kD;
    for (int64_t h0 = 0; h0 < BH; h0 += group) {
        const int64_t hc = (BH - h0 < group) ? (BH - h0) : group;
        const size_t off = static_cast<size_t>(h0) * head_elems * esz;
        st = launch_materialized(static_cast<const uint8_t*>(q) + off, static_cast<const uint8_t*>(k) + off,
                                 static_cast<const uint8_t*>(v) + off, static_cast<uint8_t*>(o) + off, scratch,
                                 per, hc, N, causal != 0, dtype, static_cast<cudaStream_t>(stream));
        if (st != ATTN_OK) return st;
    }
    return ATTN_OK;
}
