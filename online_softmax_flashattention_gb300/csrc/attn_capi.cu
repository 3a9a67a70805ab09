// The C ABI of libattn.so (declared in include/attn.h): argument checks, dispatch to the
// fp32 (FFMA) or bf16/fp16 (tcgen05) online kernels or to the materialised ablation, and
// status reporting. Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "attn.h"
#include <algorithm>
#include <vector>

#include "attn_internal.h"

namespace {

constexpr int64_t kHeadDim = 64;

size_t elem_size(int dtype) { return dtype == ATTN_F32 ? 4 : 2; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Host-side fault injection for tests: ATTN_FAULT=launch makes every entry point report a
// launch failure after its argument checks, without launching anything.
bool inject_launch_fault() {
    const char* f = std::getenv("ATTN_FAULT");
    return f != nullptr && std::strcmp(f, "launch") == 0;
}

// Common checks of the entry points over [B, H, N, d] tensors. On success *bh and *bytes
// hold B*H and the size of one tensor; *skip is set when there is no work. d = 128 is
// accepted only where `wide` is set (the forward entry points).
int check_common(const void* q, const void* k, const void* v, const void* o, int64_t B, int64_t H,
                 int64_t N, int64_t d, int causal, int dtype, int64_t* bh, size_t* bytes,
                 bool* skip, bool wide = false) {
    if (B < 0 || H < 0 || N < 0 || d < 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
    if (d != kHeadDim && !(wide && d == 2 * kHeadDim)) return ATTN_ERR_UNSUPPORTED;
    if (N > ATTN_MAX_N) return ATTN_ERR_UNSUPPORTED;
    if (B > 0x7FFFFFFFll || H > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    *bh = BH;
    *skip = (BH == 0 || N == 0);
    if (*skip) return ATTN_OK;
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return ATTN_ERR_ALIGN;
    *bytes = static_cast<size_t>(BH) * static_cast<size_t>(N) * static_cast<size_t>(d) * elem_size(dtype);
    if (overlap(o, *bytes, q, *bytes) || overlap(o, *bytes, k, *bytes) || overlap(o, *bytes, v, *bytes))
        return ATTN_ERR_ALIAS;
    return ATTN_OK;
}

// The kernels are built for sm_103a only; any other device is refused up front. The compute
// capability and SM count of each device ordinal are read once and kept.
int check_device(int* num_sms) {
    constexpr int kMaxDev = 64;
    static int sms_of[kMaxDev];  // 0: not read yet, -1: not an sm_103 device, else the SM count
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    int known = (dev >= 0 && dev < kMaxDev) ? __atomic_load_n(&sms_of[dev], __ATOMIC_ACQUIRE) : 0;
    if (known == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_DEVICE;
        known = (major == 10 && minor == 3 && n > 0) ? n : -1;
        if (dev >= 0 && dev < kMaxDev) __atomic_store_n(&sms_of[dev], known, __ATOMIC_RELEASE);
    }
    if (known < 0) return ATTN_ERR_DEVICE;
    *num_sms = known;
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H,
             int64_t N, int64_t d, int causal, int dtype, void* stream) {
    return attn_fwd_lse(q, k, v, o, nullptr, B, H, N, d, causal, dtype, stream);
}

int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                 int64_t H, int64_t N, int64_t d, int causal, int dtype, void* stream) {
    int64_t BH = 0;
    size_t bytes = 0;
    bool skip = false;
    int st = check_common(q, k, v, o, B, H, N, d, causal, dtype, &BH, &bytes, &skip, true);
    if (st != ATTN_OK || skip) return st;
    if (lse != nullptr) {
        if (!aligned(lse, 4)) return ATTN_ERR_ALIGN;
        const size_t lbytes = static_cast<size_t>(BH) * static_cast<size_t>(N) * sizeof(float);
        if (overlap(lse, lbytes, q, bytes) || overlap(lse, lbytes, k, bytes) || overlap(lse, lbytes, v, bytes) ||
            overlap(lse, lbytes, o, bytes))
            return ATTN_ERR_ALIAS;
    }
    int num_sms = 0;
    if ((st = check_device(&num_sms)) != ATTN_OK) return st;
    if (inject_launch_fault()) return ATTN_ERR_LAUNCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == ATTN_F32)
        return attn::launch_fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), static_cast<float*>(o), lse, BH, N, d,
                                    causal != 0, num_sms, s);
    return attn::launch_fwd_tc(q, k, v, o, lse, BH, N, d, causal != 0, dtype == ATTN_BF16, num_sms, s);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N,
             int64_t d, int causal, int dtype, void* stream) {
    int64_t BH = 0;
    size_t bytes = 0;
    bool skip = false;
    // q, k, v and o get the forward's checks (o plays the output's part, so it may not alias
    // q, k or v); then the backward's own tensors.
    int st = check_common(q, k, v, o, B, H, N, d, causal, dtype, &BH, &bytes, &skip, true);
    if (st != ATTN_OK || skip) return st;
    if (!dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (!aligned(dout, 16) || !aligned(lse, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
        return ATTN_ERR_ALIGN;
    const size_t lbytes = static_cast<size_t>(BH) * static_cast<size_t>(N) * sizeof(float);
    const void* ins[6] = {q, k, v, o, dout, lse};
    const size_t in_bytes[6] = {bytes, bytes, bytes, bytes, bytes, lbytes};
    void* outs[3] = {dq, dk, dv};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlap(outs[a], bytes, ins[b], in_bytes[b])) return ATTN_ERR_ALIAS;
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], bytes, outs[b], bytes)) return ATTN_ERR_ALIAS;
    }
    int num_sms = 0;
    if ((st = check_device(&num_sms)) != ATTN_OK) return st;
    if (inject_launch_fault()) return ATTN_ERR_LAUNCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == ATTN_F32)
        return attn::launch_bwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), static_cast<const float*>(o),
                                    static_cast<const float*>(dout), lse, static_cast<float*>(dq),
                                    static_cast<float*>(dk), static_cast<float*>(dv), BH, N, d, causal != 0, s);
    return attn::launch_bwd_tc(q, k, v, o, dout, lse, dq, dk, dv, BH, N, d, causal != 0, dtype == ATTN_BF16, num_sms,
                               s);
}

size_t attn_kvcache_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int num_splits,
                                    int dtype) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < Nq || B > 0x7FFFFFFFll || H > 0x7FFFFFFFll) return 0;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16) return 0;
    if (d != kHeadDim && d != 2 * kHeadDim) return 0;
    int num_sms = 0;
    if (num_splits == 0 && check_device(&num_sms) != ATTN_OK) return 0;
    return attn::decode_workspace_bytes(B * H, Nq, Nk, d, num_splits, dtype, num_sms);
}

int attn_fwd_kvcache(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                     size_t workspace_bytes, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                     int causal, int dtype, int num_splits, void* stream) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (Nq > Nk || num_splits < 0) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_UNSUPPORTED;
    if (d != kHeadDim && d != 2 * kHeadDim) return ATTN_ERR_UNSUPPORTED;
    if (Nk > ATTN_MAX_N || Nq > 8 * 65535ll || num_splits > ATTN_KV_MAX_SPLITS) return ATTN_ERR_UNSUPPORTED;
    if (B > 0x7FFFFFFFll || H > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
    if (BH == 0 || Nq == 0) return ATTN_OK;
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return ATTN_ERR_ALIGN;
    const size_t esz = elem_size(dtype);
    const size_t qbytes = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * static_cast<size_t>(d) * esz;
    const size_t kbytes = static_cast<size_t>(BH) * static_cast<size_t>(Nk) * static_cast<size_t>(d) * esz;
    if (overlap(o, qbytes, q, qbytes) || overlap(o, qbytes, k, kbytes) || overlap(o, qbytes, v, kbytes))
        return ATTN_ERR_ALIAS;
    const size_t lbytes = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * sizeof(float);
    if (lse != nullptr) {
        if (!aligned(lse, 4)) return ATTN_ERR_ALIGN;
        if (overlap(lse, lbytes, q, qbytes) || overlap(lse, lbytes, k, kbytes) || overlap(lse, lbytes, v, kbytes) ||
            overlap(lse, lbytes, o, qbytes))
            return ATTN_ERR_ALIAS;
    }
    // An explicit share count is checked against the workspace before the device is queried;
    // the balanced plan needs the SM count and the kernel's occupancy first.
    int num_sms = 0;
    int st = ATTN_OK;
    if (num_splits == 0 && (st = check_device(&num_sms)) != ATTN_OK) return st;
    const size_t need = attn::decode_workspace_bytes(BH, Nq, Nk, d, num_splits, dtype, num_sms);
    // (A balanced plan of one piece per segment needs none; the launch re-checks the size.)
    const bool needs_ws = num_splits > 1 || (num_splits == 0 && need > 0);
    if (needs_ws) {
        if (need == 0) return ATTN_ERR_UNSUPPORTED;
        if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
        if (overlap(workspace, need, q, qbytes) || overlap(workspace, need, k, kbytes) ||
            overlap(workspace, need, v, kbytes) || overlap(workspace, need, o, qbytes) ||
            (lse != nullptr && overlap(workspace, need, lse, lbytes)))
            return ATTN_ERR_ALIAS;
    }
    if (num_splits != 0 && (st = check_device(&num_sms)) != ATTN_OK) return st;
    if (inject_launch_fault()) return ATTN_ERR_LAUNCH;
    return attn::launch_decode(q, k, v, o, lse, workspace, workspace_bytes, BH, Nq, Nk, d, causal != 0, dtype,
                               num_splits, num_sms, static_cast<cudaStream_t>(stream));
}

size_t attn_materialized_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B < 0 || H < 0 || N < 0 || B > 0x7FFFFFFFll || H > 0x7FFFFFFFll) return 0;
    const size_t per = attn::materialized_head_bytes(N);
    if (per == 0 && N != 0) return 0;
    const size_t bh = static_cast<size_t>(B) * static_cast<size_t>(H);
    if (bh != 0 && per > SIZE_MAX / bh) return 0;
    return per * bh;
}

int attn_fwd_materialized(const void* q, const void* k, const void* v, void* o, void* workspace,
                          size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d,
                          int causal, int dtype, void* stream) {
    int64_t BH = 0;
    size_t bytes = 0;
    bool skip = false;
    int st = check_common(q, k, v, o, B, H, N, d, causal, dtype, &BH, &bytes, &skip);
    if (st != ATTN_OK || skip) return st;
    const size_t per = attn::materialized_head_bytes(N);
    if (per == 0) return ATTN_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < per) return ATTN_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
    if (overlap(workspace, workspace_bytes, q, bytes) || overlap(workspace, workspace_bytes, k, bytes) ||
        overlap(workspace, workspace_bytes, v, bytes) || overlap(workspace, workspace_bytes, o, bytes))
        return ATTN_ERR_ALIAS;
    int num_sms = 0;
    if ((st = check_device(&num_sms)) != ATTN_OK) return st;
    if (inject_launch_fault()) return ATTN_ERR_LAUNCH;
    int64_t group = static_cast<int64_t>(workspace_bytes / per);
    if (group > BH) group = BH;
    if (group > 65535) group = 65535;
    const size_t head_elems = static_cast<size_t>(N) * kHeadDim;
    const size_t esz = elem_size(dtype);
    for (int64_t h0 = 0; h0 < BH; h0 += group) {
        const int64_t hc = (BH - h0 < group) ? (BH - h0) : group;
        const size_t off = static_cast<size_t>(h0) * head_elems * esz;
        st = attn::launch_materialized(static_cast<const uint8_t*>(q) + off,
                                       static_cast<const uint8_t*>(k) + off,
                                       static_cast<const uint8_t*>(v) + off,
                                       static_cast<uint8_t*>(o) + off, workspace, per, hc, N,
                                       causal != 0, dtype, static_cast<cudaStream_t>(stream));
        if (st != ATTN_OK) return st;
    }
    return ATTN_OK;
}

int attn_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000 || timeout_ns > 2000000000ull) return ATTN_ERR_INVALID_ARG;
    int num_sms = 0;
    int st = check_device(&num_sms);
    if (st != ATTN_OK) return st;
    return attn::launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream));
}

int attn_device_status(void* stream, int clear) {
    unsigned err = 0, berr = 0, derr = 0, dterr = 0;
    int st = attn::tc_device_error(static_cast<cudaStream_t>(stream), clear != 0, &err);
    if (st != ATTN_OK) return st;
    if ((st = attn::bwd_tc_device_error(clear != 0, &berr)) != ATTN_OK) return st;
    if ((st = attn::decode_device_error(clear != 0, &derr)) != ATTN_OK) return st;
    if ((st = attn::decode_tc_device_error(clear != 0, &dterr)) != ATTN_OK) return st;
    return (err || berr || derr || dterr) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or causal not 0/1)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported (head dim 64 or 128, 64 for the ablation; dtype f32/bf16/f16; size limits)";
        case ATTN_ERR_ALIGN: return "pointer not aligned (tensors 16 bytes, workspace 256 bytes)";
        case ATTN_ERR_ALIAS: return "output or workspace overlaps another buffer";
        case ATTN_ERR_DEVICE: return "current device is not sm_103 or a CUDA query failed";
        case ATTN_ERR_LAUNCH: return "kernel launch failed";
        case ATTN_ERR_TIMEOUT: return "a device-side wait ran out its time limit";
        case ATTN_ERR_WORKSPACE: return "workspace missing or smaller than one head needs";
        default: return "unknown status";
    }
}

int attn_plan_launch_order(const int32_t* weights, int64_t n, int32_t fixed, int32_t num_sms, uint16_t* order) {
    // Each capacity try costs n * num_sms steps; the bounds keep the whole search well under a
    // second (the kernels plan at most 2048 items over the device's SMs).
    if (!weights || !order || n < 1 || n > 8192 || fixed < 0 || fixed > (1 << 24) || num_sms < 1 ||
        num_sms > 1024 || n * num_sms > (int64_t{1} << 20))
        return ATTN_ERR_INVALID_ARG;
    std::vector<int> w(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) {
        if (weights[i] < 0 || weights[i] > (1 << 24)) return ATTN_ERR_INVALID_ARG;
        w[static_cast<size_t>(i)] = weights[i];
    }
    const std::vector<uint16_t> ord = attn::plan_order_compute(w, fixed, num_sms);
    std::copy(ord.begin(), ord.end(), order);
    return ATTN_OK;
}

int attn_abi_version(void) { return (1 << 16) | 9; }

}  // extern "C"
