/*
 * attn.h — C ABI of libattn.so: exact scaled-dot-product attention forward on GB300
 * (sm_103a), computed tile by tile with the online-softmax recurrence.
 *
 * Operation (all entry points). For every batch b < B, head h < H and query row i < N:
 *
 *     o[b,h,i,:] = sum_{j in vis(i)} softmax_j( q[b,h,i,:] . k[b,h,j,:] / sqrt(d) ) * v[b,h,j,:]
 *
 * with vis(i) = {0 .. N-1}, or {0 .. i} when causal (the diagonal is kept). This is the
 * definition on the "Flash attention in PyTorch, then in Triton" page, section "Attention's
 * table of scores"; the tiled evaluation with a running maximum, running denominator and
 * running output is the online softmax of its section "Flash attention" and of attention.cu
 * (attentionOnline). The scale 1/sqrt(d) is fixed, as in both pages.
 *
 * Layout. q, k, v and o are contiguous row-major [B, H, N, d] device arrays of one element
 * type (dtype). Element (b,h,i,e) lives at offset ((b*H + h)*N + i)*d + e.
 *
 * Ownership and synchronisation. The caller owns every buffer and the stream. Calls are
 * stream-ordered and asynchronous: they validate, enqueue on `stream` (a cudaStream_t;
 * NULL is the legacy default stream) and return. The library keeps no state between calls
 * apart from host-side caches: per device, its properties, driver entry points and kernel
 * attributes (set once); the forward's tensor maps of the last 8 (pointer, shape) combinations;
 * and causal launch orders per problem shape and kernel (at most 256 entries, a few KiB each).
 * It is safe to call from several host threads (the caches are guarded by mutexes). attn_fwd
 * allocates no device memory.
 *
 * Errors. Every entry point returns an attn_status_t and never exits the process.
 * Argument checks happen before any launch; a non-OK status means nothing was enqueued.
 * Faults that happen on the device surface at the caller's next synchronisation, as for
 * any CUDA call. A device-side wait that exceeds its time limit stops the kernel, leaves
 * o partly written and records ATTN_ERR_TIMEOUT, which attn_device_status() reports.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_F32 = 0,  /* float32 in and out; FFMA path with fp32 accumulation */
    ATTN_BF16 = 1, /* bfloat16 in and out; tcgen05 tensor cores, fp32 accumulation */
    ATTN_F16 = 2   /* float16 in and out; tcgen05 tensor cores, fp32 accumulation */
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null pointer with work to do, negative size, causal not 0/1 */
    ATTN_ERR_UNSUPPORTED = 2, /* head width not taken, unknown dtype, or a size beyond the limits */
    ATTN_ERR_ALIGN = 3,       /* a tensor or workspace pointer not 16-byte aligned */
    ATTN_ERR_ALIAS = 4,       /* o overlaps q, k, v (or the workspace overlaps a tensor) */
    ATTN_ERR_DEVICE = 5,      /* current device is not compute capability 10.3, or a CUDA
                                 query failed */
    ATTN_ERR_LAUNCH = 6,      /* the kernel launch itself failed (cudaGetLastError) */
    ATTN_ERR_TIMEOUT = 7,     /* a device-side wait ran out its time limit (see attn_device_status) */
    ATTN_ERR_WORKSPACE = 8    /* workspace null or smaller than one head needs */
} attn_status_t;

/* Largest N accepted by every entry point (2^30 rows per head). */
#define ATTN_MAX_N ((int64_t)1 << 30)

/*
 * attn_fwd — the flash (online-softmax) forward. N x N scores never reach device memory.
 *
 *   q, k, v : const device pointers, [B, H, N, d] of dtype, 16-byte aligned
 *   o       : device pointer, [B, H, N, d] of dtype, 16-byte aligned, must not overlap
 *             q, k or v; every element is written
 *   B, H, N : sizes >= 0, N <= ATTN_MAX_N, B*H < 2^31. B*H == 0 or N == 0 is a successful
 *             no-op (pointers may then be NULL)
 *   d       : head width, 64 or 128 (ATTN_ERR_UNSUPPORTED otherwise). The pages fix 64; 128
 *             is the other common width (scale 1/sqrt(128)). attn_fwd, attn_fwd_lse, attn_bwd
 *             and attn_fwd_kvcache take both; the materialised path takes 64.
 *   causal  : 0 (every key visible) or 1 (key j visible to query i iff j <= i)
 *   dtype   : attn_dtype_t. bf16/f16 inputs are multiplied on tcgen05 tensor cores with
 *             fp32 accumulation; the probabilities are rounded to the input type before
 *             they weigh v, and o is rounded to nearest even. f32 runs on FFMA.
 *   stream  : cudaStream_t (may be NULL)
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, int64_t B, int64_t H,
             int64_t N, int64_t d, int causal, int dtype, void* stream);

/*
 * attn_fwd_lse — attn_fwd that also stores each row's log-sum-exp, the log of the sum the
 * softmax divides by, which a backward pass needs to rebuild the probabilities from the
 * scores. Following the "Flash attention in PyTorch, then in Triton" page (section
 * "Backwards, and training with it": the forward kernel saves, per row, its running maximum
 * plus the base-2 log of its running total), it is kept in base 2:
 *
 *     lse[b,h,i] = log2( sum_{j in vis(i)} exp( q[b,h,i,:] . k[b,h,j,:] / sqrt(d) ) )
 *
 * (multiply by ln 2 for the natural-log value).
 *
 *   lse            : device pointer, float32 [B, H, N] contiguous, 4-byte aligned, must not
 *                    overlap q, k, v or o; every element is written
 *   other arguments: as attn_fwd; o is bit-identical to what attn_fwd writes.
 */
int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                 int64_t H, int64_t N, int64_t d, int causal, int dtype, void* stream);

/*
 * attn_bwd — gradients of the loss with respect to q, k and v, given its gradient with
 * respect to the output, dout: the backward pass of the "Flash attention in PyTorch, then in
 * Triton" page, section "Backwards, and training with it". With S = q k^T / sqrt(d) (masked
 * when causal) and P = softmax(S) rebuilt from the scores and the forward's log-sum-exps,
 *
 *     dv = P^T dout,   dP = dout v^T,   delta_i = sum_e dout[i,e] o[i,e],
 *     dS = P * (dP - delta),   dq = dS k / sqrt(d),   dk = dS^T q / sqrt(d).
 *
 * Two kernels as on the page (one program per key block writes dk and dv, one per query block
 * writes dq), so no program adds into another's rows. bf16/fp16 run on tcgen05 tensor cores
 * (products with bf16/fp16 operands and fp32 accumulation; P and dS are rounded to dtype before
 * the products that take them, as the forward rounds P); f32 runs on FFMA in fp32. Results are
 * rounded to dtype (RNE). Nothing is allocated. A device-side wait timeout is reported by
 * attn_device_status like the forward's.
 *
 *   q, k, v, o, dout : const device pointers, [B, H, N, d] of dtype, 16-byte aligned; o is the
 *                      forward's output for these q, k, v (from attn_fwd_lse)
 *   lse              : const device pointer, float32 [B, H, N], 16-byte aligned: the base-2
 *                      log-sum-exps attn_fwd_lse stored for the same q, k
 *   dq, dk, dv       : device pointers, [B, H, N, d] of dtype, 16-byte aligned; they must not
 *                      overlap each other or any input; every element is written (bf16/fp16:
 *                      dq's rows hold intermediate values until the last kernel of the call
 *                      overwrites them, so dq must not be read before the call completes)
 *   other arguments  : as attn_fwd (same checks and status codes)
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N,
             int64_t d, int causal, int dtype, void* stream);

/*
 * attn_fwd_kvcache — attention of Nq new queries against a key-value cache of Nk >= Nq rows:
 * the generation case that the "Flash attention in PyTorch, then in Triton" page names and
 * leaves out of its kernel (section "Backwards, and training with it"). The queries are the
 * last Nq positions of the sequence, so query i sits at position Nk - Nq + i and
 *
 *     o[b,h,i,:] = sum_{j in vis(i)} softmax_j( q[b,h,i,:] . k[b,h,j,:] / sqrt(d) ) v[b,h,j,:]
 *
 * with vis(i) = {0 .. Nk-1}, or {0 .. Nk-Nq+i} when causal (with Nq == Nk this is attn_fwd's
 * mask). The keys of each (head, group of queries) are cut into pieces that run on
 * different CTAs; every piece runs the page's online softmax (section "Flash attention") over
 * its keys and leaves its normalised output O_p and base-2 log-sum-exp lse_p, and a second
 * kernel merges the pieces the way the online softmax merges tiles: lse = log2 sum_p 2^lse_p,
 * o = sum_p 2^(lse_p - lse) O_p. A piece that covers all of its head's keys writes o directly.
 * The work is bound by reading the cache. Two or more bf16/f16 queries run in groups of up to
 * 128 on tcgen05 tensor cores (S = q k^T and o += P v with bf16/f16 operands and fp32
 * accumulation, P rounded to dtype before it weighs v, as attn_fwd does) where that measured
 * faster: always at d = 128; at d = 64 from 8 queries, from 3 on caches of 1024 keys or more
 * (and 2^18 cached rows in the call), and from 2 on caches of 32768 keys or more. Everything
 * else (one query, fp32, the short cases) runs in groups of up to 8 queries with all arithmetic
 * fp32 on CUDA cores. o is rounded to dtype (RNE). Nothing is allocated.
 *
 *   q, o          : device pointers, [B, H, Nq, d] of dtype, 16-byte aligned; o must not
 *                   overlap q, k, v, lse or the workspace
 *   k, v          : const device pointers, [B, H, Nk, d] of dtype, 16-byte aligned
 *   lse           : NULL, or device pointer float32 [B, H, Nq], 4-byte aligned, receiving each
 *                   row's base-2 log-sum-exp as attn_fwd_lse defines it; must not overlap the
 *                   other buffers
 *   workspace     : device pointer, 256-byte aligned, caller-owned fp32 scratch for the pieces'
 *                   partial results (contents on entry ignored, on exit unspecified); may be
 *                   NULL when no workspace is needed. It must not overlap any tensor.
 *   workspace_bytes: its size; attn_kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits, dtype)
 *                   with the same device current is enough; less returns ATTN_ERR_WORKSPACE
 *   Nq, Nk        : 0 <= Nq <= Nk <= ATTN_MAX_N, Nq <= 8 * 65535; Nq == 0 or B*H == 0 is a
 *                   successful no-op
 *   num_splits    : 0 — balanced: a persistent grid of as many CTAs as the device holds, each
 *                   streaming the same number of key tiles (within one; 128 keys, or 64 on
 *                   tensor cores at d = 128) of all heads' keys,
 *                   cut at head boundaries; 1 .. ATTN_KV_MAX_SPLITS — every (head, query
 *                   group) is cut into that many equal shares (shares past the last key are
 *                   empty and carry weight 0 in the merge).
 *   d             : head width, 64 or 128 (scale 1/sqrt(d))
 *   other arguments: as attn_fwd (dtype f32, bf16 or f16; causal 0/1).
 */
#define ATTN_KV_MAX_SPLITS 1024
int attn_fwd_kvcache(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                     size_t workspace_bytes, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                     int causal, int dtype, int num_splits, void* stream);

/* Bytes of workspace attn_fwd_kvcache needs: B*H*Nq*P rows of d + 1 floats in two regions
 * rounded up to 256 bytes, where P is num_splits, or for num_splits == 0 the most pieces the
 * balanced plan gives one head on the current device; 0 when every head is a single piece.
 * Returns 0 also for invalid sizes or dtype, on overflow, or (num_splits == 0) when the
 * current device cannot be queried. */
size_t attn_kvcache_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int num_splits,
                                    int dtype);

/*
 * attn_fwd_materialized — the same result by the materialised path of attention.cu
 * (scoresQKt, softmaxRows, weightedV): S = q k^T / sqrt(d) with masked entries set to
 * -inf, written in full as fp32; a three-pass safe softmax that writes exp(S - rowmax) to
 * a second N x N buffer and the row totals to a vector; then o = (P v) / rowtotal.
 * Kept as an ablation that moves 5 * 4 * N^2 bytes of scores per head.
 *
 *   workspace       : device pointer, 256-byte aligned, caller-owned scratch; it must not
 *                     overlap q, k, v or o. Contents on entry are ignored and on exit are
 *                     unspecified.
 *   workspace_bytes : its size. At least attn_materialized_workspace_bytes(1, 1, N) (one
 *                     head); heads are processed in groups of as many as fit, so
 *                     attn_materialized_workspace_bytes(B, H, N) processes all at once.
 *   other arguments : as attn_fwd; every dtype is computed in fp32 arithmetic.
 */
int attn_fwd_materialized(const void* q, const void* k, const void* v, void* o, void* workspace,
                          size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d,
                          int causal, int dtype, void* stream);

/* Bytes of workspace attn_fwd_materialized needs to process all B*H heads in one group:
 * B*H * (two N x N fp32 buffers + N fp32 row totals), each rounded up to 256 bytes.
 * Returns 0 for negative sizes or on overflow. */
size_t attn_materialized_workspace_bytes(int64_t B, int64_t H, int64_t N);

/*
 * attn_fwd_materialized_noalloc — the materialised path of attn_fwd_materialized with no
 * workspace argument and no allocation of any kind. (The attention pages have no counterpart:
 * this is a convenience of this library.) It is meant for callers that cannot allocate
 * device memory or hand over a scratch buffer — for example code running under an allocator
 * it does not own, or on a path that must not call cudaMalloc/cudaFree because those can
 * synchronise the device.
 *
 *   Scratch: a fixed array of ATTN_NOALLOC_SCRATCH_BYTES compiled into the library, in a
 *            module of its own: a GPU holds it from the first call of this entry point on that
 *            device until the process exits (callers of the other entry points never load it).
 *            Heads run in groups of as many as fit.
 *   Limit:   N <= ATTN_NOALLOC_MAX_N (one head's scores and probabilities must fit the
 *            array); larger N returns ATTN_ERR_UNSUPPORTED and launches nothing.
 *   Set-up:  every call looks up the array's device address (cudaGetSymbolAddress) on the
 *            current device, so a device reset cannot leave a stale address; the first call on
 *            a device also loads the array's module, so make it before capturing a stream
 *            into a graph.
 *   Sharing: all calls use the same array, which keeps the previous call's contents (no call
 *            depends on them: everything is written before it is read). Calls whose kernels
 *            overlap on the GPU — unordered streams, several host threads — race on it.
 *   Other arguments, layout and errors: as attn_fwd.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
#define ATTN_NOALLOC_MAX_N ((int64_t)2896)
int attn_fwd_materialized_noalloc(const void* q, const void* k, const void* v, void* o, int64_t B,
                                  int64_t H, int64_t N, int64_t d, int causal, int dtype,
                                  void* stream);

/*
 * attn_device_status — synchronises `stream`, then reports whether any kernel of this
 * library on the current device recorded a device-side wait timeout since the flag was
 * last cleared. Returns ATTN_OK or ATTN_ERR_TIMEOUT (ATTN_ERR_DEVICE if a CUDA call
 * fails). clear != 0 resets the flag.
 */
int attn_device_status(void* stream, int clear);

/*
 * attn_selftest_wait_timeout — exercises the device-side timeout path without any fault: one
 * warp waits on an mbarrier that nothing arrives on, with a limit of timeout_ns (1 us .. 2 s);
 * when it runs out the warp records ATTN_ERR_TIMEOUT the way every kernel of this library does
 * and returns, leaving the context usable. attn_device_status then reports the timeout (and
 * clears it when asked). Returns ATTN_OK once launched, ATTN_ERR_INVALID_ARG for a limit out of
 * range, ATTN_ERR_DEVICE off sm_103.
 */
int attn_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * attn_plan_launch_order — the block order the causal kernels use (host only, no device): items
 * of unequal length, one CTA resident per SM at a time, and the hardware giving the next block
 * to the first SM that frees up. The items, weights[i] + fixed each, are packed best-fit
 * decreasing into num_sms bins at the smallest capacity that packs (capacities tried upward
 * from the even split in unit steps; after 64 tries the step doubles, which bounds the host
 * time for very large weights), and returned in order of their start time in that packing
 * (ties: heavier first), so that list scheduling in this order follows the packing. attn_fwd, attn_fwd_lse and attn_bwd plan their causal grids this
 * way (weights = key or query tiles of each work item) when a call has at most 2048 items.
 *   weights : host array of n weights, each 0 .. 2^24
 *   n       : 1 .. 8192
 *   fixed   : per-item cost added to every weight, 0 .. 2^24
 *   num_sms : bins, 1 .. 1024, with n * num_sms <= 2^20 (each capacity tried costs n * num_sms
 *             steps; the bound keeps a call well under a second)
 *   order   : host array of n entries; receives the permutation (position -> item index)
 * Returns ATTN_OK, or ATTN_ERR_INVALID_ARG for a null pointer or a value out of range.
 */
int attn_plan_launch_order(const int32_t* weights, int64_t n, int32_t fixed, int32_t num_sms, uint16_t* order);

/*
 * attn_probe_fp32_fma — the fp32 roofline that the FFMA (float32) kernels are measured against,
 * taken on the device itself (the pages give no fp32 peak for it; their own kernels ran on
 * CUDA cores). Enqueues one kernel of one 1024-thread block per SM in which every thread runs 8
 * independent chains of `iters` fused multiply-adds, and writes that launch's flop count
 * (2 per multiply-add) to *flop on the host; the caller times the launch with CUDA events on
 * `stream` and divides. Not a step of the attention path.
 *   sink        : device buffer of sink_floats float32, at least SMs x 1024 (each thread writes
 *                 one value so the chains are not optimised away); ATTN_ERR_WORKSPACE if smaller
 *   iters       : 1 .. 2^24
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_DEVICE off sm_103, ATTN_ERR_LAUNCH.
 */
int attn_probe_fp32_fma(float* sink, int64_t sink_floats, int64_t iters, double* flop, void* stream);

/*
 * attn_probe_sfu_ex2 — the rate of the exponential the softmax uses (ex2.approx, base 2), which
 * co-bounds the tensor-core forward at d = 64 (one exponential per 256 flop of its products).
 * Same grid and arguments as attn_probe_fp32_fma: every thread runs 8 independent chains of
 * `iters` steps a = 2^(-a), and *ops receives the launch's count of exponentials. Not a step of
 * the attention path.
 */
int attn_probe_sfu_ex2(float* sink, int64_t sink_floats, int64_t iters, double* ops, void* stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* attn_status_string(int status);

/* ABI version of this header: (major << 16) | minor (1.1 added attn_fwd_lse, 1.2 attn_bwd,
 * 1.3 attn_fwd_kvcache, 1.4 head width 128 for the forward entry points, 1.5
 * attn_selftest_wait_timeout, 1.6 head width 128 for attn_bwd, 1.7 attn_plan_launch_order, 1.8
 * attn_probe_fp32_fma, 1.9 attn_probe_sfu_ex2). */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
