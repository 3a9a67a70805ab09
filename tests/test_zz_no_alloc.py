"""The no-allocation materialised entry point, called through the C ABI.

attn_fwd_materialized_noalloc serves callers that cannot allocate device memory (or hand
over a workspace): its scratch is a fixed array compiled into the library. This checks it
against the existing workspace entry point, attn_fwd_materialized, on two calls in a row —
the second call finds the first call's data still in the shared array and must not depend
on it — and that sizes beyond the array are refused. The file is named to run last, so a
run that stops at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import online_softmax_flashattention_gb300 as fa
import seeded_inputs as si
from attn_testlib import TORCH_DT, fp32_bound, to_dev

pytestmark = pytest.mark.gpu


def _noalloc_c(qd, kd, vd, od, causal):
    lib = fa.raw()
    fn = lib.attn_fwd_materialized_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp]
    fn.restype = ci
    B, H, N, d = qd.shape
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[qd.dtype]
    return fn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), B, H, N, d, int(causal), dt,
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare(dtype, B, H, N, causal, seed):
    q, k, v = si.qkv(seed, B, H, N, 64, dtype)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    got = torch.full_like(qd, float("nan"))
    assert _noalloc_c(qd, kd, vd, got, causal) == 0
    want = fa.attn_fwd_materialized(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    g, w = got.double().cpu().numpy(), want.double().cpu().numpy()
    assert np.all(np.isfinite(g))
    err = float(np.abs(g - w).max())
    tol = fp32_bound(N, float(np.abs(w).max())) if dtype == "f32" else 2e-2
    assert err <= tol, (dtype, N, err, tol)


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # First call fills the shared scratch; the second, with other sizes and another type,
    # runs on top of the first call's leftovers.
    _compare("bf16", 2, 3, 1000, True, 0x5EED01)
    _compare("f32", 1, 4, 2896, False, 0x5EED02)


def test_binding_wrapper_and_size_limit():
    q, k, v = si.qkv(0x5EED03, 1, 2, 300, 64, "f16")
    qd, kd, vd = (to_dev(x, "f16") for x in (q, k, v))
    a = fa.attn_fwd_materialized_noalloc(qd, kd, vd, causal=True)
    b = fa.attn_fwd_materialized(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert float((a.double() - b.double()).abs().max()) <= 2e-2
    big = torch.zeros(1, 1, fa.ATTN_NOALLOC_MAX_N + 1, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(big)
    assert _noalloc_c(big, big, big, out, False) == 2  # ATTN_ERR_UNSUPPORTED, nothing launched
