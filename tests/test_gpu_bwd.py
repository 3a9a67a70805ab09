"""GPU parity of attn_bwd against the double backward oracle.

Gate (the "Flash attention in PyTorch, then in Triton" page's test, section "Backwards, and
training with it"): for each of dq, dk, dv, our max error against the float64 answer is at
most twice that of PyTorch's own attention in the test's precision on the same inputs
(PyTorch's backward, through autograd, on the GPU). An absolute sanity bound is asserted
too, derived from the arithmetic: our kernels compute in fp32 and round once to the output
type, so |err| <= 2 * ulp_out(max |ref|) + 1e-3 * max |ref| for bf16/fp16 outputs (their o
and lse inputs carry the forward's own rounding), and <= 1e-4 * max |ref| for fp32.
"""

import numpy as np
import pytest
import torch

import online_softmax_flashattention_gb300 as fa
import oracle
import seeded_inputs as si
from attn_testlib import to_dev

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
ULP = {"f32": 2.0 ** -23, "bf16": 2.0 ** -7, "f16": 2.0 ** -10}


def _torch_grads(q, k, v, do, dtype, causal):
    tq, tk, tv = (to_dev(x, dtype).requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    o.backward(to_dev(do, dtype))
    return [t.grad.float().cpu().numpy().astype(np.float64) for t in (tq, tk, tv)]


def _case(seed, B, H, N, dtype, causal, qk_scale=1.0, d=64):
    q, k, v = si.qkv(seed, B, H, N, d, dtype, qk_scale=qk_scale)
    do = si.qkv(seed + 1, B, H, N, d, dtype)[0]
    qd, kd, vd, dod = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    ours = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    ref = oracle.attn_bwd(q, k, v, do, causal)
    theirs = _torch_grads(q, k, v, do, dtype, causal)
    for name, got, want, tg in zip(("dq", "dk", "dv"), ours, ref, theirs):
        assert np.all(np.isfinite(got)), name
        err = float(np.max(np.abs(got - want)))
        terr = float(np.max(np.abs(tg - want)))
        mx = float(np.max(np.abs(want)))
        bound = 1e-4 * mx if dtype == "f32" else 2 * ULP[dtype] * mx + 1e-3 * mx
        assert err <= max(bound, 2.0 * terr), f"{name}: err {err:.3e}, PyTorch {terr:.3e}, bound {bound:.3e}, max {mx:.3e}"
        assert err <= 2.0 * terr or err <= bound, name


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 200, 513])
def test_bwd_ragged_lengths(dtype, causal, N):
    _case(0xA77E0400 + N, 2, 3, N, dtype, causal)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_qk_scaled_x8(dtype, causal):
    _case(0xA77E0500, 1, 2, 300, dtype, causal, qk_scale=8.0)


def test_bwd_single_key_closed_form():
    # One key: P = 1, so dv = dout (to bf16 rounding, which absorbs P's last-bit error) and
    # dS = P (dP - delta) vanishes up to the summation order of the two 64-term dot products.
    q, k, v = (torch.randn(2, 2, 1, 64, device="cuda", dtype=torch.bfloat16) for _ in range(3))
    do = torch.randn_like(q)
    o, lse = fa.attn_fwd_lse(q, k, v, causal=True)
    dq, dk, dv = fa.attn_bwd(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dv, do)
    assert float(dq.abs().max()) <= 1e-3 and float(dk.abs().max()) <= 1e-3


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 65, 128, 129, 300, 640])
def test_bwd_head_width_128(dtype, causal, N):
    # d = 128: the tensor-core dK/dV kernel writes P^T and dS^T over S^T and dP^T and reads O's
    # rows from global memory; several key and query blocks exercise the two-stage ring.
    _case(0xA77E0600 + N, 2, 3, N, dtype, causal, d=128)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bwd_head_width_128_qk_scaled_x8(dtype):
    _case(0xA77E0700, 1, 2, 300, dtype, True, qk_scale=8.0, d=128)


def test_bwd_full_size_sum_identities():
    # The bf16 causal B1 H12 N8192 d64 backward as the bench times it (a planned launch order),
    # checked through properties that hold at any size. Each row of dS = P (dP - delta) sums to
    # zero and each row of P to one, so in exact arithmetic dK's rows sum to zero in every head
    # and dV's rows sum to dO's rows. What the kernels round breaks this only slightly: delta
    # comes from the bf16 output o, P and dS are rounded to bf16 before their products, and
    # dk, dv are rounded once. Each of these is unit roundoff (2^-9) times terms of random sign,
    # about 1e-4 of sum_j |dk_j| (or |dv_j|) at this size; the bound is 2e-3 of that sum, per
    # head and column.
    B, H, N, d = 1, 12, 8192, 64
    q, k, v = si.qkv(0xA77E0600, B, H, N, d, "bf16")
    do = si.qkv(0xA77E0601, B, H, N, d, "bf16")[0]
    qd, kd, vd, dod = (to_dev(x, "bf16") for x in (q, k, v, do))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    dq, dk, dv = fa.attn_bwd(qd, kd, vd, o, dod, lse, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    dk64, dv64, do64 = dk.double(), dv.double(), dod.double()
    dk_dev = dk64.sum(dim=2).abs()
    dk_bound = 2e-3 * dk64.abs().sum(dim=2)
    assert bool((dk_dev <= dk_bound).all()), f"max |sum dk| {float(dk_dev.max()):.3e}, bound {float(dk_bound.min()):.3e}"
    dv_dev = (dv64.sum(dim=2) - do64.sum(dim=2)).abs()
    dv_bound = 2e-3 * dv64.abs().sum(dim=2)
    assert bool((dv_dev <= dv_bound).all()), f"max |sum dv - sum do| {float(dv_dev.max()):.3e}, bound {float(dv_bound.min()):.3e}"
    print(f"max |sum dk| {float(dk_dev.max()):.3e} (sum |dk| >= {float(dk64.abs().sum(dim=2).min()):.1f}); "
          f"max |sum dv - sum do| {float(dv_dev.max()):.3e} (sum |dv| >= {float(dv64.abs().sum(dim=2).min()):.1f})")
