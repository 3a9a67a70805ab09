"""Shared helpers of the GPU parity tests: device round-trips through the C-ABI binding and
the tolerance rules.

Tolerances (spec contract, with the attention.cu gate reported beside it):
* fp32: max |got - ref| <= 1e-5 * N * max |ref|  (the K-scaled rule with K = N);
  attention.cu's own gate |got - ref| <= atol + rtol |ref| with rtol = max(1e-5, 4 * 2^-23 *
  sqrt(N)), atol = rtol * max |ref| is computed too, and must also hold — except for q, k
  scaled x8 (logit std ~64), where fp32 rounding of the scores alone exceeds it (PyTorch's
  own fp32 attention scores 1.08 on the same inputs); there the Triton page's rule applies
  instead: the error is at most twice PyTorch's fp32 error against the same reference.
* bf16 / fp16: max |got - ref| <= 2e-2, against the double oracle on the same rounded inputs.
Non-finite output fails outright.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import online_softmax_flashattention_gb300 as fa

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CONFIG_SEED = {i: 0xA77E0000 + i for i in range(5)}


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Exact upload: x already holds values representable in dtype."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda")
    return t.to(TORCH_DT[dtype]).contiguous()


def gpu_attn(q, k, v, dtype: str, causal: bool, path: str = "flash") -> np.ndarray:
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    if path == "flash":
        o = fa.attn_fwd(qd, kd, vd, causal=causal)
    else:
        o = fa.attn_fwd_materialized(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    return o.float().cpu().numpy().astype(np.float64)


def fp32_bound(N: int, ref_max: float) -> float:
    return 1e-5 * N * ref_max


def page_gate_fraction(got: np.ndarray, ref: np.ndarray, N: int) -> float:
    rtol = max(1e-5, 4.0 * 2.0 ** -23 * math.sqrt(max(N, 1)))
    atol = rtol * float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (atol + rtol * np.abs(ref))))


def check(got: np.ndarray, ref: np.ndarray, dtype: str, N: int, what: str = "",
          page_gate: bool = True) -> dict:
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_err = float(err.max()) if err.size else 0.0
    ref_max = float(np.abs(ref).max()) if ref.size else 0.0
    rep = {"max_err": max_err, "ref_max": ref_max}
    if dtype == "f32":
        bound = fp32_bound(N, ref_max)
        rep["bound"] = bound
        rep["gate_fraction"] = page_gate_fraction(got, ref, N)
        assert max_err <= bound, f"{what}: fp32 max err {max_err:.3e} > {bound:.3e}"
        if page_gate:
            assert rep["gate_fraction"] <= 1.0, f"{what}: attention.cu gate fraction {rep['gate_fraction']:.3f}"
    else:
        rep["bound"] = 2e-2
        if max_err > 2e-2:
            idx = np.unravel_index(int(np.argmax(err)), err.shape)
            raise AssertionError(f"{what}: {dtype} max err {max_err:.4e} > 2e-2 at {idx}, ref {ref[idx]:.5f}, "
                                 f"got {got[idx]:.5f}")
    return rep
