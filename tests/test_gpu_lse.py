"""GPU parity of attn_fwd_lse: each row's base-2 log-sum-exp against the double oracle.

The forward keeps lse2_i = log2(sum_j exp(q_i . k_j / sqrt(d))) for the backward pass
("Flash attention in PyTorch, then in Triton", section "Backwards, and training with it").

Tolerance, from the arithmetic: the kernels form the scores in fp32 from the exact input
values (bf16/fp16/fp32 products accumulated over d = 64), so a score carries an absolute error
of a few fp32 ulps of sum_e |q_e k_e| / sqrt(d); the log-sum-exp of the row inherits at most
that error (it is 1-Lipschitz in each score, in log2 units scaled by log2 e), and the fp32
sum l plus log2 add ~1e-6 relative. So |got - ref| <= 2e-5 * (1 + max_i |lse_i|) + 1e-4,
which for the scaled x8 inputs (|lse| ~ 800) is ~0.016 and for unit inputs ~1e-4.
The output o of attn_fwd_lse must be bit-identical to attn_fwd's.
"""

import numpy as np
import pytest
import torch

import online_softmax_flashattention_gb300 as fa
import oracle
import seeded_inputs as si
from attn_testlib import check, to_dev

pytestmark = pytest.mark.gpu


def _lse_bound(ref):
    return 2e-5 * (1.0 + float(np.max(np.abs(ref)))) + 1e-4


def _run(seed, B, H, N, dtype, causal, qk_scale=1.0):
    q, k, v = si.qkv(seed, B, H, N, 64, dtype, qk_scale=qk_scale)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=causal)
    o_plain = fa.attn_fwd(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    assert torch.equal(o, o_plain), "attn_fwd_lse changed the output"
    ref_o, ref_lse = oracle.attn_fwd_lse(q, k, v, causal)
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_lse))
    err = float(np.max(np.abs(got_lse - ref_lse)))
    assert err <= _lse_bound(ref_lse), f"lse max err {err:.3e} > {_lse_bound(ref_lse):.3e}"
    # o itself is covered by the parity tests; here the contract bound is enough (for fp32 with
    # q, k scaled x8 the attention.cu gate is replaced by the PyTorch-relative rule there).
    check(o.float().cpu().numpy().astype(np.float64), ref_o, dtype, N, f"{dtype} N={N} o",
          page_gate=(qk_scale == 1.0))
    return err


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 300, 1000])
def test_lse_ragged_lengths(dtype, causal, N):
    _run(0xA77E0100 + N, 2, 3, N, dtype, causal)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_lse_qk_scaled_x8(dtype, causal):
    _run(0xA77E0200, 1, 2, 513, dtype, causal, qk_scale=8.0)


def test_lse_headline_shape_sampled_rows():
    B, H, N = 1, 12, 8192
    q, k, v = si.qkv(0xA77E0003, B, H, N, 64, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    _, lse = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    rng = np.random.default_rng(0xA77E0300)
    rows = np.concatenate([[0, N - 1], rng.choice(N, 62, replace=False)])
    flat = np.concatenate([bh * N + rows for bh in range(B * H)])
    _, ref = oracle.attn_fwd_lse(q, k, v, True, rows=flat)
    got = lse.reshape(-1).cpu().numpy().astype(np.float64)[flat]
    assert float(np.max(np.abs(got - ref))) <= _lse_bound(ref)


def test_lse_equal_scores_is_log2_of_count():
    N = 300
    q = torch.zeros(1, 1, N, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.randn_like(q)
    v = torch.randn_like(q)
    _, lse = fa.attn_fwd_lse(q, k, v, causal=True)
    torch.cuda.synchronize()
    want = np.log2(np.arange(1, N + 1, dtype=np.float64))
    assert float(np.max(np.abs(lse[0, 0].cpu().numpy() - want))) <= 1e-5
