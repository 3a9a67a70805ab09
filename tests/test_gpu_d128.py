"""GPU parity of the forward at head width d = 128 (attn_fwd, attn_fwd_lse) against the double
oracle on the same seeded inputs. The pages fix d = 64; d = 128 is the other common head width,
with the scale 1/sqrt(128). Tolerances are the d = 64 ones: bf16/fp16 2e-2 absolute; fp32
1e-5 * N * max|ref| and attention.cu's gate; lse 2e-5 * (1 + max|lse|) + 1e-4 (the score
error grows with sum_e |q_e k_e|, which the 1/sqrt(d) scale keeps at the d = 64 size for unit
inputs).
"""

import numpy as np
import pytest
import torch

import online_softmax_flashattention_gb300 as fa
import oracle
import seeded_inputs as si
from attn_testlib import check, to_dev

pytestmark = pytest.mark.gpu
D = 128


def _lse_bound(ref):
    return 2e-5 * (1.0 + float(np.max(np.abs(ref)))) + 1e-4


def _run(seed, B, H, N, dtype, causal, qk_scale=1.0):
    q, k, v = si.qkv(seed, B, H, N, D, dtype, qk_scale=qk_scale)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=causal)
    o2 = fa.attn_fwd(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    assert torch.equal(o, o2), "attn_fwd_lse changed the output"
    ref_o, ref_lse = oracle.attn_fwd_lse(q, k, v, causal)
    rep = check(o.float().cpu().numpy().astype(np.float64), ref_o, dtype, N,
                f"d128 {dtype} B{B}H{H}N{N} causal={causal}", page_gate=(qk_scale == 1.0))
    got = lse.cpu().numpy().astype(np.float64)
    assert float(np.max(np.abs(got - ref_lse))) <= _lse_bound(ref_lse)
    return rep


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 256, 300, 1000])
def test_d128_ragged_lengths(dtype, causal, N):
    _run(0xD1280000 + N, 2, 3, N, dtype, causal)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_d128_longer_heads(dtype, causal):
    # several key tiles per query tile and both query tiles of a CTA busy
    _run(0xD1281000, 1, 2, 2048, dtype, causal)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_d128_qk_scaled_x8(dtype):
    q, k, v = si.qkv(0xD1282000, 1, 2, 700, D, dtype, qk_scale=8.0)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o = fa.attn_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    ref = oracle.attn_fwd(q, k, v, True)
    got = o.float().cpu().numpy().astype(np.float64)
    rep = check(got, ref, dtype, 700, "d128 x8", page_gate=(dtype != "f32"))
    if dtype == "f32":
        # the Triton page's rule: at most twice PyTorch's own fp32 error against the same reference
        t = [torch.from_numpy(x) for x in (q, k, v)]
        theirs = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=True).double().numpy()
        assert rep["max_err"] <= 2.0 * float(np.abs(theirs - ref).max())


def test_d128_single_key_is_v_and_first_causal_row_is_v0():
    for dtype in ("bf16", "f16", "f32"):
        q, k, v = si.qkv(0xD1283000, 1, 2, 1, D, dtype)
        o = fa.attn_fwd(*(to_dev(x, dtype) for x in (q, k, v)), causal=False)
        torch.cuda.synchronize()
        assert np.array_equal(o.float().cpu().numpy(), v.astype(np.float32))
        q, k, v = si.qkv(0xD1283001, 1, 2, 200, D, dtype)
        o = fa.attn_fwd(*(to_dev(x, dtype) for x in (q, k, v)), causal=True)
        torch.cuda.synchronize()
        assert np.array_equal(o[:, :, 0].float().cpu().numpy(), v[:, :, 0].astype(np.float32))


def test_d128_full_size_sampled_rows():
    # B1 H12 N8192 d128 bf16 causal: 64 sampled rows per head (and rows 0, N-1) against the oracle.
    B, H, N = 1, 12, 8192
    q, k, v = si.qkv(0xD1284000, B, H, N, D, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    rows = np.concatenate([[0, N - 1], si.sample_rows(0xD1284001, N, 62)])
    flat = np.concatenate([h * N + rows for h in range(B * H)])
    ref_o, ref_l = oracle.attn_fwd_lse(q, k, v, True, rows=flat)
    got_o = o.reshape(-1, D).float().cpu().numpy().astype(np.float64)[flat]
    got_l = lse.reshape(-1).cpu().numpy().astype(np.float64)[flat]
    check(got_o, ref_o, "bf16", N, "d128 B1H12N8192 sampled")
    assert float(np.max(np.abs(got_l - ref_l))) <= _lse_bound(ref_l)


def test_d128_matches_torch_sdpa_within_the_page_gate():
    # The Triton page's test: error against float64 at most twice PyTorch's own in bf16.
    q, k, v = si.qkv(0xD1285000, 2, 3, 1000, D, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o = fa.attn_fwd(qd, kd, vd, causal=True)
    theirs = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True)
    torch.cuda.synchronize()
    ref = oracle.attn_fwd(q, k, v, True)
    ours = float(np.abs(o.float().cpu().numpy() - ref).max())
    torch_err = float(np.abs(theirs.float().cpu().numpy() - ref).max())
    assert ours <= 2.0 * torch_err, (ours, torch_err)


def test_d128_long_context_sampled_rows():
    # B1 H4 N32768 d128 bf16 causal: 128 sampled rows per head (and rows 0, N-1) against the
    # oracle; row offsets and key-tile counts well past the headline's.
    B, H, N = 1, 4, 32768
    q, k, v = si.qkv(0xD1286000, B, H, N, D, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    rows = np.concatenate([[0, N - 1], si.sample_rows(0xD1286001, N, 126)])
    flat = np.concatenate([h * N + rows for h in range(B * H)])
    ref_o, ref_l = oracle.attn_fwd_lse(q, k, v, True, rows=flat)
    got_o = o.reshape(-1, D).float().cpu().numpy().astype(np.float64)[flat]
    got_l = lse.reshape(-1).cpu().numpy().astype(np.float64)[flat]
    check(got_o, ref_o, "bf16", N, "d128 B1H4N32768 sampled")
    assert float(np.max(np.abs(got_l - ref_l))) <= _lse_bound(ref_l)
