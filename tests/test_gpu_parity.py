"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU oracle on the
same seeded inputs, element by element; at full size on sampled rows.

Configurations (shapes of the workloads the attention pages measure):
  1. B1 H1 N256 fp32 non-causal
  2. B1 H1 N{1024, 4096} fp32, causal and non-causal, plus q, k scaled x8
  3. B2 H3 N{1, 100, 256, 1000} fp32 causal (ragged N)
  4. B1 H12 N8192 bf16 causal (the throughput case; sampled rows)
  5. B1 H12 N{32768, 131072} bf16 causal (long context; 512 sampled rows per head)
"""

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from attn_testlib import CONFIG_SEED, check, gpu_attn

pytestmark = pytest.mark.gpu


def _full(seed, B, H, N, dtype, causal, qk_scale=1.0, path="flash"):
    q, k, v = si.qkv(seed, B, H, N, 64, dtype, qk_scale=qk_scale)
    ref = oracle.attn_fwd(q, k, v, causal)
    got = gpu_attn(q, k, v, dtype, causal, path)
    page_gate = qk_scale == 1.0 or dtype != "f32"
    rep = check(got, ref, dtype, N, f"{path} {dtype} B{B}H{H}N{N} causal={causal}", page_gate=page_gate)
    if not page_gate:
        # "A kernel in Triton": at most twice the error of PyTorch's attention in that precision.
        t = [torch.from_numpy(x) for x in (q, k, v)]
        theirs = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal).double().numpy()
        assert rep["max_err"] <= 2.0 * float(np.abs(theirs - ref).max())
    return rep


def test_config1_single_head_noncausal_fp32():
    _full(CONFIG_SEED[0], 1, 1, 256, "f32", False)


@pytest.mark.parametrize("N", [1024, 4096])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("qk_scale", [1.0, 8.0])
def test_config2_single_head_fp32(N, causal, qk_scale):
    _full(CONFIG_SEED[1], 1, 1, N, "f32", causal, qk_scale)


@pytest.mark.parametrize("N", [1, 100, 256, 1000])
def test_config3_multihead_ragged_causal_fp32(N):
    _full(CONFIG_SEED[2], 2, 3, N, "f32", True)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 77, 127, 128, 129, 255, 256, 257, 300, 383, 384, 385, 1000, 1024])
def test_tensor_core_path_ragged_lengths(dtype, causal, N):
    _full(CONFIG_SEED[3] + N, 2, 3, N, dtype, causal)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_tensor_core_path_qk_scaled_x8(dtype, causal):
    # Logit std ~64: the running max moves on many tiles and the softmax is nearly one-hot.
    _full(CONFIG_SEED[1] + 7, 1, 2, 2048, dtype, causal, qk_scale=8.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [256, 1000, 4096])
@pytest.mark.parametrize("causal", [False, True])
def test_spike_late_pattern(dtype, N, causal):
    # attention.cu's deterministic inputs: key N-3 tripled so the max moves on the last tile.
    q, k, v = (si.round_to(x, dtype)[None, None] for x in si.spike_late(N, 64))
    ref = oracle.attn_fwd(q, k, v, causal)
    got = gpu_attn(q, k, v, dtype, causal)
    check(got, ref, dtype, N, f"spike-late {dtype} N{N}")


def _sampled(seed, B, H, N, dtype, causal, per_head):
    q, k, v = si.qkv(seed, B, H, N, 64, dtype)
    got = gpu_attn(q, k, v, dtype, causal).reshape(B * H * N, 64)
    rows = si.sample_rows(seed, N, per_head)
    flat = np.concatenate([bh * N + rows for bh in range(B * H)])
    ref = oracle.attn_fwd(q, k, v, causal, rows=flat)
    return check(got[flat], ref, dtype, N, f"{dtype} B{B}H{H}N{N} sampled")


def test_config4_headline_bf16_causal_sampled():
    _sampled(CONFIG_SEED[3], 1, 12, 8192, "bf16", True, 256)


@pytest.mark.parametrize("N", [32768, 131072])
def test_config5_long_context_bf16_causal_sampled(N):
    _sampled(CONFIG_SEED[4], 1, 12, N, "bf16", True, 512)
