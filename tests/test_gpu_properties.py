"""GPU properties that hold exactly at any size: single-key identity, causality, run-to-run
determinism, guard bands around the output, the materialised ablation against the oracle
and against the flash path, and the C-ABI error statuses on a real device."""

import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_flashattention_gb300 as fa
import seeded_inputs as si
from attn_testlib import CONFIG_SEED, check, gpu_attn, page_gate_fraction, to_dev

pytestmark = pytest.mark.gpu
DTYPES = ["f32", "bf16", "f16"]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_v_bit_exactly(dtype, causal):
    q, k, v = si.qkv(3, 3, 5, 1, 64, dtype)
    got = gpu_attn(q, k, v, dtype, causal)
    assert np.array_equal(got, v.astype(np.float64))


@pytest.mark.parametrize("dtype", DTYPES)
def test_empty_problems_are_no_ops(dtype):
    z = torch.empty(1, 2, 0, 64, device="cuda", dtype={"f32": torch.float32, "bf16": torch.bfloat16,
                                                        "f16": torch.float16}[dtype])
    assert fa.attn_fwd(z, z, z, causal=True).shape == z.shape
    z2 = z.new_empty(0, 3, 16, 64)
    assert fa.attn_fwd(z2, z2, z2).shape == z2.shape


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("t", [0, 100, 127, 128, 300])
def test_causal_rows_ignore_later_keys_bit_exactly(dtype, t):
    N = 515
    q, k, v = si.qkv(17, 1, 2, N, 64, dtype)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:], v2[:, :, t + 1:] = si.qkv(18, 1, 2, N, 64, dtype)[1:][0][:, :, t + 1:], \
        si.qkv(18, 1, 2, N, 64, dtype)[2][:, :, t + 1:]
    a = gpu_attn(q, k, v, dtype, True)
    b = gpu_attn(q, k2, v2, dtype, True)
    assert np.array_equal(a[:, :, : t + 1], b[:, :, : t + 1])
    assert not np.array_equal(a[:, :, t + 1:], b[:, :, t + 1:])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("causal", [False, True])
def test_runs_are_bit_identical(dtype, causal):
    q, k, v = si.qkv(23, 2, 3, 700, 64, dtype)
    a = gpu_attn(q, k, v, dtype, causal)
    b = gpu_attn(q, k, v, dtype, causal)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_output_guard_band_and_full_coverage(dtype, N):
    B, H = 2, 3
    q, k, v = si.qkv(29, B, H, N, 64, dtype)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    n = B * H * N * 64
    slack = 4096
    buf = torch.full((n + 2 * slack,), float("nan"), device="cuda", dtype=qd.dtype)
    out = buf[slack: slack + n].view(B, H, N, 64)
    fa.attn_fwd(qd, kd, vd, causal=True, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:slack]).all() and torch.isnan(buf[slack + n:]).all()
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 256, 1000])
def test_materialized_path_matches_oracle_and_flash(dtype, causal, N):
    q, k, v = si.qkv(CONFIG_SEED[2] + N, 2, 3, N, 64, dtype)
    ref = oracle.attn_fwd(q, k, v, causal)
    mat = gpu_attn(q, k, v, dtype, causal, path="materialized")
    check(mat, ref, dtype, N, "materialized")
    flash = gpu_attn(q, k, v, dtype, causal)
    if dtype == "f32":
        # attention.cu's pair check: the two GPU paths against each other under the gate.
        assert page_gate_fraction(flash, mat, N) <= 1.0
    else:
        assert np.max(np.abs(flash - mat)) <= 4e-2


def test_materialized_small_workspace_runs_heads_in_groups():
    B, H, N = 2, 3, 300
    q, k, v = si.qkv(31, B, H, N, 64, "f32")
    qd, kd, vd = (to_dev(x, "f32") for x in (q, k, v))
    per = fa.attn_materialized_workspace_bytes(1, 1, N)
    ws = torch.empty(2 * per + 100, dtype=torch.uint8, device="cuda")  # two heads per group
    got = fa.attn_fwd_materialized(qd, kd, vd, causal=True, workspace=ws)
    torch.cuda.synchronize()
    check(got.double().cpu().numpy(), oracle.attn_fwd(q, k, v, True), "f32", N, "grouped")


def test_non_default_stream():
    q, k, v = si.qkv(37, 1, 4, 512, 64, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o = fa.attn_fwd(qd, kd, vd, causal=True)
    s.synchronize()
    check(o.double().cpu().numpy(), oracle.attn_fwd(q, k, v, True), "bf16", 512, "stream")


def test_error_statuses_on_device():
    lib = fa.raw()
    x = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    base = (x.data_ptr(), x.data_ptr(), x.data_ptr(), y.data_ptr())
    assert lib.attn_fwd(*base, 1, 1, 64, 64, 0, 1, None) == 0
    assert lib.attn_fwd(base[0] + 2, *base[1:], 1, 1, 60, 64, 0, 1, None) == 3
    assert lib.attn_fwd(*base[:3], base[0], 1, 1, 64, 64, 0, 1, None) == 4
    assert lib.attn_fwd(*base, 1, 1, 64, 96, 0, 1, None) == 2   # head width neither 64 nor 128
    assert lib.attn_fwd(*base, 1, 1, 32, 128, 0, 1, None) == 0  # d = 128 over the same bytes
    with pytest.raises(fa.AttnError):
        fa.attn_fwd(x, x, x, out=x)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0


def test_injected_launch_fault_is_reported(monkeypatch):
    x = torch.zeros(1, 1, 64, 64, dtype=torch.float16, device="cuda")
    monkeypatch.setenv("ATTN_FAULT", "launch")
    with pytest.raises(fa.AttnError) as ei:
        fa.attn_fwd(x, x, x)
    assert ei.value.status == 6
    monkeypatch.delenv("ATTN_FAULT")
    fa.attn_fwd(x, x, x)
    torch.cuda.synchronize()


def test_device_wait_timeout_is_reported_and_the_context_stays_usable():
    # A wait that nothing completes runs out after 2 ms; the status reports it once, clearing
    # works, and the next real call runs normally.
    assert fa.attn_device_status(clear=True) == 0
    fa.attn_selftest_wait_timeout(2_000_000)
    assert fa.attn_device_status(clear=False) == 7
    assert fa.attn_device_status(clear=True) == 7
    assert fa.attn_device_status(clear=True) == 0
    x = torch.randn(1, 2, 100, 64, device="cuda", dtype=torch.bfloat16)
    o = fa.attn_fwd(x, x, x, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    assert torch.isfinite(o.float()).all()


def test_calls_capture_into_a_cuda_graph_and_replay_bit_identically():
    # Every entry point is stream-ordered and allocation-free once its workspace exists, so a
    # step of forward, log-sum-exps, backward and key-value cache calls can be captured once and
    # replayed; the replay must reproduce the eager results bit for bit.
    torch.manual_seed(0)
    q, k, v, do = (torch.randn(2, 3, 300, 64, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    kc, vc = (torch.randn(2, 3, 5000, 64, device="cuda", dtype=torch.bfloat16) for _ in range(2))
    q1 = torch.randn(2, 3, 1, 64, device="cuda", dtype=torch.bfloat16)
    q8 = torch.randn(2, 3, 8, 64, device="cuda", dtype=torch.bfloat16)  # eight queries: tensor-core cache kernel
    ws = torch.empty(max(1, fa.attn_kvcache_workspace_bytes(2, 3, 1, 5000, 0, torch.bfloat16)), dtype=torch.uint8,
                     device="cuda")
    ws8 = torch.empty(max(1, fa.attn_kvcache_workspace_bytes(2, 3, 8, 5000, 0, torch.bfloat16)), dtype=torch.uint8,
                      device="cuda")
    o, lse = torch.empty_like(q), torch.empty(2, 3, 300, device="cuda")
    od, od8 = torch.empty_like(q1), torch.empty_like(q8)

    def step():
        fa.attn_fwd_lse(q, k, v, causal=True, out=o, lse=lse)
        grads = fa.attn_bwd(q, k, v, o, do, lse, causal=True)
        fa.attn_fwd_kvcache(q1, kc, vc, causal=True, workspace=ws, out=od)
        fa.attn_fwd_kvcache(q8, kc, vc, causal=True, workspace=ws8, out=od8)
        return grads

    eager = [x.clone() for x in (*step(), o, lse, od, od8)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm the per-function attribute caches outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        grads = step()
    for x in (o, lse, od, od8, *grads):
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    for a, b in zip(eager, (*grads, o, lse, od, od8)):
        assert torch.equal(a, b)


def test_throughput_probes_run_and_report_plausible_rates():
    # The roofline probes: FFMA chains and ex2.approx chains on every SM. Their counts follow
    # from the grid (SMs x 1024 threads x 8 chains x iters), and the measured rates sit between
    # a tenth of and twice the GB300's nominal figures (128 FMA lanes and 32 ex2 per SM per
    # clock at up to 2.07 GHz), which catches a probe that stops doing its work.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.empty(sms * 1024, dtype=torch.float32, device="cuda")
    iters = 4096
    for probe, per_item, nominal in ((fa.attn_probe_fp32_fma, 2.0, 128 * 2 * 2.07e9 * sms),
                                     (fa.attn_probe_sfu_ex2, 1.0, 32 * 2.07e9 * sms)):
        probe(sink, 64)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        count = probe(sink, iters)
        e1.record()
        torch.cuda.synchronize()
        assert count == per_item * sms * 1024 * 8 * iters
        rate = count / (e0.elapsed_time(e1) * 1e-3)
        assert 0.1 * nominal < rate < 2.0 * nominal, (probe.__name__, rate, nominal)
        assert bool(torch.isfinite(sink).all())
    with pytest.raises(fa.AttnError):
        fa.attn_probe_sfu_ex2(sink[:-1], 16)  # one float short of SMs x 1024
