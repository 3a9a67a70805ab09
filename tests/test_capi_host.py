"""C-ABI checks that need no GPU: the library loads, exports every function declared in
include/attn.h, and rejects bad arguments before touching a device."""

import ctypes
import os
import re
import subprocess

import pytest

import online_softmax_flashattention_gb300 as fa
from online_softmax_flashattention_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.raw()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("attn_fwd", "attn_fwd_lse", "attn_fwd_materialized", "attn_materialized_workspace_bytes",
                 "attn_device_status", "attn_status_string", "attn_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert fa.attn_abi_version() >> 16 == 1
    assert fa.attn_abi_version() & 0xFFFF >= 1  # 1.1: attn_fwd_lse
    for code in range(9):
        s = fa.attn_status_string(code)
        assert s and s != "unknown status"
    assert fa.attn_status_string(99) == "unknown status"


P = 0x10000  # a 16-byte aligned non-null address; never dereferenced by these calls


@pytest.mark.parametrize("args,want", [
    ((P, P, P, P * 9, -1, 1, 8, 64, 0, 1), 1),            # negative B
    ((P, P, P, P * 9, 1, 1, 8, 64, 2, 1), 1),             # causal not 0/1
    ((P, P, P, P * 9, 1, 1, 8, 32, 0, 1), 2),             # d != 64
    ((P, P, P, P * 9, 1, 1, 8, 64, 0, 7), 2),             # unknown dtype
    ((P, P, P, P * 9, 1, 1, (1 << 30) + 1, 64, 0, 1), 2),  # N beyond the limit
    ((None, P, P, P * 9, 1, 1, 8, 64, 0, 1), 1),          # null q with work to do
    ((P + 2, P, P, P * 9, 1, 1, 8, 64, 0, 1), 3),         # misaligned q
    ((P, P, P, P + 64, 1, 1, 8, 64, 0, 1), 4),            # o overlaps q
    ((None, None, None, None, 0, 3, 8, 64, 1, 1), 0),     # B = 0: no-op
    ((None, None, None, None, 2, 3, 0, 64, 1, 0), 0),     # N = 0: no-op
])
def test_argument_checks_before_any_device_work(lib, args, want):
    assert lib.attn_fwd(*args, None) == want


@pytest.mark.parametrize("lse,want", [
    (P * 20 + 2, 3),   # lse not 4-byte aligned
    (P + 16, 4),       # lse overlaps q
    (P * 9 + 64, 4),   # lse overlaps o
])
def test_lse_argument_checks(lib, lse, want):
    # q, k, v, o: 1 x 1 x 8 x 64 bf16 = 1 KiB each at P, 3P, 5P, 9P
    assert lib.attn_fwd_lse(P, P * 3, P * 5, P * 9, lse, 1, 1, 8, 64, 0, 1, None) == want


def test_head_width_128_is_taken_by_all_but_the_ablation(lib):
    # d = 128 passes the checks of the forward, backward and key-value cache entry points (and
    # then needs the device); the materialised ablation refuses it before touching one.
    if not __import__("torch").cuda.is_available():
        assert lib.attn_fwd(P, P * 3, P * 5, P * 9, 1, 1, 8, 128, 0, 1, None) == 5
        assert lib.attn_fwd_lse(P, P * 3, P * 5, P * 9, P * 20, 1, 1, 8, 128, 0, 1, None) == 5
        assert lib.attn_bwd(P, P * 3, P * 5, P * 7, P * 9, P * 11, P * 13, P * 15, P * 17, 1, 1, 8, 128, 0, 1,
                            None) == 5
    assert lib.attn_fwd(P, P * 3, P * 5, P * 9, 1, 1, 8, 96, 0, 1, None) == 2
    assert lib.attn_fwd(P, P * 3, P * 5, P * 9, 1, 1, 8, 256, 0, 1, None) == 2
    assert lib.attn_bwd(P, P * 3, P * 5, P * 7, P * 9, P * 11, P * 13, P * 15, P * 17, 1, 1, 8, 96, 0, 1, None) == 2
    assert lib.attn_fwd_materialized(P, P * 3, P * 5, P * 9, P * 40, 1 << 20, 1, 1, 8, 128, 0, 1, None) == 2


def test_lse_shares_the_forward_checks(lib):
    assert lib.attn_fwd_lse(P, P, P, P * 9, P * 20, 1, 1, 8, 32, 0, 1, None) == 2       # d != 64
    assert lib.attn_fwd_lse(None, None, None, None, None, 0, 1, 8, 64, 0, 1, None) == 0  # no work


def test_materialized_workspace_checks(lib):
    per = lib.attn_materialized_workspace_bytes(1, 1, 100)
    assert per == 2 * ((100 * 100 * 4 + 255) // 256 * 256) + (400 + 255) // 256 * 256
    assert lib.attn_materialized_workspace_bytes(2, 3, 100) == 6 * per
    assert lib.attn_materialized_workspace_bytes(-1, 3, 100) == 0
    ws = 0x4000000
    assert lib.attn_fwd_materialized(P, P, P, P * 9, None, per, 1, 1, 100, 64, 0, 1, None) == 8
    assert lib.attn_fwd_materialized(P, P, P, P * 9, ws, per - 1, 1, 1, 100, 64, 0, 1, None) == 8
    assert lib.attn_fwd_materialized(P, P, P, P * 9, ws + 16, per, 1, 1, 100, 64, 0, 1, None) == 3
    assert lib.attn_fwd_materialized(P, P, P, P * 9, P, per, 1, 1, 100, 64, 0, 1, None) == 4


def test_binding_has_no_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(fa.AttnLibraryMissing):
        fa.raw()


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="needs a machine without a GPU")
def test_valid_call_without_gpu_reports_device_error(lib):
    assert lib.attn_fwd(P, P * 3, P * 5, P * 9, 1, 1, 8, 64, 0, 1, None) == 5
    assert lib.attn_fwd_lse(P, P * 3, P * 5, P * 9, P * 20, 1, 1, 8, 64, 0, 1, None) == 5


# attn_fwd_kvcache(q, k, v, o, lse, ws, ws_bytes, B, H, Nq, Nk, d, causal, dtype, splits, stream)
# q, o: 1 x 2 x 4 x 64 bf16 = 1 KiB at P and 9P; k, v: 1 x 2 x 100 x 64 bf16 = 25.6 KiB at 3P, 5P.
@pytest.mark.parametrize("args,want", [
    ((P, P * 3, P * 5, P * 9, None, None, 0, -1, 2, 4, 100, 64, 1, 1, 1), 1),   # negative B
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 101, 100, 64, 1, 1, 1), 1),  # Nq > Nk
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 2, 1, 1), 1),    # causal not 0/1
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, -1), 1),   # negative split count
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 96, 1, 1, 1), 2),    # d neither 64 nor 128
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 5, 1), 2),    # unknown dtype
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 1025), 2),  # too many shares
    ((None, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 1), 1),  # null q
    ((P, P * 3 + 8, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 1), 3),  # misaligned k
    ((P, P * 3, P * 5, P * 3 + 512, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 1), 4),  # o overlaps k
    ((P, P * 3, P * 5, P * 9, P * 20 + 1, None, 0, 1, 2, 4, 100, 64, 1, 1, 1), 3),  # lse misaligned
    ((P, P * 3, P * 5, P * 9, P * 5 + 64, None, 0, 1, 2, 4, 100, 64, 1, 1, 1), 4),  # lse overlaps v
    ((P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 4), 8),    # 4 shares, no workspace
    ((P, P * 3, P * 5, P * 9, None, P * 40, 100, 1, 2, 4, 100, 64, 1, 1, 4), 8),  # workspace too small
    ((P, P * 3, P * 5, P * 9, None, P * 40 + 16, 1 << 20, 1, 2, 4, 100, 64, 1, 1, 4), 3),  # ws misaligned
    ((P, P * 3, P * 5, P * 9, None, P * 5, 1 << 20, 1, 2, 4, 100, 64, 1, 1, 4), 4),  # ws overlaps v
    ((None, None, None, None, None, None, 0, 1, 2, 0, 100, 64, 1, 1, 0), 0),    # Nq = 0: no-op
    ((None, None, None, None, None, None, 0, 0, 2, 4, 100, 64, 1, 1, 0), 0),    # B = 0: no-op
])
def test_kvcache_argument_checks(lib, args, want):
    assert lib.attn_fwd_kvcache(*args, None) == want


def test_kvcache_workspace_bytes(lib):
    r = 2 * 3 * 5 * 7  # B * H * Nq * splits
    want = (r * 64 * 4 + 255) // 256 * 256 + (r * 4 + 255) // 256 * 256
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 64, 7, 1) == want
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 64, 1, 1) == 0   # one share writes o directly
    assert lib.attn_kvcache_workspace_bytes(-1, 3, 5, 100, 64, 7, 1) == 0
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 4, 64, 7, 1) == 0     # Nq > Nk
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 64, 1025, 1) == 0
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 64, 7, 9) == 0   # unknown dtype
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 128, 7, 1) == (r * 128 * 4 + 255) // 256 * 256 + (r * 4 + 255) // 256 * 256
    assert lib.attn_kvcache_workspace_bytes(2, 3, 5, 100, 96, 7, 1) == 0   # head width


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="needs a machine without a GPU")
def test_kvcache_valid_call_without_gpu_reports_device_error(lib):
    ws = P * 64
    assert lib.attn_fwd_kvcache(P, P * 3, P * 5, P * 9, None, ws, 1 << 20, 1, 2, 4, 100, 64, 1, 1, 4, None) == 5
    assert lib.attn_fwd_kvcache(P, P * 3, P * 5, P * 9, None, None, 0, 1, 2, 4, 100, 64, 1, 1, 0, None) == 5
    assert lib.attn_kvcache_workspace_bytes(1, 2, 4, 100, 64, 0, 1) == 0  # balanced plan needs the device


def test_selftest_limit_is_checked_before_the_device(lib):
    assert lib.attn_selftest_wait_timeout(10, None) == 1           # below 1 us
    assert lib.attn_selftest_wait_timeout(3_000_000_000, None) == 1  # above 2 s
    if not __import__("torch").cuda.is_available():
        assert lib.attn_selftest_wait_timeout(1_000_000, None) == 5


def test_fma_probe_checks_before_the_device(lib):
    import ctypes

    flop = ctypes.c_double(0.0)
    fp = ctypes.byref(flop)
    assert lib.attn_probe_fp32_fma(None, 1 << 20, 16, fp, None) == 1      # no sink
    assert lib.attn_probe_fp32_fma(P, 1 << 20, 0, fp, None) == 1          # iters < 1
    assert lib.attn_probe_fp32_fma(P, 1 << 20, (1 << 24) + 1, fp, None) == 1
    assert lib.attn_probe_fp32_fma(P, 1 << 20, 16, None, None) == 1       # no flop out


def test_sfu_probe_checks_before_the_device(lib):
    import ctypes

    ops = ctypes.c_double(0.0)
    op = ctypes.byref(ops)
    assert lib.attn_probe_sfu_ex2(None, 1 << 20, 16, op, None) == 1      # no sink
    assert lib.attn_probe_sfu_ex2(P, 1 << 20, 0, op, None) == 1          # iters < 1
    assert lib.attn_probe_sfu_ex2(P, 1 << 20, (1 << 24) + 1, op, None) == 1
    assert lib.attn_probe_sfu_ex2(P, 1 << 20, 16, None, None) == 1       # no count out
