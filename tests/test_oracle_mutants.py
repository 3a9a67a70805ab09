"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is the oracle's C source with one plausible error edited in, compiled with gcc
into a temporary library on the CPU. The same checks the pins use (closed-form fixtures,
PyTorch's float64 attention, the single-key identity) must reject every mutant; the
unmodified source must pass them.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import seeded_inputs as si

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()

MUTANTS = {
    "scale_dropped": ("s[j] = dot * scale;", "s[j] = dot;"),
    "scale_one_over_d": ("const double scale = 1.0 / sqrt((double)d);\n    const int64_t visible",
                         "const double scale = 1.0 / (double)d;\n    const int64_t visible"),
    "diagonal_masked": ("const int64_t visible = causal ? i + 1 : N;\n    double best = -HUGE_VAL;\n    for (int64_t j = 0; j < visible; ++j) {\n        double dot",
                        "const int64_t visible = causal ? (i > 0 ? i : 1) : N;\n    double best = -HUGE_VAL;\n    for (int64_t j = 0; j < visible; ++j) {\n        double dot"),
    "one_key_too_many": ("const int64_t visible = causal ? i + 1 : N;\n    double best = -HUGE_VAL;\n    for (int64_t j = 0; j < visible; ++j) {\n        double dot",
                         "const int64_t visible = causal ? (i + 2 < N ? i + 2 : N) : N;\n    double best = -HUGE_VAL;\n    for (int64_t j = 0; j < visible; ++j) {\n        double dot"),
    "scores_transposed": ("dot += (double)qh[i * d + e] * (double)kh[j * d + e];",
                          "dot += (double)qh[j * d + e] * (double)kh[i * d + e];"),
    "max_sign_flipped": ("s[j] = exp(s[j] - best);", "s[j] = exp(best - s[j]);"),
    "not_normalised": ("o_row[e] = acc[e] / total;", "o_row[e] = acc[e];"),
    "value_of_query_row": ("acc[e] += w * (double)vh[j * d + e];", "acc[e] += w * (double)vh[i * d + e];"),
}


def _build(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    i64, fp = ctypes.c_int64, ctypes.POINTER(ctypes.c_float)
    lib.oracle_attn_fwd.argtypes = [fp, fp, fp, i64, i64, i64, i64, ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_int64), i64,
                                    ctypes.POINTER(ctypes.c_double), ctypes.c_int]
    return lib


def _run(lib, q, k, v, causal):
    B, H, N, d = q.shape
    out = np.empty((B, H, N, d))
    fp = ctypes.POINTER(ctypes.c_float)
    st = lib.oracle_attn_fwd(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp),
                             B, H, N, d, causal, None, 0,
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), 2)
    assert st == 0
    return out


def _pins_pass(lib):
    torch = pytest.importorskip("torch")
    for causal in (0, 1):
        for shape, scale in (((1, 2, 1, 64), 1.0), ((2, 1, 40, 64), 1.0), ((1, 1, 33, 64), 8.0)):
            q, k, v = si.qkv(5, *shape, qk_scale=scale)
            got = _run(lib, q, k, v, causal)
            if shape[2] == 1 and not np.array_equal(got, v.astype(np.float64)):
                return False
            t = [torch.from_numpy(x).double() for x in (q, k, v)]
            want = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=bool(causal)).numpy()
            if not np.allclose(got, want, rtol=1e-12, atol=1e-12):
                return False
    return True


def test_unmodified_source_passes(tmp_path):
    assert _pins_pass(_build(tmp_path, "orig", SRC))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    before, after = MUTANTS[name]
    assert SRC.count(before) >= 1, f"mutation site for {name} not found"
    lib = _build(tmp_path, name, SRC.replace(before, after, 1))
    with np.errstate(all="ignore"):
        assert not _pins_pass(lib)
