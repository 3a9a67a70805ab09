"""Pins for the oracle's log-sum-exp, the value the forward pass keeps for the backward pass.

The "Flash attention in PyTorch, then in Triton" page (section "Backwards, and training with
it") defines it as the log of the sum the softmax divides by, kept in base 2 as the
running maximum plus the base-2 log of the running total: lse2_i = log2(sum_{j visible} exp(q_i . k_j / sqrt(d))). The pins:
closed forms (one key, equal scores, two keys), 40-digit decimal brute force, PyTorch's
float64 logsumexp, and its relation to the softmax weights; planted mistakes in the C source
(natural log, the maximum dropped, the wrong base) must fail them.
"""

import ctypes
import math
import os
import subprocess
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import seeded_inputs as si


@pytest.mark.parametrize("causal", [0, 1])
def test_single_key_lse_is_the_score_in_base_two(causal):
    q, k, v = si.qkv(12, 2, 3, 1, 64)
    _, lse = oracle.attn_fwd_lse(q, k, v, causal)
    getcontext().prec = 40
    for b in range(2):
        for h in range(3):
            s = sum(Decimal(float(q[b, h, 0, e])) * Decimal(float(k[b, h, 0, e])) for e in range(64)) / 8
            want = float(s / Decimal(2).ln())
            assert abs(lse[b, h, 0] - want) <= 1e-14 * max(1.0, abs(want))


@pytest.mark.parametrize("causal", [0, 1])
def test_equal_scores_give_log2_of_the_visible_count(causal):
    N, d = 37, 64
    _, k, v = si.qkv(5, 1, 1, N, d)
    q = np.zeros_like(v)
    _, lse = oracle.attn_fwd_lse(q, k, v, causal)
    for i in range(N):
        count = i + 1 if causal else N
        assert abs(lse[0, 0, i] - math.log2(count)) <= 1e-14


def test_two_keys_closed_form():
    # Scores s0, s1 set through one nonzero dimension: lse2 = log2(e^s0 + e^s1).
    N, d = 2, 64
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros_like(q)
    v = np.zeros_like(q)
    q[0, 0, :, 0] = [1.5, -2.0]
    k[0, 0, :, 0] = [4.0, -8.0]
    _, lse = oracle.attn_fwd_lse(q, k, v, False)
    for i in range(2):
        s0, s1 = q[0, 0, i, 0] * k[0, 0, 0, 0] / 8.0, q[0, 0, i, 0] * k[0, 0, 1, 0] / 8.0
        want = math.log2(math.exp(s0) + math.exp(s1))
        assert abs(lse[0, 0, i] - want) <= 1e-15 * max(1.0, abs(want))


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("N,d", [(1, 8), (3, 4), (6, 16)])
def test_lse_matches_decimal_brute_force(causal, N, d):
    q, k, v = si.qkv(71 + N, 1, 1, N, d, qk_scale=4.0)
    _, lse = oracle.attn_fwd_lse(q, k, v, causal)
    getcontext().prec = 40
    scale = Decimal(1) / Decimal(d).sqrt()
    for i in range(N):
        vis = range(i + 1) if causal else range(N)
        tot = sum((sum(Decimal(float(q[0, 0, i, e])) * Decimal(float(k[0, 0, j, e])) for e in range(d)) * scale).exp()
                  for j in vis)
        want = float(tot.ln() / Decimal(2).ln())
        assert abs(lse[0, 0, i] - want) <= 1e-13 * max(1.0, abs(want))


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("qk_scale", [1.0, 8.0])
def test_lse_matches_torch_float64_logsumexp(causal, qk_scale):
    torch = pytest.importorskip("torch")
    q, k, v = si.qkv(81, 2, 3, 100, 64, qk_scale=qk_scale)
    o, lse = oracle.attn_fwd_lse(q, k, v, causal)
    s = torch.from_numpy(q).double() @ torch.from_numpy(k).double().transpose(-1, -2) / 8.0
    if causal:
        s = s.masked_fill(torch.ones(100, 100, dtype=torch.bool).triu(1), float("-inf"))
    want = (torch.logsumexp(s, dim=-1) / math.log(2.0)).numpy()
    np.testing.assert_allclose(lse, want, rtol=1e-13, atol=1e-13)
    # o is unchanged by asking for the log-sum-exps
    assert np.array_equal(o, oracle.attn_fwd(q, k, v, causal))


def test_weights_are_exp_of_score_minus_lse():
    # P_ij = exp(s_ij) / 2^lse2_i: the identity the backward pass uses to rebuild P.
    N, d = 40, 64
    q, k, v = si.qkv(91, 1, 1, N, d, qk_scale=2.0)
    _, lse = oracle.attn_fwd_lse(q, k, v, True)
    s = (q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T) / 8.0
    for i in [0, 7, 39]:
        w = oracle.attn_weights(q[0, 0], k[0, 0], True, i)
        rebuilt = np.exp(s[i, : i + 1] - lse[0, 0, i] * math.log(2.0))
        np.testing.assert_allclose(w[: i + 1], rebuilt, rtol=1e-12, atol=0)


SRC = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
LSE_LINE = "if (lse_row) *lse_row = (best + log(total)) / log(2.0);"
MUTANTS = {
    "natural_log": "if (lse_row) *lse_row = best + log(total);",
    "max_dropped": "if (lse_row) *lse_row = log(total) / log(2.0);",
    "log2_of_max_only": "if (lse_row) *lse_row = best / log(2.0);",
    "log10": "if (lse_row) *lse_row = (best + log(total)) / log(10.0);",
}


def _lse_with(tmp_path, name, src, q, k, v, causal):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    i64, fp, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    lib.oracle_attn_fwd_lse.argtypes = [fp, fp, fp, i64, i64, i64, i64, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int64), i64, dp, dp, ctypes.c_int]
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    assert lib.oracle_attn_fwd_lse(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp), B, H, N, d,
                                   causal, None, 0, o.ctypes.data_as(dp), lse.ctypes.data_as(dp), 2) == 0
    return lse


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_lse_mistakes_are_caught(tmp_path, name):
    assert SRC.count(LSE_LINE) == 1
    q, k, v = si.qkv(101, 1, 2, 33, 64, qk_scale=2.0)
    torch = pytest.importorskip("torch")
    s = torch.from_numpy(q).double() @ torch.from_numpy(k).double().transpose(-1, -2) / 8.0
    s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
    want = (torch.logsumexp(s, dim=-1) / math.log(2.0)).numpy()
    good = _lse_with(tmp_path, "good", SRC, q, k, v, 1)
    np.testing.assert_allclose(good, want, rtol=1e-13, atol=1e-13)
    bad = _lse_with(tmp_path, name, SRC.replace(LSE_LINE, MUTANTS[name]), q, k, v, 1)
    assert not np.allclose(bad, want, rtol=1e-6, atol=1e-6)
