"""Pins for the backward-pass oracle: each test ties it to something other than its own code.

The oracle (oracle/attn_bwd_oracle.c) follows the steps of the "Flash attention in PyTorch,
then in Triton" page, section "Backwards, and training with it": dV = P^T dO, dP = dO V^T,
delta = rowsum(dO * O), dS = P (dP - delta), dQ = dS K scale, dK = dS^T Q scale. The pins:
central finite differences of a float64 forward written here (a different method: no
gradient formula), PyTorch's float64 autograd through its own attention, closed forms (one
key; equal scores), two exact sum identities (dK's rows sum to zero, dV's rows to dO's rows),
and planted mistakes in the C source that these must catch.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import seeded_inputs as si


def _fwd64(q, k, v, causal):
    """Plain float64 attention of one head, for finite differences only."""
    s = (q @ k.T) / np.sqrt(q.shape[1])
    if causal:
        s = np.where(np.tril(np.ones_like(s, dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


@pytest.mark.parametrize("causal", [0, 1])
def test_matches_central_finite_differences(causal):
    N, d = 5, 8
    q, k, v, do = si.qkv(201, 1, 1, N, d) + (si.qkv(202, 1, 1, N, d)[0],)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal)
    q64, k64, v64, do64 = (x[0, 0].astype(np.float64) for x in (q, k, v, do))
    h = 1e-5

    def loss(qq, kk, vv):
        return float(np.sum(_fwd64(qq, kk, vv, causal) * do64))

    for name, arr, grad in (("q", q64, dq), ("k", k64, dk), ("v", v64, dv)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q64, "k": k64, "v": v64}
            args[name] = plus
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = minus
            lm = loss(args["q"], args["k"], args["v"])
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad[0, 0], fd, rtol=1e-7, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("shape,qk_scale", [((2, 3, 33, 64), 1.0), ((1, 2, 70, 64), 8.0), ((1, 1, 9, 16), 1.0)])
def test_matches_torch_float64_autograd(causal, shape, qk_scale):
    torch = pytest.importorskip("torch")
    q, k, v = si.qkv(211, *shape, qk_scale=qk_scale)
    do = si.qkv(212, *shape)[0]
    got = oracle.attn_bwd(q, k, v, do, causal)
    tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=bool(causal))
    o.backward(torch.from_numpy(do).double())
    for g, t, name in zip(got, (tq, tk, tv), "qkv"):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("causal", [0, 1])
def test_single_key_gradients(causal):
    # One key: o = v exactly, so dV = dO and dQ = dK = 0 (the softmax of one score is 1).
    q, k, v = si.qkv(221, 2, 2, 1, 64)
    do = si.qkv(222, 2, 2, 1, 64)[0]
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal)
    assert np.array_equal(dv, do.astype(np.float64))
    assert np.all(np.abs(dq) <= 1e-15) and np.all(np.abs(dk) <= 1e-15)


def test_equal_scores_closed_form():
    # q = 0: every visible weight is 1/n_i, o_i = mean of visible v, and
    # dV_j = sum_{i sees j} dO_i / n_i;  dQ_i = scale * sum_j (dO_i.v_j - dO_i.o_i) k_j / n_i.
    N, d = 12, 16
    _, k, v = si.qkv(231, 1, 1, N, d)
    do = si.qkv(232, 1, 1, N, d)[0]
    q = np.zeros_like(k)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True)
    k64, v64, do64 = (x[0, 0].astype(np.float64) for x in (k, v, do))
    for i in range(N):
        n = i + 1
        o_i = v64[:n].mean(axis=0)
        want = sum((do64[i] @ v64[j] - do64[i] @ o_i) * k64[j] for j in range(n)) / n / np.sqrt(d)
        np.testing.assert_allclose(dq[0, 0, i], want, rtol=1e-12, atol=1e-13)
    for j in range(N):
        want = sum(do64[i] / (i + 1) for i in range(j, N))
        np.testing.assert_allclose(dv[0, 0, j], want, rtol=1e-12, atol=1e-13)


SRC = open(os.path.join(os.path.dirname(oracle.__file__), "attn_bwd_oracle.c")).read()
MUTANTS = {
    "dq_unscaled": ("dq[i * d + e] += ds * (double)k[j * d + e] * scale;", "dq[i * d + e] += ds * (double)k[j * d + e];"),
    "dk_from_k": ("dk[j * d + e] += ds * (double)q[i * d + e] * scale;", "dk[j * d + e] += ds * (double)k[i * d + e] * scale;"),
    "delta_sign": ("const double ds = p * (dp[j] - delta);", "const double ds = p * (dp[j] + delta);"),
    "delta_dropped": ("const double ds = p * (dp[j] - delta);", "const double ds = p * dp[j];"),
    "dv_not_transposed": ("dv[j * d + e] += p * (double)dout[i * d + e];", "dv[i * d + e] += p * (double)dout[j * d + e];"),
    "mask_off_by_one": ("const int64_t vis = causal ? i + 1 : N;", "const int64_t vis = causal ? (i + 2 < N ? i + 2 : N) : N;"),
}


def _mutant_bwd(tmp_path, name, q, k, v, do, causal):
    """dq, dk, dv from the oracle's C source with mutant `name` planted."""
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, name
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(SRC.replace(old, new))
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    i64, fp, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    lib.oracle_attn_bwd.argtypes = [fp, fp, fp, fp, i64, i64, i64, i64, ctypes.c_int, dp, dp, dp, ctypes.c_int]
    outs = [np.empty(q.shape) for _ in range(3)]
    assert lib.oracle_attn_bwd(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp), do.ctypes.data_as(fp),
                               *q.shape, int(causal), *(x.ctypes.data_as(dp) for x in outs), 2) == 0
    return outs


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistakes_are_caught(tmp_path, name):
    torch = pytest.importorskip("torch")
    shape = (1, 2, 17, 64)
    q, k, v = si.qkv(241, *shape)
    do = si.qkv(242, *shape)[0]
    outs = _mutant_bwd(tmp_path, name, q, k, v, do, 1)
    tq, tk, tv = (torch.from_numpy(x).double().requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    o.backward(torch.from_numpy(do).double())
    ok = all(np.allclose(g, t.grad.numpy(), rtol=1e-9, atol=1e-10) for g, t in zip(outs, (tq, tk, tv)))
    assert not ok, f"mutant {name} not caught"


def _sum_identities_hold(dk, dv, do):
    # Each row of dS = P (dP - delta) sums to zero (delta is the row's P-weighted dP), so the
    # rows of dK = scale dS^T Q sum to zero in every head; each row of P sums to one, so the
    # rows of dV = P^T dO sum to the rows of dO.
    dk_ok = np.abs(dk.sum(axis=2)).max() <= 1e-12 * np.abs(dk).sum(axis=2).max()
    dv_ok = np.abs(dv.sum(axis=2) - do.astype(np.float64).sum(axis=2)).max() <= 1e-12 * np.abs(do).sum(axis=2).max()
    return dk_ok, dv_ok


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("d", [64, 128])
def test_gradient_sum_identities(causal, d):
    shape = (2, 3, 37, d)
    q, k, v = si.qkv(251, *shape)
    do = si.qkv(252, *shape)[0]
    _, dk, dv = oracle.attn_bwd(q, k, v, do, causal)
    assert _sum_identities_hold(dk, dv, do) == (True, True)


@pytest.mark.parametrize("name,broken", [("delta_sign", 0), ("delta_dropped", 0), ("dv_not_transposed", 1)])
def test_sum_identities_catch_mutants(tmp_path, name, broken):
    # Without PyTorch: the identities alone reject a wrong or missing delta and an
    # untransposed P in dV.
    shape = (1, 2, 17, 64)
    q, k, v = si.qkv(243, *shape)
    do = si.qkv(244, *shape)[0]
    _, dk, dv = _mutant_bwd(tmp_path, name, q, k, v, do, 1)
    assert not _sum_identities_hold(dk, dv, do)[broken], name

