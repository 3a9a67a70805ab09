"""Pins for the CPU oracle: each test ties it to something other than its own code.

The oracle computes exact attention forward (scores q.k / sqrt(d), causal mask keeping the
diagonal, row softmax, weighted values) as stated on the "Flash attention in PyTorch, then
in Triton" page ("Attention's table of scores", "Attention by hand") and in attention.cu's
double-precision CPU reference. The pins below are closed forms, brute force in 40-digit
decimal arithmetic, an independent library routine (PyTorch's float64 CPU
scaled_dot_product_attention), and invariants of the definition. Each plausible mistake —
a dropped or wrong scale, a transposed q.k^T, a mask on the wrong side of or excluding the
diagonal, a missing normalisation, the max subtracted with the wrong sign — fails at
least one of them.
"""

import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def _parse_golden(path):
    cases, cur = [], None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        parts = line.split()
        if parts[0] == "case":
            cur = {"name": parts[1], "N": int(parts[2].split("=")[1]), "in": [], "out": []}
            cases.append(cur)
        elif parts[0] == "in":
            cur["in"].append((parts[1], int(parts[2]), int(parts[3]), float(parts[4])))
        elif parts[0] == "out":
            cur["out"].append((int(parts[1]), int(parts[2]), int(parts[3]), float(parts[4])))
    return cases


@pytest.mark.parametrize("case", _parse_golden(GOLDEN), ids=lambda c: c["name"])
@pytest.mark.parametrize("causal", [0, 1])
def test_closed_form_fixtures(case, causal):
    N, d = case["N"], 64
    t = {n: np.zeros((1, 1, N, d), np.float32) for n in "qkv"}
    for name, row, dim, val in case["in"]:
        t[name][0, 0, row, dim] = val
    got = oracle.attn_fwd(t["q"], t["k"], t["v"], causal)[0, 0]
    want = np.zeros((N, d))
    for c, row, dim, val in case["out"]:
        if c == causal:
            want[row, dim] = val
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-15)


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_single_key_returns_v_exactly(causal, dtype):
    q, k, v = si.qkv(11, 2, 3, 1, 64, dtype)
    o = oracle.attn_fwd(q, k, v, causal)
    assert np.array_equal(o, v.astype(np.float64))


@pytest.mark.parametrize("causal", [0, 1])
def test_equal_scores_give_mean_of_visible_values(causal):
    N, d = 37, 64
    _, _, v = si.qkv(5, 1, 1, N, d)
    q = np.zeros_like(v)
    k = si.qkv(6, 1, 1, N, d)[1]
    o = oracle.attn_fwd(q, k, v, causal)[0, 0]
    for i in range(N):
        vis = range(i + 1) if causal else range(N)
        for e in range(d):
            mean = math.fsum(float(v[0, 0, j, e]) for j in vis) / len(vis)
            assert abs(o[i, e] - mean) <= 1e-15 * max(1.0, abs(mean)) + 1e-15


def test_causal_row_depends_only_on_keys_up_to_it():
    N, d, t = 50, 64, 20
    q, k, v = si.qkv(21, 1, 2, N, d)
    base = oracle.attn_fwd(q, k, v, True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:] = si.qkv(22, 1, 2, N, d)[1][:, :, t + 1:]
    v2[:, :, t + 1:] = si.qkv(22, 1, 2, N, d)[2][:, :, t + 1:]
    pert = oracle.attn_fwd(q, k2, v2, True)
    assert np.array_equal(base[:, :, : t + 1], pert[:, :, : t + 1])
    assert not np.array_equal(base[:, :, t + 1:], pert[:, :, t + 1:])
    # The diagonal is visible: changing only v_t changes row t.
    v3 = v.copy()
    v3[:, :, t] += 1.0
    assert not np.array_equal(oracle.attn_fwd(q, k, v3, True)[:, :, t], base[:, :, t])


@pytest.mark.parametrize("causal", [0, 1])
def test_weights_are_a_distribution_over_visible_keys(causal):
    N, d = 64, 64
    q, k, _ = si.qkv(31, 1, 1, N, d, qk_scale=8.0)
    for i in [0, 1, 17, 63]:
        w = oracle.attn_weights(q[0, 0], k[0, 0], causal, i)
        vis = i + 1 if causal else N
        assert abs(math.fsum(w) - 1.0) <= 1e-15 * N
        assert np.all(w[:vis] > 0) or i == 0 or not causal
        assert np.all(w[vis:] == 0.0)
        assert np.all(w >= 0.0)


def _decimal_attention(q, k, v, causal):
    """Brute force: the whole masked score matrix, softmax by exp / sum, in 40 digits."""
    getcontext().prec = 40
    N, d = q.shape
    scale = Decimal(1) / Decimal(d).sqrt()
    out = np.zeros((N, d))
    for i in range(N):
        s = []
        for j in range(N):
            if causal and j > i:
                s.append(None)
                continue
            s.append(sum(Decimal(float(q[i, e])) * Decimal(float(k[j, e])) for e in range(d)) * scale)
        ex = [x.exp() if x is not None else Decimal(0) for x in s]
        tot = sum(ex)
        for e in range(d):
            out[i, e] = float(sum(ex[j] * Decimal(float(v[j, e])) for j in range(N)) / tot)
    return out


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("N,d", [(1, 8), (2, 4), (5, 16), (6, 64), (3, 128)])
def test_matches_decimal_brute_force(causal, N, d):
    q, k, v = si.qkv(41 + N, 1, 1, N, d)
    got = oracle.attn_fwd(q, k, v, causal)[0, 0]
    want = _decimal_attention(q[0, 0], k[0, 0], v[0, 0], causal)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("shape", [(2, 3, 1, 64), (2, 3, 100, 64), (1, 2, 257, 64), (1, 1, 33, 16),
                                   (1, 2, 130, 128)])
@pytest.mark.parametrize("qk_scale", [1.0, 8.0])
def test_matches_torch_float64_sdpa(causal, shape, qk_scale):
    torch = pytest.importorskip("torch")
    q, k, v = si.qkv(51, *shape, qk_scale=qk_scale)
    got = oracle.attn_fwd(q, k, v, causal)
    t = [torch.from_numpy(x).double() for x in (q, k, v)]
    want = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=bool(causal)).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_value_shift_and_scale_are_linear():
    # bf16-valued inputs, so v + 0.75 is exact in float32 and the shift is the only change.
    q, k, v = si.qkv(61, 1, 2, 70, 64, "bf16")
    base = oracle.attn_fwd(q, k, v, True)
    c = np.float32(0.75)
    shifted = oracle.attn_fwd(q, k, (v + c).astype(np.float32), True)
    np.testing.assert_allclose(shifted, base + float(c), rtol=0, atol=1e-12)
    doubled = oracle.attn_fwd(q, k, (v * np.float32(2)).astype(np.float32), True)
    np.testing.assert_array_equal(doubled, 2.0 * base)


def test_key_shift_leaves_output_unchanged():
    # q.(k_j + c) = q.k_j + q.c, a constant along each row, and a softmax ignores constants.
    # bf16-valued keys, so k + c is exact in float32.
    q, k, v = si.qkv(71, 1, 1, 90, 64, "bf16")
    c = np.zeros(64, np.float32)
    c[3], c[40] = 0.5, -1.25
    base = oracle.attn_fwd(q, k, v, False)
    moved = oracle.attn_fwd(q, (k + c).astype(np.float32), v, False)
    np.testing.assert_allclose(moved, base, rtol=0, atol=1e-12)


def test_noncausal_is_invariant_to_joint_key_value_permutation():
    q, k, v = si.qkv(81, 1, 1, 64, 64)
    perm = np.random.default_rng(3).permutation(64)
    base = oracle.attn_fwd(q, k, v, False)
    moved = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], False)
    np.testing.assert_allclose(moved, base, rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value_exactly():
    # One score 1000 above the rest: exp(-1000) underflows to 0 in double, so the row is v_j.
    N, d, j = 16, 64, 9
    _, _, v = si.qkv(91, 1, 1, N, d)
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    q[..., 0] = 8.0
    k[0, 0, j, 0] = 1000.0
    o = oracle.attn_fwd(q, k, v, False)[0, 0]
    assert np.array_equal(o, np.repeat(v[0, 0, j][None].astype(np.float64), N, axis=0))
    # The same key under the causal mask only wins for rows at or after it.
    oc = oracle.attn_fwd(q, k, v, True)[0, 0]
    assert np.array_equal(oc[j:], o[j:])
    assert not np.allclose(oc[j - 1], v[0, 0, j])


def test_row_subset_and_thread_count_do_not_change_bits():
    q, k, v = si.qkv(101, 2, 2, 200, 64, "bf16")
    full = oracle.attn_fwd(q, k, v, True, threads=1)
    rows = np.array([0, 5, 199, 200, 399, 777], np.int64)
    part = oracle.attn_fwd(q, k, v, True, rows=rows, threads=7)
    flat = full.reshape(-1, 64)
    assert np.array_equal(part, flat[rows])
    assert np.array_equal(oracle.attn_fwd(q, k, v, True, threads=5), full)


def test_empty_problem_is_a_no_op():
    z = np.zeros((1, 2, 0, 64), np.float32)
    assert oracle.attn_fwd(z, z, z, True).shape == (1, 2, 0, 64)
