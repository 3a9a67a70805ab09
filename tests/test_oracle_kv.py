"""Pins for the oracle's key-value cache case: Nq new queries, the last Nq positions, against
Nk >= Nq keys; when causal, query i sees keys 0 .. Nk - Nq + i (the plain reading of the page's
mention of generation with a cache, where a few new tokens attend to every cached key, section
"Backwards, and training with it"). Pins: PyTorch float64 attention with that mask written out, 40-digit
decimal brute force, closed forms (equal scores; one visible key), and the reduction to the
ordinary causal case when Nq = Nk.
"""

import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import seeded_inputs as si


def _qkv(seed, B, H, Nq, Nk, d, qk_scale=1.0):
    q = si.qkv(seed, B, H, Nq, d, qk_scale=qk_scale)[0]
    _, k, v = si.qkv(seed + 1, B, H, Nk, d, qk_scale=qk_scale)
    return q, k, v


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 300), (4, 257), (16, 1000), (33, 64)])
def test_matches_torch_float64_with_bottom_right_mask(causal, Nq, Nk):
    torch = pytest.importorskip("torch")
    q, k, v = _qkv(301, 2, 3, Nq, Nk, 64)
    o, lse = oracle.attn_fwd_kv(q, k, v, causal)
    tq, tk, tv = (torch.from_numpy(x).double() for x in (q, k, v))
    mask = None
    if causal:
        mask = torch.arange(Nk)[None, :] <= (Nk - Nq + torch.arange(Nq))[:, None]
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).numpy()
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-13)
    s = tq @ tk.transpose(-1, -2) / 8.0
    if causal:
        s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, (torch.logsumexp(s, -1) / math.log(2.0)).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [0, 1])
def test_square_case_is_the_ordinary_attention(causal):
    q, k, v = si.qkv(311, 1, 2, 50, 64)
    o, lse = oracle.attn_fwd_kv(q, k, v, causal)
    o2, lse2 = oracle.attn_fwd_lse(q, k, v, causal)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [0, 1])
def test_equal_scores_give_mean_of_visible_values(causal):
    Nq, Nk, d = 5, 40, 64
    _, k, v = _qkv(321, 1, 1, Nq, Nk, d)
    q = np.zeros((1, 1, Nq, d), np.float32)
    o, lse = oracle.attn_fwd_kv(q, k, v, causal)
    for i in range(Nq):
        n = (Nk - Nq + i + 1) if causal else Nk
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log2(n)) <= 1e-13


def test_decimal_brute_force():
    Nq, Nk, d = 3, 7, 8
    q, k, v = _qkv(331, 1, 1, Nq, Nk, d, qk_scale=2.0)
    o, lse = oracle.attn_fwd_kv(q, k, v, True)
    getcontext().prec = 40
    scale = Decimal(1) / Decimal(d).sqrt()
    for i in range(Nq):
        vis = range(Nk - Nq + i + 1)
        sc = [sum(Decimal(float(q[0, 0, i, e])) * Decimal(float(k[0, 0, j, e])) for e in range(d)) * scale for j in vis]
        ex = [x.exp() for x in sc]
        tot = sum(ex)
        for e in range(d):
            want = float(sum(ex[n] * Decimal(float(v[0, 0, j, e])) for n, j in enumerate(vis)) / tot)
            assert abs(o[0, 0, i, e] - want) <= 1e-14 * max(1.0, abs(want))
        assert abs(lse[0, 0, i] - float(tot.ln() / Decimal(2).ln())) <= 1e-13


def test_first_query_of_causal_cache_sees_whole_cache_and_itself():
    # Query 0 is at position Nk - Nq: changing key Nk - Nq + 1 (a later new token) leaves it alone.
    Nq, Nk = 4, 30
    q, k, v = _qkv(341, 1, 1, Nq, Nk, 64)
    o, _ = oracle.attn_fwd_kv(q, k, v, True)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, Nk - Nq + 1:] += 1.0
    v2[0, 0, Nk - Nq + 1:] += 1.0
    o2, _ = oracle.attn_fwd_kv(q, k2, v2, True)
    assert np.array_equal(o[0, 0, 0], o2[0, 0, 0])
    assert not np.array_equal(o[0, 0, 1:], o2[0, 0, 1:])
