"""GPU parity of attn_fwd_kvcache: Nq new queries (the last Nq positions) against a key-value
cache of Nk keys, the key range cut into shares merged by their log-sum-exps, against the
double oracle's key-value cache case on the same seeded inputs.

Tolerances: o as the forward's (bf16/fp16 2e-2 absolute against the double oracle on the same
rounded inputs; fp32 1e-5 * Nk * max|ref| and the attention.cu gate with N = Nk); lse as
attn_fwd_lse's, 2e-5 * (1 + max|lse|) + 1e-4 (fp32 scores from exact products over d = 64; the
merge adds one fp32 log2 and exp2 per share). Different share counts give the same result
within those bounds, not bit for bit (the sums are taken in another order).
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


def _inputs(seed, B, H, Nq, Nk, dtype, qk_scale=1.0, d=64):
    q = si.qkv(seed, B, H, Nq, d, dtype, qk_scale=qk_scale)[0]
    _, k, v = si.qkv(seed + 1, B, H, Nk, d, dtype, qk_scale=qk_scale)
    return q, k, v


def _run(seed, B, H, Nq, Nk, dtype, causal, splits, qk_scale=1.0, d=64):
    q, k, v = _inputs(seed, B, H, Nq, Nk, dtype, qk_scale, d)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=causal, num_splits=splits, lse=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, causal)
    got_o = o.float().cpu().numpy().astype(np.float64)
    check(got_o, ref_o, dtype, Nk, f"kvcache {dtype} Nq={Nq} Nk={Nk} splits={splits}", page_gate=(qk_scale == 1.0))
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_lse))
    err = float(np.max(np.abs(got_lse - ref_lse)))
    assert err <= _lse_bound(ref_lse), f"lse max err {err:.3e} > {_lse_bound(ref_lse):.3e}"
    return got_o, got_lse


SHAPES = [(1, 1), (1, 300), (1, 4096), (2, 77), (4, 257), (5, 1000), (8, 8), (16, 1000), (33, 64), (100, 100)]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_kvcache_against_oracle(dtype, causal, Nq, Nk, splits):
    _run(0xCAC30000 + Nq * 7919 + Nk, 2, 3, Nq, Nk, dtype, causal, splits)


@pytest.mark.parametrize("splits", [2, 7, 64, 200, 1024])
def test_kvcache_many_shares_including_empty_ones(splits):
    # 1024 shares over 300 keys: shares are whole 128-key tiles, so most are empty and must
    # carry weight 0 in the merge.
    _run(0xCAC31000 + splits, 1, 2, 3, 300, "bf16", True, splits)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kvcache_qk_scaled_x8(dtype):
    # Scores of std ~64: the online rescale and the share merge both see large maxima.
    _run(0xCAC32000, 1, 2, 4, 700, dtype, True, 5, qk_scale=8.0)


def test_kvcache_share_count_does_not_change_the_result_beyond_rounding():
    q, k, v = _inputs(0xCAC33000, 2, 4, 3, 2048, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    outs = [fa.attn_fwd_kvcache(qd, kd, vd, causal=True, num_splits=s, lse=True) for s in (1, 2, 5, 16, 64)]
    torch.cuda.synchronize()
    o0, l0 = outs[0]
    for o, l in outs[1:]:
        assert float((o.float() - o0.float()).abs().max()) <= 2 ** -7  # one bf16 ulp at |o| < 1, twice
        assert float((l - l0).abs().max()) <= 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_kvcache_square_case_matches_the_flash_forward(causal):
    # Nq == Nk is ordinary attention: same result as attn_fwd_lse within the forward's bounds.
    q, k, v = si.qkv(0xCAC34000, 1, 2, 200, 64, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=causal, num_splits=3, lse=True)
    o2, lse2 = fa.attn_fwd_lse(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert float((o.float() - o2.float()).abs().max()) <= 2e-2
    assert float((lse - lse2).abs().max()) <= 2e-4


def test_kvcache_single_visible_key_returns_its_value():
    # Causal with Nq == Nk: query 0 sees key 0 alone, so o[0] == v[0] exactly and lse == s_00 * log2 e.
    q, k, v = si.qkv(0xCAC35000, 1, 1, 16, 64, "f32")
    qd, kd, vd = (to_dev(x, "f32") for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, num_splits=4, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o[0, 0, 0].cpu(), torch.from_numpy(v[0, 0, 0]))
    s00 = float(np.dot(q[0, 0, 0].astype(np.float64), k[0, 0, 0].astype(np.float64))) / 8.0
    assert abs(float(lse[0, 0, 0]) - s00 / np.log(2.0)) <= 1e-5 * (1 + abs(s00))


@pytest.mark.parametrize("B,H,Nq,Nk", [(1, 1, 1, 100), (1, 2, 1, 100000), (3, 5, 2, 3000), (64, 12, 1, 300),
                                       (2, 3, 40, 5000), (1, 1, 9, 129)])
@pytest.mark.parametrize("causal", [False, True])
def test_kvcache_balanced_plan_over_head_boundaries(B, H, Nq, Nk, causal):
    # The balanced plan cuts the tiles of all heads into equal runs, so runs start and end
    # inside heads (several pieces per head, merged) or hold several whole heads (written
    # directly); tiny cases give fewer tiles than CTAs.
    _run(0xCAC38000 + B * 1000 + Nq * 10 + Nk, B, H, Nq, Nk, "bf16", causal, 0)


def test_kvcache_decode_workload_sampled():
    # One new token per sequence against an 8192-key cache, B16 H12 (the decode measurement's
    # shape), balanced plan; every query row is checked against the oracle.
    B, H, Nq, Nk = 16, 12, 1, 8192
    q, k, v = _inputs(0xCAC36000, B, H, Nq, Nk, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, lse=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, True)
    check(o.float().cpu().numpy().astype(np.float64), ref_o, "bf16", Nk, "decode B16H12 Nk8192")
    assert float(np.max(np.abs(lse.cpu().numpy() - ref_lse))) <= _lse_bound(ref_lse)


def test_kvcache_explicit_workspace_and_outputs_are_used():
    B, H, Nq, Nk, S = 1, 3, 2, 500, 6
    q, k, v = _inputs(0xCAC37000, B, H, Nq, Nk, "f16")
    qd, kd, vd = (to_dev(x, "f16") for x in (q, k, v))
    ws = torch.empty(fa.attn_kvcache_workspace_bytes(B, H, Nq, Nk, S, torch.float16), dtype=torch.uint8, device="cuda")
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), device="cuda")
    r = fa.attn_fwd_kvcache(qd, kd, vd, causal=False, num_splits=S, workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert r[0] is out and r[1] is lse
    ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, False)
    check(out.float().cpu().numpy().astype(np.float64), ref_o, "f16", Nk, "explicit workspace")
    assert float(np.max(np.abs(lse.cpu().numpy() - ref_lse))) <= _lse_bound(ref_lse)
    with pytest.raises(fa.AttnError):  # one byte short
        fa.attn_fwd_kvcache(qd, kd, vd, num_splits=S, workspace=ws[:-1])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 300), (3, 1000), (8, 129), (20, 700)])
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_kvcache_head_width_128(dtype, causal, Nq, Nk, splits):
    _run(0xCAC39000 + Nq * 7919 + Nk, 2, 3, Nq, Nk, dtype, causal, splits, d=128)


def test_kvcache_head_width_128_decode_shape():
    B, H, Nq, Nk = 8, 8, 1, 8192
    q, k, v = _inputs(0xCAC3A000, B, H, Nq, Nk, "bf16", d=128)
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, lse=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, True)
    check(o.float().cpu().numpy().astype(np.float64), ref_o, "bf16", Nk, "decode d128 B8H8 Nk8192")
    assert float(np.max(np.abs(lse.cpu().numpy() - ref_lse))) <= _lse_bound(ref_lse)


def test_kvcache_workspace_reused_across_calls_and_shapes():
    # One workspace serves a sequence of calls with different shapes and share counts, with
    # whatever the previous call left in it.
    ws = torch.full((1 << 22,), 0xFF, dtype=torch.uint8, device="cuda")
    for seed, (B, H, Nq, Nk, S) in enumerate([(1, 3, 2, 500, 6), (2, 2, 1, 3000, 0), (1, 3, 2, 500, 6),
                                              (3, 1, 9, 700, 4), (2, 2, 1, 3000, 0)]):
        q, k, v = _inputs(0xCAC3B000 + seed, B, H, Nq, Nk, "bf16")
        qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
        assert fa.attn_kvcache_workspace_bytes(B, H, Nq, Nk, S, torch.bfloat16) <= ws.numel()
        o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, num_splits=S, workspace=ws, lse=True)
        torch.cuda.synchronize()
        ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, True)
        check(o.float().cpu().numpy().astype(np.float64), ref_o, "bf16", Nk, f"reuse call {seed}")
        assert float(np.max(np.abs(lse.cpu().numpy() - ref_lse))) <= _lse_bound(ref_lse)


@pytest.mark.parametrize("splits", [0, 1, 4])
def test_kvcache_causal_rows_ignore_keys_they_cannot_see(splits):
    # Causal with Nq = 6 new queries: query i sees keys 0 .. Nk - Nq + i. Rewriting the keys and
    # values past query 2's position must leave queries 0..2 bit-identical (their weights on
    # those keys are exactly zero) and change query 5.
    B, H, Nq, Nk = 1, 2, 6, 700
    q, k, v = _inputs(0xCAC3C000, B, H, Nq, Nk, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o1, l1 = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, num_splits=splits, lse=True)
    last_seen = Nk - Nq + 2
    kd2, vd2 = kd.clone(), vd.clone()
    kd2[:, :, last_seen + 1:] = torch.randn_like(kd2[:, :, last_seen + 1:]) * 3
    vd2[:, :, last_seen + 1:] = torch.randn_like(vd2[:, :, last_seen + 1:]) * 3
    o2, l2 = fa.attn_fwd_kvcache(qd, kd2, vd2, causal=True, num_splits=splits, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :, :3], o2[:, :, :3]) and torch.equal(l1[:, :, :3], l2[:, :, :3])
    assert not torch.equal(o1[:, :, 5], o2[:, :, 5])


def test_kvcache_noncausal_ignores_key_order():
    # Without the mask, permuting the cache rows (keys and values together) permutes nothing in
    # the result: equal within rounding of the summation order.
    B, H, Nq, Nk = 2, 2, 3, 900
    q, k, v = _inputs(0xCAC3D000, B, H, Nq, Nk, "f32")
    qd, kd, vd = (to_dev(x, "f32") for x in (q, k, v))
    perm = torch.randperm(Nk, generator=torch.Generator().manual_seed(5)).to("cuda")
    o1 = fa.attn_fwd_kvcache(qd, kd, vd, causal=False)
    o2 = fa.attn_fwd_kvcache(qd, kd[:, :, perm].contiguous(), vd[:, :, perm].contiguous(), causal=False)
    torch.cuda.synchronize()
    assert float((o1 - o2).abs().max()) <= 1e-5


@pytest.mark.parametrize("Nq", [2, 3, 4, 8])
def test_kvcache_tensor_core_decode_shape(Nq):
    # A few new tokens per sequence against an 8192-key cache, B16 H12: at d = 64, 3 to 8 queries
    # run on the tensor-core kernel (queries padded to a 128-row tile), 2 on CUDA cores; balanced
    # plan, every query row against the oracle.
    B, H, Nk = 16, 12, 8192
    q, k, v = _inputs(0xCAC3E000 + Nq, B, H, Nq, Nk, "bf16")
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    o, lse = fa.attn_fwd_kvcache(qd, kd, vd, causal=True, lse=True)
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0
    ref_o, ref_lse = oracle.attn_fwd_kv(q, k, v, True)
    check(o.float().cpu().numpy().astype(np.float64), ref_o, "bf16", Nk, f"decode B16H12 Nq{Nq} Nk8192")
    assert float(np.max(np.abs(lse.cpu().numpy() - ref_lse))) <= _lse_bound(ref_lse)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(127, 300), (128, 128), (129, 1000), (200, 200), (300, 5000)])
@pytest.mark.parametrize("splits", [0, 2])
def test_kvcache_query_groups_of_128(dtype, causal, Nq, Nk, splits):
    # The tensor-core kernel takes a head's queries 128 at a time: a group filling the tile, a
    # ragged last group, several groups with the causal diagonal inside the cache, Nq == Nk.
    _run(0xCAC3F000 + Nq * 7919 + Nk, 2, 2, Nq, Nk, dtype, causal, splits)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(2, 65), (8, 8192), (129, 1000), (200, 200)])
@pytest.mark.parametrize("splits", [0, 3])
def test_kvcache_tensor_cores_head_width_128(dtype, causal, Nq, Nk, splits):
    # At d = 128 the tensor-core kernel streams 64-key tiles (two 64-value column blocks per
    # row): a ragged single key past one tile, a long cache, several query groups, Nq == Nk.
    _run(0xCAC3F800 + Nq * 7919 + Nk, 2, 2, Nq, Nk, dtype, causal, splits, d=128)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,splits", [(1, 2, 2, 40000, 0), (1, 1, 3, 33000, 0), (1, 1, 2, 33000, 7)])
def test_kvcache_tensor_cores_long_cache_few_queries(B, H, Nq, Nk, splits, causal):
    # Two 16-bit queries at d = 64 take the tensor-core kernel only on long caches (32768 keys or
    # more); three take it from 1024 keys: balanced and explicit shares over a cache of a few
    # hundred tiles.
    _run(0xCAC3FC00 + Nq * 7919 + Nk, B, H, Nq, Nk, "bf16", causal, splits)


@pytest.mark.parametrize("H,Nk", [(256, 1024), (255, 1024), (256, 1023)])
def test_kvcache_kernel_choice_boundary(H, Nk):
    # Three 16-bit queries at d = 64 move to the tensor-core kernel at 1024 keys and 2^18 cached
    # rows in the call (H256 Nk1024); one head fewer, or one key fewer, stays on CUDA cores. Both
    # sides of the boundary against the oracle.
    _run(0xCAC3FE00 + H * 7 + Nk, 1, H, 3, Nk, "bf16", True, 0)
