"""The causal launch orders (a block -> work-item table planned on the host for calls of up
to 2048 work items, heaviest items first beyond that) decide only which SM runs which work item
(a pair of query tiles in the forward, a key or query block in the backward kernels), never
what an item computes. So a batched call must reproduce, bit for bit, the same heads computed
one call per head (whose plans differ), on both sides of the 2048-item limit; the per-head
calls themselves are checked against the oracle elsewhere.
"""

import pytest
import torch

import online_softmax_flashattention_gb300 as fa
import seeded_inputs as si
from attn_testlib import to_dev

pytestmark = pytest.mark.gpu


def _per_head_equal(B, H, N, d, dtype, seed):
    q, k, v = si.qkv(seed, B, H, N, d, dtype)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o_all, lse_all = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o1, lse1 = fa.attn_fwd_lse(qd[sl].contiguous(), kd[sl].contiguous(), vd[sl].contiguous(), causal=True)
            assert torch.equal(o1, o_all[sl]), f"head ({b}, {h}) of B{B} H{H} N{N} d{d} differs"
            assert torch.equal(lse1, lse_all[sl]), f"lse of head ({b}, {h}) differs"
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_planned_order_matches_per_head(d):
    # 2 x 12 heads x 16 pairs = 384 work items: a planned order, like the 16 of each head alone.
    _per_head_equal(2, 12, 4096, d, "bf16", 901)


def test_ragged_planned_order_matches_per_head():
    # N = 3000: the last pair of each head holds a ragged tile.
    _per_head_equal(1, 5, 3000, 64, "f16", 902)


def test_unplanned_order_matches_per_head():
    # 3 x 24 heads x 32 pairs = 2304 work items: past the table, heaviest pairs first; each head
    # alone (32 items) runs with a planned order.
    _per_head_equal(3, 24, 8192, 64, "bf16", 903)


def _bwd_per_head_equal(B, H, N, d, dtype, seed):
    q, k, v = si.qkv(seed, B, H, N, d, dtype)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    g = torch.Generator(device="cuda").manual_seed(seed)
    dout = torch.randn(qd.shape, generator=g, device="cuda", dtype=torch.float32).to(qd.dtype)
    o, lse = fa.attn_fwd_lse(qd, kd, vd, causal=True)
    grads = fa.attn_bwd(qd, kd, vd, o, dout, lse, causal=True)
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            one = fa.attn_bwd(*(t[sl].contiguous() for t in (qd, kd, vd, o, dout)), lse[sl].contiguous(), causal=True)
            for name, x1, xa in zip(("dq", "dk", "dv"), one, grads):
                assert torch.equal(x1, xa[sl]), f"{name} of head ({b}, {h}) of B{B} H{H} N{N} d{d} differs"
    torch.cuda.synchronize()
    assert fa.attn_device_status(clear=True) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_backward_planned_order_matches_per_head(d):
    # 2 x 12 heads x 32 blocks = 768 items per kernel: planned orders, like each head alone.
    _bwd_per_head_equal(2, 12, 4096, d, "bf16", 904)


def test_backward_unplanned_order_matches_per_head():
    # 3 x 24 heads x 64 blocks = 4608 items: heaviest first; each head alone is planned.
    _bwd_per_head_equal(3, 24, 8192, 64, "bf16", 905)
