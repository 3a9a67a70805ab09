"""Host tests of the launch-order planner (attn_plan_launch_order), no GPU: the order is a
permutation of the items, list scheduling in that order (the next item to the first free bin,
as the hardware dispatches blocks) never ends later than heaviest-first and on the causal
shapes of the library's kernels ends within a few per cent of the even split; degenerate
inputs and invalid arguments behave as the header states.
"""

import heapq

import pytest

import online_softmax_flashattention_gb300 as fa


def list_schedule(weights, order, fixed, bins):
    """Makespan of dispatching items in `order`, each to the bin that frees up first."""
    heap = [(0, b) for b in range(bins)]
    heapq.heapify(heap)
    for i in order:
        t, b = heapq.heappop(heap)
        heapq.heappush(heap, (t + weights[i] + fixed, b))
    return max(t for t, _ in heap)


def causal_pairs(n_pairs, heads):
    # forward work items: pair p of 128-row query tiles sees 2p + 2 key tiles of 128 keys
    return [2 * p + 2 for p in range(n_pairs) for _ in range(heads)]


def causal_pairs_wide(n_pairs, heads):
    # head width 128: 64-key tiles, so pair p of 128-row query tiles sees 4p + 4 of them
    return [4 * p + 4 for p in range(n_pairs) for _ in range(heads)]


def causal_blocks(n_blocks, heads):
    # backward dK/dV items: key block kb sees n_blocks - kb query blocks
    return [n_blocks - kb for kb in range(n_blocks) for _ in range(heads)]


def kv_blocks_wide(n, heads):
    # backward dK/dV at head width 128: key block kb (128 keys) sees the 64-query blocks from
    # its own on, n / 64 - 2 kb of them
    return [n // 64 - 2 * kb for kb in range(n // 128) for _ in range(heads)]


@pytest.mark.parametrize("weights,fixed,bins", [
    (causal_pairs(32, 12), 5, 152),   # forward, B1 H12 N8192
    (causal_pairs(16, 24), 5, 152),   # forward, B2 H12 N4096
    (causal_pairs_wide(32, 12), 5, 152),  # forward, B1 H12 N8192 d128
    (causal_blocks(64, 12), 3, 152),  # backward kernels, B1 H12 N8192
    (kv_blocks_wide(4096, 24), 3, 152),  # backward dK/dV at d128, B2 H12 N4096
    (causal_blocks(32, 12), 3, 148),
])
def test_planned_order_beats_heaviest_first(weights, fixed, bins):
    order = fa.attn_plan_launch_order(weights, fixed, bins)
    assert sorted(order) == list(range(len(weights)))
    heaviest = sorted(range(len(weights)), key=lambda i: -weights[i])
    planned = list_schedule(weights, order, fixed, bins)
    lpt = list_schedule(weights, heaviest, fixed, bins)
    even = (sum(weights) + fixed * len(weights)) / bins
    lower = max(even, max(weights) + fixed)
    assert planned <= lpt
    assert planned <= 1.03 * lower + 1


def test_headline_plan_improves_on_heaviest_first():
    # the forward's B1 H12 N8192 grid: heaviest-first ends 107 steps in, the packing about 98
    w = causal_pairs(32, 12)
    order = fa.attn_plan_launch_order(w, 5, 152)
    assert list_schedule(w, order, 5, 152) <= 99
    assert list_schedule(w, sorted(range(len(w)), key=lambda i: -w[i]), 5, 152) >= 105


def test_degenerate_inputs():
    assert fa.attn_plan_launch_order([7], 0, 152) == [0]
    order = fa.attn_plan_launch_order([3] * 10, 1, 4)
    assert sorted(order) == list(range(10))
    assert list_schedule([3] * 10, order, 1, 4) == 12  # ceil(10 / 4) items of 4 on a bin
    order = fa.attn_plan_launch_order([0, 5, 0, 9], 0, 1)
    assert sorted(order) == [0, 1, 2, 3]
    # one bin: every order has the same makespan; the plan starts with the heaviest
    assert order[0] == 3


def test_large_weights_end_quickly():
    # weights near the limit: the doubling capacity step keeps the search short
    import random
    import time

    rng = random.Random(7)
    w = [rng.randrange(1 << 24) for _ in range(2048)]
    t0 = time.perf_counter()
    order = fa.attn_plan_launch_order(w, 1 << 24, 152)
    assert time.perf_counter() - t0 < 30
    assert sorted(order) == list(range(len(w)))
    even = (sum(w) + (1 << 24) * len(w)) / 152
    assert list_schedule(w, order, 1 << 24, 152) <= even + 2 * (2 << 24)


@pytest.mark.parametrize("n,bins", [(8192, 128), (2048, 512)])
def test_largest_accepted_input_is_cheap(n, bins):
    # the largest inputs the bounds accept, with the largest weights, plan in well under a second
    import random
    import time

    rng = random.Random(n + bins)
    w = [rng.randrange(1 << 24) for _ in range(n)]
    t0 = time.perf_counter()
    order = fa.attn_plan_launch_order(w, 1 << 24, bins)
    assert time.perf_counter() - t0 < 3.0
    assert sorted(order) == list(range(n))


def test_invalid_arguments():
    import ctypes

    lib = fa.raw()
    w = (ctypes.c_int32 * 3)(1, 2, 3)
    out = (ctypes.c_uint16 * 3)()
    wp, op = ctypes.cast(w, ctypes.c_void_p), ctypes.cast(out, ctypes.c_void_p)
    assert lib.attn_plan_launch_order(wp, 3, 0, 4, op) == 0
    assert lib.attn_plan_launch_order(None, 3, 0, 4, op) == 1
    assert lib.attn_plan_launch_order(wp, 3, 0, 4, None) == 1
    assert lib.attn_plan_launch_order(wp, 0, 0, 4, op) == 1
    assert lib.attn_plan_launch_order(wp, 8193, 0, 4, op) == 1
    assert lib.attn_plan_launch_order(wp, 3, -1, 4, op) == 1
    assert lib.attn_plan_launch_order(wp, 3, 0, 0, op) == 1
    assert lib.attn_plan_launch_order(wp, 3, 0, 1025, op) == 1
    big = (ctypes.c_int32 * 2049)()
    bigo = (ctypes.c_uint16 * 2049)()
    # 2049 items over 512 bins exceeds the n * num_sms bound of 2^20
    assert lib.attn_plan_launch_order(ctypes.cast(big, ctypes.c_void_p), 2049, 0, 512,
                                      ctypes.cast(bigo, ctypes.c_void_p)) == 1
    assert lib.attn_plan_launch_order(wp, 3, (1 << 24) + 1, 4, op) == 1
    bad = (ctypes.c_int32 * 3)(1, -2, 3)
    assert lib.attn_plan_launch_order(ctypes.cast(bad, ctypes.c_void_p), 3, 0, 4, op) == 1
    with pytest.raises(fa.AttnError):
        fa.attn_plan_launch_order([1, 2], 0, 0)
