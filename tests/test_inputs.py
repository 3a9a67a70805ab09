"""The seeded input generator: published SplitMix64 vectors, rounding, determinism."""

import numpy as np
import pytest

import seeded_inputs as si


def test_splitmix64_matches_published_outputs_for_state_zero():
    # First three outputs of SplitMix64 started from state 0 (Vigna's reference splitmix64.c).
    g = 0x9E3779B97F4A7C15
    z = np.array([(g * n) % 2**64 for n in (1, 2, 3)], dtype=np.uint64)
    assert [int(x) for x in si._mix64(z)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_deterministic_and_distinct():
    a = si.normal_f32(7, 0, 1001)
    assert np.array_equal(a, si.normal_f32(7, 0, 1001))
    assert not np.array_equal(a, si.normal_f32(7, 1, 1001))
    assert not np.array_equal(a, si.normal_f32(8, 0, 1001))
    # Chunking does not change values: a prefix of a longer draw is the shorter draw.
    assert np.array_equal(si.normal_f32(7, 0, 4000)[:1001], a)


def test_c_generator_matches_numpy_definition():
    # Same arithmetic; the two libm implementations may differ in a last double bit, which
    # can move a float32 rounding by one ulp in about one element in 2**29.
    c = si.normal_f32(12, 2, 200001)
    n = si.normal_f32_numpy(12, 2, 200001)
    diff = np.flatnonzero(c != n)
    assert len(diff) <= 2
    assert np.all(np.abs(c[diff] - n[diff]) <= np.spacing(np.abs(n[diff])))


def test_normal_moments():
    x = si.normal_f32(3, 2, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs(np.mean(x ** 4) - 3.0) < 0.05


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = si.normal_f32(4, 0, 1 << 16) * np.float32(3.7)
    ours = si.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_round_to_is_idempotent_and_exact():
    x = si.normal_f32(9, 1, 4096)
    for dt in ("f32", "bf16", "f16"):
        r = si.round_to(x, dt)
        assert np.array_equal(si.round_to(r, dt), r)


def test_sample_rows_includes_ends_and_is_sorted():
    rows = si.sample_rows(5, 131072, 512)
    assert rows[0] == 0 and rows[-1] == 131071
    assert np.all(np.diff(rows) > 0)
    assert 512 <= len(rows) <= 514
    assert np.array_equal(si.sample_rows(5, 10, 512), np.arange(10))


def test_spike_late_pattern():
    q, k, v = si.spike_late(64, 64)
    i, e = 5, 3
    assert q[i, e] == np.float32(((i * 31 + e * 7) % 97) - 48) * np.float32(0.021)
    assert k[61, e] == np.float32(((61 * 17 + e * 11) % 89) - 44) * np.float32(0.019) * np.float32(3.0)
