"""Pins of the shared seeded input generator (conversions, distributions, random access)."""
import math

import numpy as np
import pytest

import syngen


def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 lies exactly between bf16 1.0 (0x3F80) and 1 + 2^-7 (0x3F81): ties to even.
    assert syngen.f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 lies between 0x3F81 and 0x3F82: ties to even -> 0x3F82.
    assert syngen.f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the midpoint rounds up
    assert syngen.f32_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 0x3F81
    assert syngen.f32_to_bf16(-2.0) == 0xC000
    assert syngen.f32_to_bf16(0.0) == 0x0000
    assert syngen.f32_to_bf16(-0.0) == 0x8000


def test_bf16_matches_exact_rounding_on_random_values():
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(20000).astype(np.float32)
    for x in xs[:2000]:
        b = syngen.f32_to_bf16(float(x))
        # candidate neighbours by truncation; the chosen one must be nearest
        bits = int(np.float32(x).view(np.uint32))
        lo = (bits >> 16) & 0xFFFF
        cands = [lo, lo + 1]
        vals = [np.uint32(c << 16).view(np.float32) for c in cands]
        d = [abs(float(v) - float(x)) for v in vals]
        if d[0] != d[1]:
            assert b == cands[int(np.argmin(d))]
        else:
            assert b == (lo if lo % 2 == 0 else lo + 1)


def test_f16_conversion_special_values():
    assert syngen.f64_to_f16(1.0) == 0x3C00
    assert syngen.f64_to_f16(1.0 / 3.0) == 0x3555
    assert syngen.f64_to_f16(65504.0) == 0x7BFF
    assert syngen.f64_to_f16(65519.0) == 0x7BFF
    assert syngen.f64_to_f16(65520.0) == 0x7C00
    assert syngen.f64_to_f16(2.0 ** -24) == 0x0001
    assert syngen.f64_to_f16(2.0 ** -25) == 0x0000          # tie -> even (0)
    assert syngen.f64_to_f16(3 * 2.0 ** -25) == 0x0002      # 1.5 units -> even (2)
    assert syngen.f64_to_f16(2.0 ** -14) == 0x0400
    assert syngen.f64_to_f16(-2.0) == 0xC000


def test_f16_conversion_matches_numpy():
    # numpy's float64 -> float16 cast rounds to nearest even (a library routine)
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(20000) * 0.02, rng.standard_normal(2000) * 1e-5,
                         rng.standard_normal(2000) * 3e4])
    ours = np.array([syngen.f64_to_f16(float(v)) for v in xs], np.uint16)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_q4_uniform_over_minus8_to_7():
    q = syngen.q4(0, 0, syngen.T_GATE_Q, 0, 1 << 20)
    assert q.min() == -8 and q.max() == 7
    counts = np.bincount(q.astype(np.int64) + 8, minlength=16)
    expected = q.size / 16
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 60.0  # 15 dof; p ~ 1e-7 threshold


def test_normal_moments():
    z = syngen.normal_f32(0, 3, syngen.T_ROUTER, 0, 1 << 18, 0.02).astype(np.float64)
    assert abs(z.mean()) < 0.02 * 5 / math.sqrt(z.size)
    assert abs(z.std() - 0.02) < 0.02 * 0.01
    s = syngen.absnormal_f16(0, 3, syngen.T_GATE_S, 0, 1 << 16, 0.02).view(np.float16).astype(np.float64)
    assert (s >= 0).all()
    # median of |N(0, sigma)| is sigma * 0.6745
    assert abs(np.median(s) - 0.02 * 0.67449) < 0.02 * 0.02


def test_random_access_matches_sequential():
    full = syngen.q4(7, 2, syngen.T_DOWN_Q, 0, 1000)
    for a, b in [(0, 1), (3, 17), (15, 16), (16, 33), (999, 1000), (123, 877)]:
        np.testing.assert_array_equal(syngen.q4(7, 2, syngen.T_DOWN_Q, a, b - a), full[a:b])
    fn = syngen.normal_f32(7, 2, syngen.T_ROUTER, 0, 300, 0.02)
    np.testing.assert_array_equal(syngen.normal_f32(7, 2, syngen.T_ROUTER, 100, 50, 0.02), fn[100:150])


def test_streams_are_distinct():
    a = syngen.q4(0, 0, syngen.T_GATE_Q, 0, 4096)
    assert not np.array_equal(a, syngen.q4(0, 1, syngen.T_GATE_Q, 0, 4096))
    assert not np.array_equal(a, syngen.q4(0, 0, syngen.T_UP_Q, 0, 4096))
    assert not np.array_equal(a, syngen.q4(1, 0, syngen.T_GATE_Q, 0, 4096))


def test_rows_recipe():
    cfg = syngen.CONFIGS["a3b_r4"]
    x = syngen.rows(cfg, 0)
    assert x.shape == (4, 2048) and x.dtype == np.uint16
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    # rows share x0: their mean difference has variance 2 sigma^2
    d = (xf[1] - xf[0]).astype(np.float64)
    assert abs(d.std() - 0.5 * math.sqrt(2)) < 0.05
    # sigma = 0 gives identical rows equal to bf16(x0)
    x1 = syngen.rows(cfg, 0, n_rows=3, sigma=0.0)
    assert (x1 == x1[0]).all()
    x0 = syngen.normal_f32(cfg.seed, 0, syngen.T_X0, 0, 2048, 1.0)
    np.testing.assert_array_equal(x1[0], np.array([syngen.f32_to_bf16(float(v)) for v in x0], np.uint16))
