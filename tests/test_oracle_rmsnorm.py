"""Pins of the oracle's fused RMSNorm + per-token quantization (CPU only).

The step follows "Activation Quantization Architecture" (Fusion: the fused
norm-and-quantize pseudocode): rms = sqrt(mean(x * x) + eps), y = x / rms * gamma,
then the symmetric per-token quantizer on y. The pages leave the order of the sum
in mean(x * x) open; the reading taken is the exact sum of squares rounded once
to fp32. Each pin below fails for a plausible mistake: a dropped root, a sum in
place of the mean, eps outside the root, gamma ignored or misplaced, a fp32
running sum, a multiply by the reciprocal instead of the division.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from tests import gates


def _nearest_f32(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 value of a non-negative rational."""
    f = np.float32(float(q))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - q), int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def _brute_rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Exact rational sum of squares, one rounding, then numpy fp32 operations in order."""
    rows, cols = x.shape
    y = np.empty_like(x)
    for r in range(rows):
        s = sum(Fraction(float(v)) ** 2 for v in x[r])
        ms = _nearest_f32(s)
        mean = np.float32(ms / np.float32(cols))
        rms = np.sqrt(np.float32(mean + np.float32(eps)), dtype=np.float32)
        y[r] = (x[r] / rms).astype(np.float32) * gamma
    return y


def test_constant_row_gives_gamma():
    # x_k = c: S = K c^2 exactly, mean = c^2, rms = |c|, x / rms = sign(c): y = +-gamma exactly
    gamma = np.linspace(0.25, 3.0, 64, dtype=np.float32)
    for c in (3.0, 0.75, -12.0):
        x = np.full((2, 64), c, np.float32)
        y, ss = oracle.rmsnorm(x, gamma, 0.0)
        np.testing.assert_array_equal(y, np.sign(c) * np.broadcast_to(gamma, (2, 64)))
        assert ss[0] == 64 * c * c


def test_power_of_two_scale_invariance():
    # with eps = 0, scaling a row by 2^k scales S by 4^k exactly and rms by 2^k exactly
    x = workloads.gaussian((8, 512), 3)
    gamma = (1.0 + 0.1 * workloads.gaussian((512,), 4)).astype(np.float32)
    y0, _ = oracle.rmsnorm(x, gamma, 0.0)
    for k in (-6, 3, 10):
        yk, _ = oracle.rmsnorm((x * np.float32(2.0 ** k)).astype(np.float32), gamma, 0.0)
        np.testing.assert_array_equal(yk, y0)


def test_unit_rms_with_unit_gamma():
    x = workloads.gaussian((16, 2048), 5) * np.float32(7.0)
    y, _ = oracle.rmsnorm(x, np.ones(2048, np.float32), 0.0)
    rms = np.sqrt(np.mean(y.astype(np.float64) ** 2, axis=1))
    np.testing.assert_allclose(rms, 1.0, rtol=2e-6)


def test_eps_sits_under_the_root():
    x = np.full((1, 16), 1e-4, np.float32)
    y, _ = oracle.rmsnorm(x, np.ones(16, np.float32), 1e-2)
    want = 1e-4 / np.sqrt(1e-8 + 1e-2)
    np.testing.assert_allclose(y, want, rtol=1e-6)


def test_gamma_is_per_channel():
    x = workloads.gaussian((4, 256), 6)
    g1 = np.ones(256, np.float32)
    g2 = g1.copy()
    g2[17] = 2.0
    y1, _ = oracle.rmsnorm(x, g1, 1e-6)
    y2, _ = oracle.rmsnorm(x, g2, 1e-6)
    np.testing.assert_array_equal(y2[:, 17], 2.0 * y1[:, 17])
    np.testing.assert_array_equal(np.delete(y2, 17, axis=1), np.delete(y1, 17, axis=1))


def test_brute_force_exact_sum_then_fp32_steps():
    x = workloads.gaussian((5, 48), 7) * np.float32(3.0)
    # a row where a fp32 running sum loses every small square: 1 + 16 * 2^-24 is exact in
    # fp32 (1 + 2^-20) but 1 + 2^-24 rounds back to 1 at every step
    x[4] = 0.0
    x[4, 0] = 1.0
    x[4, 1:17] = np.float32(2.0 ** -12)
    gamma = (1.0 + 0.2 * workloads.gaussian((48,), 17)).astype(np.float32)
    for eps in (0.0, 1e-6):
        y, _ = oracle.rmsnorm(x, gamma, eps)
        np.testing.assert_array_equal(y, _brute_rmsnorm(x, gamma, eps))
    y4, ss4 = oracle.rmsnorm(x[4:5], np.ones(48, np.float32), 0.0)
    assert ss4[0] == 1.0 + 16 * 2.0 ** -24


def test_zero_row_quantizes_to_zero_with_guarded_scale():
    x = np.zeros((2, 64), np.float32)
    out = oracle.rmsnorm_quantize(x, np.ones(64, np.float32), 1e-6)
    assert np.all(out["qa"] == 0)
    assert np.all(out["y"] == 0)
    np.testing.assert_array_equal(out["sa"], np.float32(np.float32(1e-8) / np.float32(127.0)))


def test_codes_follow_the_per_token_quantizer_on_y():
    x = workloads.gaussian((6, 320), 8)
    x[:, 5] *= 40.0                       # an outlier channel, as in the pages' harness
    gamma = (1.0 + 0.1 * workloads.gaussian((320,), 18)).astype(np.float32)
    out = oracle.rmsnorm_quantize(x, gamma, 1e-6)
    y = out["y"]
    s_want = (np.max(np.abs(y), axis=1) / np.float32(127.0)).astype(np.float32)
    np.testing.assert_array_equal(out["sa"], s_want)
    q_want = np.clip(np.rint(y / s_want[:, None]), -127, 127).astype(np.int8)
    np.testing.assert_array_equal(out["qa"], q_want)


def test_midpoint_flag():
    # exactly on a midpoint between two fp32 values, and far from one
    one = np.float64(1.0)
    mid = one + 2.0 ** -24
    flags = gates.near_f32_midpoint(np.array([mid, one, 1.0 + 2.0 ** -23 * 0.25]))
    assert flags.tolist() == [True, False, False]


def test_mean_plus_eps_rounds_in_fp32():
    # mean = c^2 exactly (constant row); fl32(c^2 + eps) rounds up across a point where the
    # root changes, so an fp64 root argument would give rms = c exactly and y = 1
    c = np.float32(2.890625)
    eps = float(np.float32(5.193561491978471e-07))
    x = np.full((1, 64), c, np.float32)
    y, _ = oracle.rmsnorm(x, np.ones(64, np.float32), eps)
    rms32 = np.sqrt(np.float32(c * c + np.float32(eps)), dtype=np.float32)
    assert rms32 != c
    np.testing.assert_array_equal(y, np.float32(c / rms32))
    assert y[0, 0] != 1.0
