"""Error gates from the pages, in fp64 (test helpers, not part of the product).

column_gate_atol: "100 Days of GPU, Day 98" (The program, and the gate that
has to be per column; Exercise 'Check'): |got - ref| <= 4*K*max|A|*max|B[:,c]|/127,
with max|A| taken per token row when A is quantized per token, as the page's
Solution to the exercise does for a per-row scale.

scale_gate_atol: the same derivation written with the actual scales, which
also covers per-tensor weights: one term carries at most |a|*s_w/2 + |w|*s_a/2,
the slack 4 absorbs the second-order term and summation order.

relative_l2 / mismatch_ratio / max error: the three metrics of TileLang ch. 27
section 5.2; sqnr_db: Activation Quantization Architecture (sqnr_db helper).
"""
import numpy as np

GATE_SLACK = 4.0
INT8_MAX = 127.0


def reference_fp64(a, w):
    """fp64 matmul of the ORIGINAL fp32 inputs (never the dequantized copies)."""
    return np.asarray(a, np.float64) @ np.asarray(w, np.float64).T


def column_gate_atol(a, w, act_per_row):
    a = np.abs(np.asarray(a, np.float64))
    w = np.abs(np.asarray(w, np.float64))
    K = a.shape[1]
    amax = a.max(axis=1) if act_per_row else np.full(a.shape[0], a.max())
    wcol = w.max(axis=1)
    return GATE_SLACK * K * np.outer(amax, wcol) / INT8_MAX


def column_stat_atol(a, w, act_per_row):
    K = np.asarray(a).shape[1]
    return column_gate_atol(a, w, act_per_row) * np.sqrt(K) / K


def scale_gate_atol(a, w, sa, sw):
    a = np.abs(np.asarray(a, np.float64))
    w = np.abs(np.asarray(w, np.float64))
    K = a.shape[1]
    sa = np.broadcast_to(np.asarray(sa, np.float64).reshape(-1), (a.shape[0],))
    sw = np.broadcast_to(np.asarray(sw, np.float64).reshape(-1), (w.shape[0],))
    amax = a.max(axis=1)
    wcol = w.max(axis=1)
    per_term = np.outer(amax, sw) / 2 + np.outer(sa, wcol) / 2 + np.outer(sa, sw) / 4
    return GATE_SLACK * K * per_term


def first_violation(err, atol):
    bad = np.argwhere(err > atol)
    return None if bad.size == 0 else tuple(int(i) for i in bad[0])


def relative_l2(ref, got):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def sqnr_db(ref, got):
    ref = np.asarray(ref, np.float64)
    noise = np.sum((ref - np.asarray(got, np.float64)) ** 2)
    return float(10 * np.log10(np.sum(ref ** 2) / max(noise, 1e-30)))


def ulp_distance(x, y):
    """Distance in units in the last place between fp32 arrays (same sign assumed near 0)."""
    xi = np.asarray(x, np.float32).view(np.int32).astype(np.int64)
    yi = np.asarray(y, np.float32).view(np.int32).astype(np.int64)
    xi = np.where(xi < 0, np.int64(-2**31) - xi, xi)
    yi = np.where(yi < 0, np.int64(-2**31) - yi, yi)
    return np.abs(xi - yi)


def near_f32_midpoint(s, rel: float = 2.0 ** -36) -> np.ndarray:
    """True where the value s (float64) lies within rel * |s| of a midpoint between two
    adjacent fp32 values: there an accurate sum formed in another order may round to
    either neighbour, so both are correct results of the reading "exact sum, rounded once"."""
    s = np.asarray(s, np.float64)
    f = s.astype(np.float32)
    lo = np.nextafter(f, np.float32(-np.inf)).astype(np.float64)
    hi = np.nextafter(f, np.float32(np.inf)).astype(np.float64)
    f64 = f.astype(np.float64)
    d = np.minimum(np.abs(s - (f64 + lo) / 2), np.abs(s - (f64 + hi) / 2))
    return d <= rel * np.abs(s)
