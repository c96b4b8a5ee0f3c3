"""Pins of the oracle's block-scaled (MX-style) int8 weights (CPU only).

TileLang tutorial ch. 27 (low-precision quantization), 2.3 MX / block-scaled:
every G consecutive K elements share one E8M0 scale, a power of two stored as its
biased exponent; the scale is amax / qmax rounded UP to a power of two (exponent
field of x plus one when x's mantissa is not zero); four scale bytes are packed
per 32-bit word, b0 | b1 << 8 | b2 << 16 | b3 << 24, words indexed group-major
(g * rows + row); the granularity must be explicit, and a reversed byte order or
a row-major index gives errors of the size of the values themselves. Oracle
readings: qmax = 127, codes clamp(rint(w / s), -127, 127), exponent clamped to
[103, 136] (2^-24 .. 2^9), T = sum_k qa q s exact and rounded once to fp32.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads


def ceil_pow2_exponent(x: float) -> int:
    """Biased exponent of the smallest power of two >= x, by frexp (x = m 2^e, 0.5 <= m < 1)."""
    if x == 0.0:
        return 0
    m, e = math.frexp(x)
    return 127 + (e - 1 if m == 0.5 else e)


def nearest_f32(v: Fraction) -> np.float32:
    """The fp32 nearest to an exact rational (ties to even), without double rounding."""
    if v == 0:
        return np.float32(0.0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a.numerator)) - math.floor(math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)                 # normal range only in these tests
    q, r = divmod(a, ulp)
    q = int(q)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    return np.float32(sign * float(q * ulp))


def decode_scales(sf: np.ndarray, N: int, K: int, G: int) -> np.ndarray:
    """float64 [N, K / G] scales from the words: group g of row n is byte g % 4 of word (g // 4, n)."""
    out = np.empty((N, K // G))
    for n in range(N):
        for g in range(K // G):
            e = (int(sf[g // 4, n]) >> (8 * (g % 4))) & 0xFF
            out[n, g] = 2.0 ** (e - 127)
    return out


def block_weights(N, K, G, seed):
    """Rows whose magnitude changes from group to group (std LU[2^-8, 1] per group)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K)).astype(np.float32)
    mag = np.exp(rng.uniform(np.log(2.0 ** -8), 0.0, size=(N, K // G))).astype(np.float32)
    return (w.reshape(N, K // G, G) * mag[:, :, None]).reshape(N, K).astype(np.float32)


def test_e8m0_rounds_up_to_a_power_of_two():
    assert oracle.e8m0_ceil(1.0) == 127                      # a power of two stays
    assert oracle.e8m0_ceil(0.75) == 127                     # 0.75 -> 1, not 0.5
    assert oracle.e8m0_ceil(0.5) == 126
    assert oracle.e8m0_ceil(float(np.nextafter(np.float32(0.5), np.float32(1)))) == 127   # one ulp above
    assert oracle.e8m0_ceil(2.0 ** -10) == 117
    assert oracle.e8m0_ceil(0.0) == 103                      # reading: clamped to 2^-24
    assert oracle.e8m0_ceil(1e6) == 136                      # reading: clamped to 2^9
    rng = np.random.default_rng(7)
    xs = np.exp(rng.uniform(np.log(2.0 ** -24), np.log(2.0 ** 9), 4000)).astype(np.float32)
    xs = np.concatenate([xs, np.float32(2.0) ** np.arange(-24, 10, dtype=np.float32)])
    for x in xs:
        want = min(max(ceil_pow2_exponent(float(x)), 103), 136)
        assert oracle.e8m0_ceil(float(x)) == want, x


@pytest.mark.parametrize("G", [32, 128])
def test_codes_fit_scales_are_tight_and_error_is_half_a_step(G):
    N, K = 24, 16 * G
    w = block_weights(N, K, G, seed=G)
    q, sf = oracle.quantize_weight_mx(w, G)
    s = decode_scales(sf, N, K, G)
    amax = np.abs(w.reshape(N, K // G, G)).max(axis=2)
    x = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    assert np.all(s >= x)                                    # rounded up
    assert np.all(s < 2 * x)                                 # the smallest such power of two
    assert q.min() >= -127 and q.max() <= 127
    deq = q.reshape(N, K // G, G) * s[:, :, None]
    err = np.abs(w.reshape(N, K // G, G).astype(np.float64) - deq)
    assert np.all(err <= s[:, :, None] / 2)
    assert np.abs(q).max(axis=1).min() >= 64                 # each row uses its top half somewhere


def test_scale_words_are_group_major_low_byte_first():
    N, G, groups = 3, 32, 6                                  # 6 groups: two words, the second half full
    K = G * groups
    w = np.zeros((N, K), np.float32)
    e = np.zeros((N, groups), np.int64)
    for n in range(N):
        for g in range(groups):
            e[n, g] = 127 - 5 - g - 2 * n
            w[n, g * G] = np.float32(127.0 * 2.0 ** (e[n, g] - 127))   # amax / 127 is an exact power of two
            w[n, g * G + 1] = -w[n, g * G] / 2
    q, sf = oracle.quantize_weight_mx(w, G)
    assert sf.shape == (2, N) and sf.dtype == np.uint32
    flat = sf.ravel()
    for wi in range(2):
        for n in range(N):
            want = 0
            for b in range(4):
                g = 4 * wi + b
                if g < groups:
                    want |= int(e[n, g]) << (8 * b)
            assert int(flat[wi * N + n]) == want
    assert np.all(q[:, ::G] == 127) and np.all(q[:, 1::G] == -64)     # -63.5 rounds to even


def test_misread_layouts_give_errors_of_the_size_of_the_values():
    N, K, G = 64, 1024, 32
    w = block_weights(N, K, G, seed=3)
    q, sf = oracle.quantize_weight_mx(w, G)

    def rel(s):
        deq = (q.reshape(N, K // G, G) * s[:, :, None]).reshape(N, K)
        return np.linalg.norm(deq - w) / np.linalg.norm(w)

    s = decode_scales(sf, N, K, G)
    good = rel(s)
    # the error of a uniform step: RMS s / sqrt(12) per element
    predicted = np.sqrt(np.sum(np.repeat(s, G, axis=1) ** 2 / 12.0)) / np.linalg.norm(w)
    assert good == pytest.approx(predicted, rel=0.1) and good < 0.02
    swapped = sf.byteswap()                                  # byte order written the other way round
    assert rel(decode_scales(swapped, N, K, G)) > 0.3
    rowmajor = sf.ravel().reshape(N, -1).T                   # row-major index n * words + w
    assert rel(decode_scales(rowmajor, N, K, G)) > 0.3
    coarse = decode_scales(sf, N, K, 128)                    # granularity 128 read from G = 32 words
    assert rel(np.repeat(coarse, 4, axis=1)[:, : K // G]) > 0.3


def test_zero_group_and_saturating_group():
    G = 32
    w = np.zeros((2, 2 * G), np.float32)
    w[1, G:] = np.linspace(-1e6, 1e6, G, dtype=np.float32)
    q, sf = oracle.quantize_weight_mx(w, G)
    assert np.all(q[0] == 0) and np.all(q[1, :G] == 0)
    assert (int(sf[0, 0]) & 0xFF) == 103 and ((int(sf[0, 1]) >> 8) & 0xFF) == 136
    assert q[1, G] == -127 and q[1, -1] == 127               # |w| / 2^9 > 127: the clamp binds


def test_gemm_mx_against_exact_fractions():
    rng = np.random.default_rng(11)
    M, N, G, groups = 3, 4, 32, 3
    K = G * groups
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    e = rng.integers(103, 137, (N, groups))
    e[0] = [136, 103, 120]                                   # 33 binades inside one row
    sf = np.zeros((1, N), np.uint32)
    for n in range(N):
        sf[0, n] = sum(int(e[n, g]) << (8 * g) for g in range(groups))
    t, absum = oracle.gemm_mx(qa, q, sf, G)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            a = 0.0
            for k in range(K):
                p = int(qa[m, k]) * int(q[n, k])
                sc = Fraction(2) ** (int(e[n, k // G]) - 127)
                exact += p * sc
                a += abs(p) * float(sc)
            assert t[m, n] == nearest_f32(exact), (m, n)
            assert absum[m, n] == pytest.approx(a, rel=1e-12)


def test_gemm_mx_rounds_ties_to_even():
    # T = 2^24 + 1 and 2^24 + 3 in units of 1: halfway cases of fp32 (ulp 2 at 2^24)
    G = 32
    qa = np.zeros((2, 2 * G), np.int8)
    q = np.zeros((1, 2 * G), np.int8)
    qa[:, :G], q[0, :G] = 32, 32                             # group 0: 32 * 1024 = 2^15, scale 2^9
    qa[0, G], qa[1, G], q[0, G] = 1, 3, 1                    # group 1: 1 or 3, scale 2^0
    sf = np.array([[136 | (127 << 8)]], np.uint32)
    t, _ = oracle.gemm_mx(qa, q, sf, G)
    assert t[0, 0] == np.float32(2.0 ** 24) and t[1, 0] == np.float32(2.0 ** 24 + 4)


def test_gemm_mx_sums_exactly_before_rounding():
    # 2^24 + 1 + 1: rounding after each group loses both ones (ties to even); the exact sum
    # 2^24 + 2 is an fp32 value
    G = 32
    qa = np.zeros((1, 3 * G), np.int8)
    q = np.zeros((1, 3 * G), np.int8)
    qa[0, :G], q[0, :G] = 32, 32
    qa[0, G], q[0, G], qa[0, 2 * G], q[0, 2 * G] = 1, 1, 1, 1
    sf = np.array([[136 | (127 << 8) | (127 << 16)]], np.uint32)
    t, _ = oracle.gemm_mx(qa, q, sf, G)
    assert t[0, 0] == np.float32(2.0 ** 24 + 2)


def test_codes_round_half_to_even():
    G = 32
    w = np.zeros((1, G), np.float32)
    w[0, :5] = np.array([127.0, 2.5, 3.5, -2.5, 0.5], np.float32) * np.float32(2.0 ** -5)   # s = 2^-5
    q, sf = oracle.quantize_weight_mx(w, G)
    assert int(sf[0, 0]) == 122 and q[0, :5].tolist() == [127, 2, 4, -2, 0]


def test_equal_scales_reduce_to_the_integer_gemm():
    rng = np.random.default_rng(5)
    M, N, K, G = 5, 7, 512, 128
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sf = np.full((1, N), 120 * 0x01010101, np.uint32)         # every group 2^-7
    t, _ = oracle.gemm_mx(qa, q, sf, G)
    acc = qa.astype(np.int64) @ q.astype(np.int64).T          # |acc| < 2^24: exact in fp32
    np.testing.assert_array_equal(t, (acc.astype(np.float32) * np.float32(2.0 ** -7)))


def test_linear_mx_order_and_accuracy():
    M, N, K, G = 16, 96, 2048, 32
    wl = workloads.WORKLOADS["prefill2k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=9)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    bias = workloads.gaussian((N,), 12)
    t, _ = oracle.gemm_mx(qa, q, sf, G)
    y = oracle.linear_mx(qa, sa, q, sf, G, bias=bias)
    np.testing.assert_array_equal(y, (t * sa[:, None]).astype(np.float32) + bias[None, :])
    # block scales follow the weights' magnitude along K: closer to the fp64 product than
    # one scale per output channel
    ref = a.astype(np.float64) @ w.astype(np.float64).T
    qw, sw = oracle.quantize_sym(w, per_row=True)
    y_pc, st = oracle.linear_codes(qa, sa, None, qw, sw, True, True)
    assert st == oracle.OK
    y_mx = oracle.linear_mx(qa, sa, q, sf, G)
    err_mx = np.linalg.norm(y_mx - ref) / np.linalg.norm(ref)
    err_pc = np.linalg.norm(y_pc - ref) / np.linalg.norm(ref)
    assert err_mx < err_pc
