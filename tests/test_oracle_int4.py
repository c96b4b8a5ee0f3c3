"""Pins of the oracle's int4 weights for W4A8 (CPU only).

TileLang tutorial ch. 27 (low-precision quantization): 2.4 int8 / int4 gives the
symmetric rule with qmax = 7 (s = absmax / 7, q = clip(round(x / s), -8, 7), error
bound 1 / (2 qmax) = 7.143e-2 of absmax); its int4 GEMM example packs two codes per
byte as (a & 0x0F) | ((b & 0x0F) << 4) and decodes by an arithmetic shift, warning
that a logical shift turns -1 into 15.
"""
import numpy as np

import oracle
import workloads


def test_packing_follows_the_pages():
    packed = oracle.pack_int4(np.array([[-8, -1, 0, 7, -1, -1]], np.int8))
    assert packed[0].tolist() == [0xF8, 0x70, 0xFF]
    assert oracle.unpack_int4(np.array([[0xFF]], np.uint8), 2).tolist() == [[-1, -1]]   # not 15


def test_pack_unpack_round_trip_every_byte():
    lo, hi = np.meshgrid(np.arange(-8, 8, dtype=np.int8), np.arange(-8, 8, dtype=np.int8))
    q = np.stack([lo.ravel(), hi.ravel()], axis=1).reshape(1, -1).astype(np.int8)     # all 256 code pairs
    packed = oracle.pack_int4(q)
    assert sorted(packed[0].tolist()) == list(range(256))
    np.testing.assert_array_equal(oracle.unpack_int4(packed, q.shape[1]), q)


def test_error_bound_is_one_fourteenth_of_absmax():
    w = workloads.gaussian((64, 4096), 23)
    q, s = oracle.quantize_int4(w)
    err = np.abs(w - q.astype(np.float32) * s[:, None]) / np.abs(w).max(axis=1, keepdims=True)
    assert err.max() <= 1.0 / 14.0 * (1 + 1e-6)
    assert err.max() > 0.07                                   # the bound is reached: 7.143e-2
    rms = np.sqrt(np.mean((w - q.astype(np.float32) * s[:, None]) ** 2, axis=1))
    np.testing.assert_allclose(rms / (s / np.sqrt(12.0)), 1.0, rtol=0.05)


def test_integer_grid_and_ties():
    w = np.array([[-7, -3, 0, 1, 7, 2, -6, 5]], np.float32)
    q, s = oracle.quantize_int4(w)
    assert s[0] == 1.0 and q[0].tolist() == w[0].astype(int).tolist()
    q, s = oracle.quantize_int4(np.array([[7.0, 2.5, 3.5, -2.5, -3.5, 0.5]], np.float32))
    assert q[0].tolist() == [7, 2, 4, -2, -4, 0]


def test_w4a8_products_brute_force_and_bound():
    rng = np.random.default_rng(24)
    qa = rng.integers(-128, 128, (3, 40), dtype=np.int8)
    q4 = rng.integers(-8, 8, (5, 40), dtype=np.int8)
    w4 = oracle.unpack_int4(oracle.pack_int4(q4), 40)
    acc = oracle.gemm_acc(qa, w4)
    want = [[sum(int(qa[m, k]) * int(q4[n, k]) for k in range(40)) for n in range(5)] for m in range(3)]
    assert acc.tolist() == want
    # worst case: -128 * -8 on every k reaches K * 1024
    K = 2048
    worst = oracle.gemm_acc(np.full((1, K), -128, np.int8), np.full((1, K), -8, np.int8))
    assert worst[0, 0] == K * 1024
