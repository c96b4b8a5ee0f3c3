"""Pins of the oracle's epilogue variants (CPU only).

"Activation Quantization Architecture" (Fusion): after the int32 accumulation the
epilogue multiplies by the per-token and per-channel scales, adds the bias and
writes bf16; some kernels quantize the output for the next GEMM directly. The
oracle's reading: y = fl((float)corr * (s_a * s_w)) + bias[n] in fp32, then fp32,
bf16 (round to nearest even) or int8 codes with a static output scale.
"""
import numpy as np
import torch

import oracle
import workloads


def test_bf16_rounding_ties_and_exact_values():
    y = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -2.5, 0.0, -0.0, 3.0e38,
                  2 ** -126, 65280.0], np.float32)
    got = oracle.to_bf16(y).tolist()
    assert got[0] == 0x3F80                      # exact
    assert got[1] == 0x3F80                      # tie between 1 and 1 + 2^-7: to even (1)
    assert got[2] == 0x3F82                      # tie between 1 + 2^-7 and 1 + 2^-6: to even
    assert got[3] == 0x3F81                      # just above the tie: up
    assert got[4] == 0xC020 and got[5] == 0x0000 and got[6] == 0x8000
    assert got[8] == 0x0080                      # smallest normal
    assert got[9] == 0x477F                      # 65280 = 255 * 256, exact in bf16


def test_bf16_matches_torch_conversion():
    y = workloads.gaussian((4096,), 21) * np.float32(37.0)
    want = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.to_bf16(y), want)


def test_static_quantizer_rounds_half_even_and_clamps():
    y = np.array([2.5, 3.5, -2.5, 0.5, 126.5, 400.0, -400.0, 0.3], np.float32)
    q = oracle.quantize_static(y, 1.0)
    assert q[:7].tolist() == [2, 4, -2, 0, 126, 127, -127]
    # the pages' outlier example: s = 60 / 127, 0.3 -> code 1
    assert oracle.quantize_static(np.array([0.3], np.float32), np.float32(60.0) / np.float32(127.0))[0] == 1
    # a value where the fp32 quotient rounds to -60.0 (a code) but y * fl(1 / s) lands past -60.5
    y, s_out = np.float32(-114.78968811035156), np.float32(1.8973501920700073)
    assert np.rint(np.float32(y / s_out)) == -60 and np.rint(y * (np.float32(1.0) / s_out)) == -61
    assert oracle.quantize_static(np.array([y], np.float32), s_out)[0] == -60


def _codes(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = (0.01 + rng.random(M)).astype(np.float32)
    sw = (0.001 + rng.random(N) * 0.01).astype(np.float32)
    return qa, qw, sa, sw


def test_bias_is_added_after_the_scales():
    qa, qw, sa, sw = _codes(5, 12, 64, 3)
    bias = workloads.gaussian((12,), 22)
    qa[2] = 0                                     # a zero row: corr = 0, so y = bias exactly
    y0, st0 = oracle.linear_codes(qa, sa, None, qw, sw, True, True)
    yb, st1 = oracle.linear_codes_bias(qa, sa, None, qw, sw, bias, True, True)
    assert st0 == oracle.OK and st1 == oracle.OK
    np.testing.assert_array_equal(yb[2], bias)
    np.testing.assert_array_equal(yb, (y0 + bias[None, :]).astype(np.float32))
    yz, _ = oracle.linear_codes_bias(qa, sa, None, qw, sw, np.zeros(12, np.float32), True, True)
    np.testing.assert_array_equal(yz, y0)
    yn, _ = oracle.linear_codes_bias(qa, sa, None, qw, sw, None, True, True)
    np.testing.assert_array_equal(yn, y0)


def test_bias_brute_force_small_integers():
    # unit scales: y = acc + bias exactly for small integers; bias is indexed by the output channel
    qa = np.array([[1, 2, 3, 0] * 4, [-1, 0, 2, 5] * 4], np.int8)
    qw = np.array([[1, 0, -1, 2] * 4, [3, 1, 1, 1] * 4, [0, 0, 0, 1] * 4], np.int8)
    acc = qa.astype(np.int64) @ qw.astype(np.int64).T
    bias = np.array([10.0, -3.0, 0.5], np.float32)
    y, st = oracle.linear_codes_bias(qa, np.ones(2, np.float32), None, qw, np.ones(3, np.float32), bias,
                                     True, True)
    assert st == oracle.OK
    np.testing.assert_array_equal(y, (acc + bias[None, :]).astype(np.float32))
