"""GPU parity of the W4A8 path (int8 activations x packed int4 weights) against the oracle.

TileLang tutorial ch. 27 (low-precision quantization): 2.4 int8 / int4 (qmax = 7) and
the int4 GEMM example (two codes per byte, low nibble first, sign-extended on decode,
exact integer accumulation). Codes, scales, column sums and INT32 accumulators must be
bit-identical; y within 2 ulp (0 expected: the epilogue follows the oracle's order).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gates

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import int8_quantized_gemm_gb300 as q8mod
    from int8_quantized_gemm_gb300 import build
    build.build()
    q8mod.load()
    return q8mod


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("N,K", [(64, 32), (1000, 4128), (300, 8192), (17, 40000)])
def test_quantize_int4_and_colsum_bit_exact(q8, N, K):
    w = workloads.make_weights(workloads.WORKLOADS["decode"], N=N, K=K)
    w[N // 2] = 0.0                                        # an all-zero channel
    qw4, s_w = q8.q8_quantize_weight_int4(dev(w))
    cs = q8.q8_colsum_int4(qw4, K)
    q, s = oracle.quantize_int4(w)
    np.testing.assert_array_equal(host(s_w), s)
    np.testing.assert_array_equal(host(qw4), oracle.pack_int4(q))
    np.testing.assert_array_equal(host(cs).astype(np.int64), oracle.colsum(q))


DECODE_CASES = [(16, 520, 2080), (1, 64, 32), (7, 1000, 4128), (16, 4096, 8192), (12, 200, 256)]


@pytest.mark.parametrize("M,N,K", DECODE_CASES)
def test_decode_w4a8_accumulators_bit_exact(q8, M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
    q4[0, :] = -8                                          # worst-case magnitudes in one row
    qa[0, :] = -128
    acc = q8.q8_gemm_w4a8_s32(dev(qa), dev(oracle.pack_int4(q4)), kernel="decode")
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(host(acc).astype(np.int64), oracle.gemm_acc(qa, q4, threads=8))


@pytest.mark.parametrize("kernel", ["decode", "tcgen05_pair"])
def test_w4a8_largest_products_at_the_largest_k(q8, kernel):
    # |a (n + 8)| and |a n| at their maxima on every k, at the largest K the API takes: the
    # decode kernel's fp32 partials reach their bound here
    M, N, K = (16, 72, 131040) if kernel == "decode" else (256, 256, 65536)
    rng = np.random.default_rng(K)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
    qa[0, :], qa[1, :], qa[2, :] = -128, 127, -128
    q4[0, :], q4[1, :], q4[2, :] = 7, -8, -8
    acc = q8.q8_gemm_w4a8_s32(dev(qa), dev(oracle.pack_int4(q4)), kernel=kernel)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    want = oracle.gemm_acc(qa, q4, threads=8)
    assert want[0, 0] == -128 * 7 * K and want[2, 2] == 1024 * K
    np.testing.assert_array_equal(host(acc).astype(np.int64), want)


@pytest.mark.parametrize("sym", [True, False])
def test_decode_w4a8_layer_matches_oracle(q8, sym):
    wl = workloads.WORKLOADS["decode"]
    M, N, K = 16, 1024, 8192
    a = workloads.make_activations(wl, M=M, K=K)
    if not sym:
        a = np.maximum(a, 0.0)
    w = workloads.make_weights(wl, N=N, K=K)
    q4, s4 = oracle.quantize_int4(w)
    qw4 = dev(oracle.pack_int4(q4))
    if sym:
        qa, sa = oracle.quantize_sym(a, per_row=True)
        za, cs = None, None
    else:
        qa, sa, za = oracle.quantize_asym(a, per_row=True)
        cs = dev(oracle.colsum(q4).astype(np.int32))
    y = q8.q8_gemm_w4a8(dev(qa), dev(sa), None if za is None else dev(za), qw4, dev(s4), colsum=cs)
    ref, st = oracle.linear_codes(qa, sa, za, q4, s4, True, True, threads=8)
    assert st == oracle.OK
    assert int(gates.ulp_distance(host(y), ref).max()) <= 2
    yb = q8.q8_gemm_w4a8(dev(qa), dev(sa), None if za is None else dev(za), qw4, dev(s4), colsum=cs,
                         out_dtype=torch.bfloat16)
    np.testing.assert_array_equal(host(yb.view(torch.int16)).view(np.uint16), oracle.to_bf16(host(y)))


PAIR_CASES = [(200, 264, 1088), (513, 777, 3104), (2048, 2048, 4096), (256, 256, 32)]


@pytest.mark.parametrize("M,N,K", PAIR_CASES)
def test_pair_w4a8_accumulators_bit_exact(q8, M, N, K):
    rng = np.random.default_rng(M + N * 3)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
    qa[1, :] = -128
    q4[1, :] = -8
    acc = q8.q8_gemm_w4a8_s32(dev(qa), dev(oracle.pack_int4(q4)), kernel="tcgen05_pair")
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(host(acc).astype(np.int64), oracle.gemm_acc(qa, q4, threads=8))
