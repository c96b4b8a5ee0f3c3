"""GPU parity of the fp16-code path: activation codes written as fp16 values
(q8_quantize_act_f16) and the CTA-pair GEMM that loads them by TMA straight into
its operand stages (q8_gemm_f16a_ex / q8_gemm_f16a_s32).

The codes must equal the oracle's int8 codes value for value, and the INT32
accumulators and the epilogue outputs must be bit-identical to the oracle's (the
int8-code path's outputs where the oracle has no counterpart), on shapes that
span several tiles, ragged M / N / K tails, the K-split grids and the largest K.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

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


def codes16(qa: np.ndarray) -> torch.Tensor:
    """int8 codes as the fp16 values of the same numbers, on the device."""
    return dev(qa.astype(np.float16))


def as_codes(qa16: torch.Tensor) -> np.ndarray:
    """fp16 code values back to int8, checking that every one is an integer in [-128, 127]."""
    v = host(qa16).astype(np.float32)
    assert np.all(v == np.rint(v)) and v.min() >= -128 and v.max() <= 127
    return v.astype(np.int8)


def no_device_error(q8):
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0


QUANT_CASES = [
    # (M, K, per_row, symmetric, maker)
    (16, 256, False, True, "tiny"),
    (512, 2048, True, True, "prefill2k"),
    (2048, 4096, True, False, "relu4k"),
    (16, 8192, True, True, "decode"),
    (64, 16384, True, True, "prefill16k"),
    (37, 528, True, False, "prefill2k"),
    (5, 40000, True, True, "prefill2k"),       # rows longer than the register budget
    (3, 40000, True, False, "relu4k"),
    (300, 48, False, False, "relu4k"),         # per-tensor asymmetric
    (7, 1040, False, True, "prefill2k"),
]


@pytest.mark.parametrize("M,K,per_row,sym,name", QUANT_CASES)
def test_fp16_codes_equal_the_oracle_codes(q8, M, K, per_row, sym, name):
    a = workloads.make_activations(workloads.WORKLOADS[name], M=M, K=K)
    a[M // 2] = 0.0
    qa16, s_a, z_a = q8.q8_quantize_act_f16(dev(a), per_row=per_row, symmetric=sym)
    no_device_error(q8)
    if sym:
        rq, rs = oracle.quantize_sym(a, per_row)
        rz = None
    else:
        rq, rs, rz = oracle.quantize_asym(a, per_row)
    np.testing.assert_array_equal(as_codes(qa16), rq)
    np.testing.assert_array_equal(host(s_a), rs)
    if rz is not None:
        np.testing.assert_array_equal(host(z_a), rz)


# (M, N, K): one tile; ragged M / N / K tails; grids whose pair kernel splits K (2 to 8 slices);
# a grid with a partial last wave; M = 1.
GEMM_CASES = [(256, 256, 64), (300, 520, 4096), (512, 2048, 2048), (257, 2052, 1024), (16, 1024, 8192),
              (1000, 1000, 1040), (1, 16, 16), (777, 384, 3088), (2304, 2560, 1024)]


@pytest.mark.parametrize("M,N,K", GEMM_CASES)
def test_gemm_s32_bit_exact(q8, M, N, K):
    rng = np.random.default_rng(3 * M + 5 * N + K)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-128, 128, (N, K), dtype=np.int8)
    acc = host(q8.q8_gemm_f16a_s32(codes16(qa), dev(qw))).astype(np.int64)
    no_device_error(q8)
    np.testing.assert_array_equal(acc, oracle.gemm_acc(qa, qw, threads=8))


def test_largest_k_extreme_codes(q8):
    """K = 131056: -128 * -128 on every k takes the INT32 sum to 2^31 - 2^18 through 128 exact
    fp32 chunks; other rows mix +127 and random codes."""
    M, N, K = 130, 260, 131056
    rng = np.random.default_rng(23)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-128, 128, (N, K), dtype=np.int8)
    qa[0] = -128
    qw[0] = -128
    qw[1] = 127
    acc = host(q8.q8_gemm_f16a_s32(codes16(qa), dev(qw))).astype(np.int64)
    no_device_error(q8)
    want = oracle.gemm_acc(qa, qw, threads=8)
    assert want[0, 0] == 16384 * K and want[0, 1] == -128 * 127 * K
    np.testing.assert_array_equal(acc, want)


@pytest.mark.parametrize("M,N,K", [(300, 520, 4096), (512, 2048, 2048), (1000, 1000, 1040)])
@pytest.mark.parametrize("apr,wpr", [(True, True), (False, False), (True, False)])
def test_layer_matches_oracle(q8, M, N, K, apr, wpr):
    """Asymmetric activations (zero points and weight column sums), per-row or per-tensor
    scales: y bit-identical to the oracle, with and without a bias."""
    rng = np.random.default_rng(M + 7 * N + K + 2 * apr + wpr)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = (rng.random(M if apr else 1, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    sw = (rng.random(N if wpr else 1, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    za = rng.integers(-128, 128, M if apr else 1, dtype=np.int32)
    cs = q8.q8_colsum(dev(qw))
    y = host(q8.q8_gemm_f16a(codes16(qa), dev(sa), dev(za), dev(qw), dev(sw), cs))
    no_device_error(q8)
    y_ref, st = oracle.linear_codes(qa, sa, za, qw, sw, apr, wpr, threads=8)
    assert st == oracle.OK
    np.testing.assert_array_equal(y.view(np.int32), y_ref.view(np.int32))
    bias = rng.standard_normal(N, dtype=np.float32)
    yb = host(q8.q8_gemm_f16a(codes16(qa), dev(sa), dev(za), dev(qw), dev(sw), cs, bias=dev(bias)))
    no_device_error(q8)
    yb_ref, st = oracle.linear_codes_bias(qa, sa, za, qw, sw, bias, apr, wpr, threads=8)
    np.testing.assert_array_equal(yb.view(np.int32), yb_ref.view(np.int32))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.int8])
def test_output_types_match_the_int8_code_path(q8, out_dtype):
    """bf16 and int8 outputs (with a bias) equal those of q8_gemm_epilogue on the int8 codes,
    whose outputs the epilogue tests pin to the oracle."""
    M, N, K = 600, 768, 2048
    rng = np.random.default_rng(41)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = (rng.random(M, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-3)
    sw = (rng.random(N, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-3)
    bias = rng.standard_normal(N, dtype=np.float32)
    scale = 0.05 if out_dtype == torch.int8 else None
    args = (dev(sa), None, dev(qw), dev(sw))
    y16 = q8.q8_gemm_f16a(codes16(qa), *args, bias=dev(bias), out_dtype=out_dtype, out_scale=scale)
    y8 = q8.q8_gemm_epilogue(dev(qa), *args, bias=dev(bias), out_dtype=out_dtype, out_scale=scale,
                             kernel="tcgen05_pair")
    no_device_error(q8)
    assert torch.equal(y16.view(torch.int16) if out_dtype == torch.bfloat16 else y16,
                       y8.view(torch.int16) if out_dtype == torch.bfloat16 else y8)


def test_empty_and_zero_k(q8):
    qw = torch.zeros((8, 0), dtype=torch.int8, device="cuda")
    qa16 = torch.zeros((4, 0), dtype=torch.float16, device="cuda")
    s = torch.ones(4, dtype=torch.float32, device="cuda")
    y = q8.q8_gemm_f16a(qa16, s, None, qw, torch.ones(8, dtype=torch.float32, device="cuda"))
    no_device_error(q8)
    assert torch.all(y == 0).item()
    empty = q8.q8_gemm_f16a_s32(torch.zeros((0, 32), dtype=torch.float16, device="cuda"),
                                torch.zeros((8, 32), dtype=torch.int8, device="cuda"))
    assert empty.shape == (0, 8)


@pytest.mark.slow
def test_full_size_prefill_layer(q8):
    """The 8192 x 16384 x 8192 layer through the fp16-code path: every code and scale bit-exact,
    y and the INT32 accumulators on sampled outputs against the oracle."""
    wl = workloads.WORKLOADS["prefill16k"]
    a = workloads.make_activations(wl)
    w = workloads.make_weights(wl)
    rqa, rsa = oracle.quantize_sym(a, True)
    rqw, rsw = oracle.quantize_sym(w, True)
    a_d, w_d = dev(a), dev(w)
    del a, w
    qw, s_w = q8.q8_quantize_weight(w_d, per_row=True)
    del w_d
    qa16, s_a, _ = q8.q8_quantize_act_f16(a_d, per_row=True, symmetric=True)
    del a_d
    y = q8.q8_gemm_f16a(qa16, s_a, None, qw, s_w)
    acc = q8.q8_gemm_f16a_s32(qa16, qw)
    no_device_error(q8)
    np.testing.assert_array_equal(host(s_a), rsa)
    np.testing.assert_array_equal(as_codes(qa16), rqa)
    np.testing.assert_array_equal(host(qw), rqw)
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    ms = np.concatenate([rng.integers(0, wl.M, 3000), [0, wl.M - 1, 127, 128, 255, 256]]).astype(np.int64)
    ns = np.concatenate([rng.integers(0, wl.N, 3000), [wl.N - 1, 0, 255, 256, 511, 512]]).astype(np.int64)
    ry, racc, st = oracle.linear_codes_at(rqa, rsa, None, rqw, rsw, ms, ns, True, True)
    assert st == oracle.OK
    mt, nt = torch.as_tensor(ms).cuda(), torch.as_tensor(ns).cuda()
    np.testing.assert_array_equal(host(acc[mt, nt]).astype(np.int64), racc)
    np.testing.assert_array_equal(host(y[mt, nt]).view(np.int32), ry.view(np.int32))


@pytest.mark.slow
def test_full_size_worst_case_codes(q8):
    """Every activation code -128 and every weight code -127 at 8192 x 16384 x 8192: each
    accumulator is K * 16256."""
    wl = workloads.WORKLOADS["prefill16k"]
    qa16 = torch.full((wl.M, wl.K), -128.0, dtype=torch.float16, device="cuda")
    qw = torch.full((wl.N, wl.K), -127, dtype=torch.int8, device="cuda")
    acc = q8.q8_gemm_f16a_s32(qa16, qw)
    no_device_error(q8)
    assert torch.all(acc == wl.K * 16256).item()
