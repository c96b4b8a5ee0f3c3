"""GPU parity of the epilogue variants (q8_gemm_epilogue_ex) against the oracle.

"Activation Quantization Architecture" (Fusion): the epilogue multiplies by the
per-token and per-channel scales, adds the bias and writes bf16, or quantizes the
output for the next GEMM. Every GEMM kernel takes the same epilogue. The fp32
value before the output conversion follows the oracle's operation order, so it is
expected bit-identical; the bf16 and int8 outputs are then compared exactly where
it is (everywhere, in practice) and within one step elsewhere.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gates

pytestmark = pytest.mark.gpu

KERNELS = ("tcgen05", "tcgen05_pair", "mma_s8", "skinny", "decode", "decode_tc")


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


def layer(M, N, K, sym, seed):
    wl = workloads.WORKLOADS["prefill2k" if sym else "relu4k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    if sym:
        qa, sa = oracle.quantize_sym(a, per_row=True)
        za = None
    else:
        qa, sa, za = oracle.quantize_asym(a, per_row=True)
    qw, sw = oracle.quantize_sym(w, per_row=True)
    cs = oracle.colsum(qw).astype(np.int32)
    bias = workloads.gaussian((N,), seed) * np.float32(0.5)
    return qa, sa, za, qw, sw, cs, bias


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("sym", [True, False])
def test_epilogue_variants_match_oracle(q8, kernel, sym):
    M, N, K = (16, 520, 2064) if kernel.startswith("decode") else (200, 264, 1088)
    qa, sa, za, qw, sw, cs, bias = layer(M, N, K, sym, seed=31)
    d = dict(qa=dev(qa), s_a=dev(sa), z_a=None if za is None else dev(za), qw=dev(qw), s_w=dev(sw),
             colsum=dev(cs), kernel=kernel)
    y_ref, st = oracle.linear_codes_bias(qa, sa, za, qw, sw, bias, True, True)
    assert st == oracle.OK
    y0_ref, _ = oracle.linear_codes_bias(qa, sa, za, qw, sw, None, True, True)

    y = host(q8.q8_gemm_epilogue(bias=dev(bias), **d))
    assert q8.q8_device_error() == 0
    assert int(gates.ulp_distance(y, y_ref).max()) <= 2
    exact = y.view(np.int32) == y_ref.view(np.int32)
    assert exact.mean() > 0.999

    yb = host(q8.q8_gemm_epilogue(bias=dev(bias), out_dtype=torch.bfloat16, **d).view(torch.int16)).view(np.uint16)
    want = oracle.to_bf16(y_ref)
    np.testing.assert_array_equal(yb[exact], want[exact])
    assert np.abs(yb.astype(np.int32) - want.astype(np.int32)).max() <= 1

    yb0 = host(q8.q8_gemm_epilogue(out_dtype=torch.bfloat16, **d).view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(yb0, oracle.to_bf16(y0_ref))

    s_out = float(np.float32(np.abs(y_ref).max() / np.float32(127.0)))
    yq = host(q8.q8_gemm_epilogue(bias=dev(bias), out_dtype=torch.int8, out_scale=s_out, **d))
    wq = oracle.quantize_static(y_ref, s_out)
    np.testing.assert_array_equal(yq[exact], wq[exact])
    assert np.abs(yq.astype(np.int32) - wq.astype(np.int32)).max() <= 1


def test_bf16_ties_through_the_epilogue(q8):
    # unit scales, codes chosen so that acc + bias lands on bf16 ties: 257 = 256 + 1 is a tie
    # between 256 and 258 in bf16 (8 significant bits): round to even (256); 259 -> 260
    K = 16
    qa = np.zeros((2, K), np.int8)
    qa[0, 0], qa[1, 0] = 1, 1
    qw = np.zeros((2, K), np.int8)
    qw[0, 0], qw[1, 0] = 1, 3
    bias = np.array([256.0, 256.0], np.float32)
    out = q8.q8_gemm_epilogue(dev(qa), dev(np.ones(2, np.float32)), None, dev(qw), dev(np.ones(2, np.float32)),
                              bias=dev(bias), out_dtype=torch.bfloat16, kernel="mma_s8")
    got = host(out.float())
    assert got.tolist() == [[256.0, 260.0], [256.0, 260.0]]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.int8])
def test_k_zero_gives_the_bias(q8, out_dtype):
    M, N = 3, 8
    bias = workloads.gaussian((N,), 40)
    z = torch.empty((M, 0), dtype=torch.int8, device="cuda")
    w = torch.empty((N, 0), dtype=torch.int8, device="cuda")
    out = q8.q8_gemm_epilogue(z, torch.ones(M, device="cuda"), None, w, torch.ones(N, device="cuda"),
                              bias=dev(bias), out_dtype=out_dtype, out_scale=0.05)
    y = np.broadcast_to(bias, (M, N)).astype(np.float32)
    if out_dtype == torch.float32:
        np.testing.assert_array_equal(host(out), y)
    elif out_dtype == torch.bfloat16:
        np.testing.assert_array_equal(host(out.view(torch.int16)).view(np.uint16), oracle.to_bf16(y))
    else:
        np.testing.assert_array_equal(host(out), oracle.quantize_static(y, 0.05))


@pytest.mark.parametrize("M,N,K", [(200, 272, 1088), (513, 520, 2064)])
def test_pair_kernel_tma_epilogue_every_output_type(q8, M, N, K):
    # N = 272: bf16 and int8 rows are whole 16-byte multiples, so all three output types take
    # the TMA-store epilogue of the pair kernel; N = 520 leaves int8 on the direct stores
    qa, sa, za, qw, sw, cs, bias = layer(M, N, K, True, seed=33)
    d = dict(qa=dev(qa), s_a=dev(sa), z_a=None, qw=dev(qw), s_w=dev(sw), kernel="tcgen05_pair")
    y_ref, _ = oracle.linear_codes_bias(qa, sa, None, qw, sw, bias, True, True)
    y = host(q8.q8_gemm_epilogue(bias=dev(bias), **d))
    np.testing.assert_array_equal(y.view(np.int32), y_ref.view(np.int32))
    yb = host(q8.q8_gemm_epilogue(bias=dev(bias), out_dtype=torch.bfloat16, **d).view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(yb, oracle.to_bf16(y_ref))
    s_out = float(np.float32(np.abs(y_ref).max() / np.float32(100.0)))   # some codes clamp at +-127
    yq = host(q8.q8_gemm_epilogue(bias=dev(bias), out_dtype=torch.int8, out_scale=s_out, **d))
    np.testing.assert_array_equal(yq, oracle.quantize_static(y_ref, s_out))
    assert q8.q8_device_error() == 0
