"""Launch ordering of the decode kernels (programmatic dependent launch).

The decode kernels may start while the kernel before them on the stream is still running.
A standalone GEMM call waits for that kernel before it reads any operand, so weights that
the kernel just before writes are seen in full: here a weight quantizer rewrites the weight
buffers right before each decode GEMM, on the same stream, with no synchronisation between.
q8_linear (activation quantizer + GEMM in one call) lets the weight stream start while its
own quantizer runs; its results must equal the oracle's layer as well.
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


def ulp_max(got, ref):
    return int(gates.ulp_distance(got, ref).max())


WL = workloads.WORKLOADS["decode"]
M, N, K = 16, 4096, 8192


def test_weight_quantizer_right_before_decode_gemm(q8):
    a = workloads.make_activations(WL, M=M, K=K)
    w_old = workloads.make_weights(WL, N=N, K=K)
    w_new = -np.flip(w_old, axis=1).copy() * np.float32(0.5)     # every code and scale changes
    qa, s_a, _ = q8.q8_quantize_act(dev(a))
    w_old_d, w_new_d = dev(w_old), dev(w_new)
    qw, s_w = q8.q8_quantize_weight(w_old_d, per_row=True)
    ref = oracle.linear(a, w_new, act_per_row=True, act_symmetric=True, w_per_row=True)
    torch.cuda.synchronize()
    for _ in range(3):
        q8.q8_quantize_weight(w_old_d, per_row=True, qw=qw, s_w=s_w)   # stale contents first
        q8.q8_quantize_weight(w_new_d, per_row=True, qw=qw, s_w=s_w)   # then the weights the GEMM must see
        y = q8.q8_gemm_dequant(qa, s_a, None, qw, s_w)                  # decode kernel, right after
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        assert ulp_max(y.cpu().numpy(), ref["y"]) <= 2


def test_int4_and_block_scaled_weights_right_before_decode_gemm(q8):
    a = workloads.make_activations(WL, M=M, K=K)
    w_old = workloads.make_weights(WL, N=N, K=K)
    w_new = -np.flip(w_old, axis=1).copy() * np.float32(0.5)
    qa, s_a, _ = q8.q8_quantize_act(dev(a))
    w_old_d, w_new_d = dev(w_old), dev(w_new)
    # int4 weights
    qw4, s4 = q8.q8_quantize_weight_int4(w_old_d)
    q8.q8_quantize_weight_int4(w_new_d, qw4=qw4, s_w=s4)
    y4 = q8.q8_gemm_w4a8(qa, s_a, None, qw4, s4)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    ref4 = q8.q8_gemm_w4a8(qa, s_a, None, q8.q8_quantize_weight_int4(w_new_d)[0], s4)   # fresh buffers
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y4.cpu().numpy().view(np.int32), ref4.cpu().numpy().view(np.int32))
    # block-scaled weights (scale words are read before the wait too)
    qwm, sf = q8.q8_quantize_weight_mx(w_old_d, 32)
    q8.q8_quantize_weight_mx(w_new_d, 32, qw=qwm, sf=sf)
    ym = q8.q8_gemm_mx(qa, s_a, qwm, sf, 32)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    qwm2, sf2 = q8.q8_quantize_weight_mx(w_new_d, 32)
    ym2 = q8.q8_gemm_mx(qa, s_a, qwm2, sf2, 32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ym.cpu().numpy().view(np.int32), ym2.cpu().numpy().view(np.int32))


@pytest.mark.parametrize("Mx,per_row,symmetric", [(16, True, True), (9, True, False), (16, False, True),
                                                 (300, True, True), (260, True, False)])
def test_q8_linear_matches_oracle(q8, Mx, per_row, symmetric):
    wl = workloads.WORKLOADS["decode" if Mx <= 16 else "relu4k"]
    Nx, Kx = 1040, 4096
    a = workloads.make_activations(wl, M=Mx, K=Kx)
    w = workloads.make_weights(wl, N=Nx, K=Kx)
    ref = oracle.linear(a, w, act_per_row=per_row, act_symmetric=symmetric, w_per_row=True)
    qw, s_w = q8.q8_quantize_weight(dev(w), per_row=True)
    colsum = q8.q8_colsum(qw)
    a_d = dev(a)
    for _ in range(2):
        y = q8.q8_linear(a_d, qw, s_w, colsum, per_row=per_row, symmetric=symmetric)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        assert ulp_max(y.cpu().numpy(), ref["y"]) <= 2


def test_q8_linear_rejects_before_enqueueing(q8):
    a = torch.zeros((16, 64), dtype=torch.float32, device="cuda")
    qw = torch.zeros((32, 64), dtype=torch.int8, device="cuda")
    s_w = torch.ones(32, device="cuda")
    qa = torch.full((16, 64), 7, dtype=torch.int8, device="cuda")
    s_a = torch.empty(16, device="cuda")
    z_a = torch.empty(16, dtype=torch.int32, device="cuda")
    y = torch.empty((16, 32), device="cuda")
    # asymmetric activations without column sums: the GEMM half is invalid, so neither half runs
    st = q8.load().q8_linear(q8._ptr(a), 16, 64, q8.Q8_PER_ROW, q8.Q8_ASYMMETRIC, q8._ptr(qa), q8._ptr(s_a),
                             q8._ptr(z_a), q8._ptr(qw), q8._ptr(s_w), q8.Q8_PER_ROW, None, 32, q8._ptr(y), None)
    assert st == q8.Q8_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int((qa != 7).sum()) == 0          # the quantizer half did not run
