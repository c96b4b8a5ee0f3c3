"""q8_gemm_dequant_ws: the layer with a caller workspace, in which the activation codes are written
once as fp16 numbers of equal value for the CTA-pair kernel to load by TMA. The INT32 sums and the
epilogue are the same operations, so y must equal q8_gemm_dequant's bit for bit, and the oracle's
layer ("100 Days of GPU, Day 98", the epilogue listing; "Activation Quantization Architecture",
the integer GEMM written out) within the usual 2 ulp (0 expected)."""
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


CASES = [
    # name, M, N, K, act_per_row, act_symmetric, w_per_row
    ("prefill2k", 512, 2048, 2048, True, True, True),      # small grid: every tile in K slices
    ("relu4k", 2048, 4096, 4096, True, False, True),       # zero points and column sums; two waves of whole tiles
    ("prefill2k", 333, 520, 1040, True, True, True),       # ragged M, N and K
    ("relu4k", 257, 2052, 1024, False, False, False),      # per-tensor scales, sliced
    ("prefill16k", 1024, 1024, 16384, True, True, True),
    ("prefill2k", 2344, 2056, 2048, True, True, True),     # 90 ragged tiles: the last wave's 14 in 4 K slices
]


@pytest.mark.parametrize("name,M,N,K,apr,sym,wpr", CASES)
def test_workspace_layer_equals_the_direct_layer_and_the_oracle(q8, name, M, N, K, apr, sym, wpr):
    wl = workloads.WORKLOADS[name]
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    ref = oracle.linear(a, w, apr, sym, wpr, threads=8)
    assert ref["status"] == oracle.OK
    qw, s_w = q8.q8_quantize_weight(dev(w), per_row=wpr)
    cs = q8.q8_colsum(qw)
    qa, s_a, z_a = q8.q8_quantize_act(dev(a), per_row=apr, symmetric=sym)
    need = q8.q8_gemm_workspace(M, N, K)
    assert need == 2 * M * K
    ws = torch.full((need,), 0x55, dtype=torch.uint8, device="cuda")   # stale contents are overwritten
    y_direct = q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, cs)
    for _ in range(2):
        y_ws = q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, cs, workspace=ws)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y_ws.cpu().numpy().view(np.int32), y_direct.cpu().numpy().view(np.int32))
    assert int(gates.ulp_distance(y_ws.cpu().numpy(), ref["y"]).max()) <= 2
    # the fp16 copy holds the codes themselves
    np.testing.assert_array_equal(ws.view(torch.float16)[:M * K].view(M, K).cpu().numpy().astype(np.int32),
                                  ref["qa"].astype(np.int32))


def test_workspace_extreme_codes_at_the_largest_k(q8):
    # -128 * -128 on every k: each fp32 chunk sum reaches 2^24 exactly, INT32 sums reach 2^31 - 2^18
    M, N, K = 260, 520, 131056
    qa = np.full((M, K), -128, np.int8)
    qw = np.full((N, K), -128, np.int8)
    qw[1::2] = 127
    sa = np.full(M, 1.0, np.float32)
    sw = np.full(N, 1.0, np.float32)
    ws = torch.empty(q8.q8_gemm_workspace(M, N, K), dtype=torch.uint8, device="cuda")
    y = q8.q8_gemm_dequant(dev(qa), dev(sa), None, dev(qw), dev(sw), workspace=ws).cpu().numpy()
    assert q8.q8_device_error() == 0
    expect = np.where(np.arange(N) % 2 == 0, 16384.0 * K, -128.0 * 127 * K).astype(np.float32)
    np.testing.assert_array_equal(y, np.broadcast_to(expect, (M, N)))


def test_small_or_absent_workspace_takes_the_direct_path(q8):
    M, N, K = 300, 520, 2048
    rng = np.random.default_rng(3)
    qa = dev(rng.integers(-128, 128, (M, K), dtype=np.int8))
    qw = dev(rng.integers(-127, 128, (N, K), dtype=np.int8))
    sa, sw = dev(rng.random(M, dtype=np.float32)), dev(rng.random(N, dtype=np.float32))
    y0 = q8.q8_gemm_dequant(qa, sa, None, qw, sw)
    small = torch.zeros(2 * M * K - 16, dtype=torch.uint8, device="cuda")
    y1 = q8.q8_gemm_dequant(qa, sa, None, qw, sw, workspace=small)
    torch.cuda.synchronize()
    assert int(small.sum()) == 0                             # untouched
    np.testing.assert_array_equal(y0.cpu().numpy().view(np.int32), y1.cpu().numpy().view(np.int32))
    # decode shapes take no workspace
    assert q8.q8_gemm_workspace(16, N, K) == 0


@pytest.mark.parametrize("M,K,per_row,sym", [(300, 4096, True, True), (257, 1040, True, False), (64, 40000, True, True),
                                             (100, 2048, False, True), (33, 64, True, False)])
def test_dual_quantizer_writes_both_code_formats(q8, M, K, per_row, sym):
    # one pass for rows of up to 32768 elements, the quantizer and the copy kernel beyond (K = 40000)
    # and for per-tensor scales: the same codes, scales and zero points as the single-format calls
    wl = workloads.WORKLOADS["relu4k" if not sym else "prefill2k"]
    a = dev(workloads.make_activations(wl, M=M, K=K))
    qa, qa16, s_a, z_a = q8.q8_quantize_act_dual(a, per_row=per_row, symmetric=sym)
    qa_ref, s_ref, z_ref = q8.q8_quantize_act(a, per_row=per_row, symmetric=sym)
    qa16_ref, _, _ = q8.q8_quantize_act_f16(a, per_row=per_row, symmetric=sym)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_ref.cpu().numpy())
    np.testing.assert_array_equal(qa16.view(torch.int16).cpu().numpy(), qa16_ref.view(torch.int16).cpu().numpy())
    np.testing.assert_array_equal(s_a.cpu().numpy().view(np.int32), s_ref.cpu().numpy().view(np.int32))
    if not sym:
        np.testing.assert_array_equal(z_a.cpu().numpy(), z_ref.cpu().numpy())
    ref = oracle.quantize_sym(a.cpu().numpy(), per_row=per_row)[0] if sym else \
        oracle.quantize_asym(a.cpu().numpy(), per_row=per_row)[0]
    np.testing.assert_array_equal(qa16.float().cpu().numpy().astype(np.int32), ref.astype(np.int32))


@pytest.mark.parametrize("name,M,N,K,sym", [("prefill2k", 512, 2048, 2048, True), ("relu4k", 2048, 4096, 4096, False),
                                            ("prefill2k", 333, 520, 1040, True), ("decode", 16, 1024, 4096, True)])
def test_linear_with_workspace_equals_linear(q8, name, M, N, K, sym):
    # the quantizer writes the fp16 copy itself and the pair kernel loads it; the decode shape
    # takes no workspace (q8_linear itself)
    wl = workloads.WORKLOADS[name]
    a = dev(workloads.make_activations(wl, M=M, K=K))
    w = dev(workloads.make_weights(wl, N=N, K=K))
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    cs = None if sym else q8.q8_colsum(qw)
    need = q8.q8_gemm_workspace(M, N, K)
    ws = torch.full((max(need, 16),), 0x55, dtype=torch.uint8, device="cuda")
    y_ref = q8.q8_linear(a, qw, s_w, cs, symmetric=sym)
    qa = torch.empty((M, K), dtype=torch.int8, device="cuda")
    for _ in range(2):
        y = q8.q8_linear(a, qw, s_w, cs, symmetric=sym, qa=qa, workspace=ws)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y.cpu().numpy().view(np.int32), y_ref.cpu().numpy().view(np.int32))
    qa_ref, _, _ = q8.q8_quantize_act(a, symmetric=sym)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_ref.cpu().numpy())
    if need == 0:
        assert bool((ws == 0x55).all())
    else:
        np.testing.assert_array_equal(ws.view(torch.float16)[:M * K].view(M, K).float().cpu().numpy().astype(np.int32),
                                      qa_ref.cpu().numpy().astype(np.int32))
