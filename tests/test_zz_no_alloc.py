"""The allocation-free host-buffer layer (q8_linear_host_static), called through the C ABI.

Some callers cannot allocate device memory themselves: a plugin whose host application
owns every device byte through its own pool, or a latency-critical path where cudaMalloc
and cudaFree (which can synchronize the device) are not allowed. For them the library
runs q8_linear_host on a fixed device array of its own. This file is collected last, so
that a run stopping at the first failure has run every other test first; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import int8_quantized_gemm_gb300 as q8mod
    from int8_quantized_gemm_gb300 import build
    build.build()
    lib = q8mod.load()
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.q8_linear_host_static.argtypes = [p, i64, i64, i32, p, p, i32, p, i64, p, i64, p]
    lib.q8_linear_host_static.restype = i32
    lib.q8_linear_host_static_limit.argtypes = []
    lib.q8_linear_host_static_limit.restype = ctypes.c_size_t
    return q8mod


def call_static(q8, a_host, qw, s_w, y_host, chunk_rows=0, colsum=None):
    """Symmetric activations, or asymmetric ones (zero point per token) when colsum is given."""
    M, K = a_host.shape
    N = qw.shape[0]
    return q8.load().q8_linear_host_static(
        ctypes.c_void_p(a_host.data_ptr()), M, K, q8.Q8_SYMMETRIC if colsum is None else q8.Q8_ASYMMETRIC,
        ctypes.c_void_p(qw.data_ptr()), ctypes.c_void_p(s_w.data_ptr()), q8.Q8_PER_ROW,
        None if colsum is None else ctypes.c_void_p(colsum.data_ptr()), N, ctypes.c_void_p(y_host.data_ptr()),
        chunk_rows, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_workspace_matches_the_caller_workspace_on_two_calls_in_a_row(q8):
    # 1536 tokens x 4096 -> 2048 channels: the two slots need more than the 64 MiB array for
    # one slice of all rows, so the call cuts the tokens into several slices itself
    M, N, K = 1536, 2048, 4096
    assert q8.q8_linear_host_workspace(M, N, K, M) > q8.load().q8_linear_host_static_limit()
    wl = workloads.WORKLOADS["prefill2k"]
    w = torch.from_numpy(workloads.make_weights(wl, N=N, K=K)).cuda()
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    for call in range(2):
        a = torch.empty((M, K), dtype=torch.float32, pin_memory=True)
        a.copy_(torch.from_numpy(workloads.make_activations(wl, M=M, K=K) * np.float32(1 + call)))
        y_static = torch.full((M, N), float("nan"), dtype=torch.float32, pin_memory=True)
        assert call_static(q8, a, qw, s_w, y_static) == q8.Q8_OK
        y_ref = q8.q8_linear_host(a, qw, s_w, None)             # the entry point with a caller workspace
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y_static.numpy().view(np.int32), y_ref.numpy().view(np.int32))


def test_static_workspace_with_asymmetric_activations(q8):
    # zero points and column sums: the z_a slots of the array are used too
    M, N, K = 1000, 1536, 4096
    wl = workloads.WORKLOADS["relu4k"]
    w = torch.from_numpy(workloads.make_weights(wl, N=N, K=K)).cuda()
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    colsum = q8.q8_colsum(qw)
    for call in range(2):
        a = torch.empty((M, K), dtype=torch.float32, pin_memory=True)
        a.copy_(torch.from_numpy(workloads.make_activations(wl, M=M, K=K) + np.float32(call)))
        y_static = torch.full((M, N), float("nan"), dtype=torch.float32, pin_memory=True)
        assert call_static(q8, a, qw, s_w, y_static, colsum=colsum) == q8.Q8_OK
        y_ref = q8.q8_linear_host(a, qw, s_w, colsum, symmetric=False)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y_static.numpy().view(np.int32), y_ref.numpy().view(np.int32))


def test_argument_errors_come_before_the_size_check(q8):
    # a shape far beyond the array with a bad argument: the argument error is reported
    lib = q8.load()
    N, K = 1 << 23, 16
    a = torch.zeros((4, K), dtype=torch.float32)
    y = torch.zeros((4, 4), dtype=torch.float32)
    qw = torch.zeros((16, K), dtype=torch.int8, device="cuda")
    s_w = torch.ones(16, device="cuda")
    args = dict(a=ctypes.c_void_p(a.data_ptr()), qw=ctypes.c_void_p(qw.data_ptr()), s_w=ctypes.c_void_p(s_w.data_ptr()),
                y=ctypes.c_void_p(y.data_ptr()))
    bad = [
        (args["a"], 7, args["qw"], args["s_w"], q8.Q8_PER_ROW, None, args["y"]),          # symmetry not an enum value
        (args["a"], q8.Q8_SYMMETRIC, args["qw"], args["s_w"], 5, None, args["y"]),         # granularity
        (args["a"], q8.Q8_ASYMMETRIC, args["qw"], args["s_w"], q8.Q8_PER_ROW, None, args["y"]),   # no colsum
        (args["a"], q8.Q8_SYMMETRIC, None, args["s_w"], q8.Q8_PER_ROW, None, args["y"]),   # no weights
        (args["a"], q8.Q8_SYMMETRIC, args["qw"], args["s_w"], q8.Q8_PER_ROW, None, None),  # no output
    ]
    for a_p, sym, qw_p, sw_p, gw, cs, y_p in bad:
        assert lib.q8_linear_host_static(a_p, 4, K, sym, qw_p, sw_p, gw, cs, N, y_p, 0, None) == q8.Q8_ERR_INVALID_ARG


def test_sizes_beyond_the_array_are_rejected(q8):
    limit = q8.load().q8_linear_host_static_limit()
    assert limit == 64 << 20
    N, K = 1 << 23, 16                     # one output row of 32 MiB: two slots need more than the array
    assert q8.q8_linear_host_workspace(4, N, K, 1) > limit
    a = torch.zeros((4, K), dtype=torch.float32)
    y = torch.zeros((4, 4), dtype=torch.float32)             # never reached: rejected before any work
    qw = torch.zeros((16, K), dtype=torch.int8, device="cuda")
    s_w = torch.ones(16, device="cuda")
    lib = q8.load()
    st = lib.q8_linear_host_static(ctypes.c_void_p(a.data_ptr()), 4, K, q8.Q8_SYMMETRIC,
                                   ctypes.c_void_p(qw.data_ptr()), ctypes.c_void_p(s_w.data_ptr()), q8.Q8_PER_ROW,
                                   None, N, ctypes.c_void_p(y.data_ptr()), 0, None)
    assert st == q8.Q8_ERR_UNSUPPORTED
    M2, N2, K2 = 4096, 4096, 4096                            # an explicit slice too large for the array
    assert q8.q8_linear_host_workspace(M2, N2, K2, M2) > limit
    a2 = torch.zeros((M2, K2), dtype=torch.float32)
    y2 = torch.zeros((M2, N2), dtype=torch.float32)
    qw2 = torch.zeros((N2, K2), dtype=torch.int8, device="cuda")
    s_w2 = torch.ones(N2, device="cuda")
    assert call_static(q8, a2, qw2, s_w2, y2, chunk_rows=M2) == q8.Q8_ERR_UNSUPPORTED
