"""The host-buffer layer q8_linear_host: A in host memory -> y in host memory, the copies
overlapped with the device work slice by slice. Per-token quantization acts row by row
and the INT32 GEMM is exact, so every slicing gives the bits of the one-call device path
(q8_quantize_act + q8_gemm_dequant), which the parity tests hold to the oracle; the
small cases are also checked against the oracle directly.
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


def device_layer(q8, a, qw, s_w, colsum, sym):
    qa, s_a, z_a = q8.q8_quantize_act(a.cuda(), per_row=True, symmetric=sym)
    y = q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum if not sym else None)
    return y.cpu()


def pinned(x):
    t = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    t.copy_(x)
    return t


@pytest.mark.parametrize("M,N,K,chunk,sym", [
    (1000, 264, 512, 0, True),        # default slices (256 rows), ragged last slice
    (1000, 264, 512, 1, True),        # one row per slice: 1000 slices through two slots
    (300, 520, 2064, 128, False),     # asymmetric with column sums
    (77, 130, 256, 500, True),        # one slice (chunk > M), N not a multiple of 4
    (4096, 2048, 4096, 0, True),      # default slices of whole tiles (256 rows)
])
def test_host_layer_matches_the_device_path(q8, M, N, K, chunk, sym):
    wl = workloads.WORKLOADS["prefill2k" if sym else "relu4k"]
    a = torch.from_numpy(workloads.make_activations(wl, M=M, K=K))
    w = torch.from_numpy(workloads.make_weights(wl, N=N, K=K)).cuda()
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    colsum = q8.q8_colsum(qw)
    y = q8.q8_linear_host(pinned(a), qw, s_w, colsum, symmetric=sym, chunk_rows=chunk)
    torch.cuda.synchronize()
    ref = device_layer(q8, a, qw, s_w, colsum, sym)
    np.testing.assert_array_equal(y.numpy().view(np.int32), ref.numpy().view(np.int32))
    if M * N * K <= 300 * 520 * 2064:
        y_or = oracle.linear(a.numpy(), w.cpu().numpy(), act_per_row=True, act_symmetric=sym, w_per_row=True,
                             threads=8)["y"]
        np.testing.assert_array_equal(y.numpy().view(np.int32), y_or.view(np.int32))


def test_repeated_calls_reuse_the_workspace_and_pageable_buffers_work(q8):
    M, N, K = 700, 256, 1024
    wl = workloads.WORKLOADS["prefill2k"]
    w = torch.from_numpy(workloads.make_weights(wl, N=N, K=K)).cuda()
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    ws = torch.empty(q8.q8_linear_host_workspace(M, N, K, 200), dtype=torch.uint8, device="cuda")
    outs = []
    for seed in range(3):
        a = torch.from_numpy(workloads.make_activations(wl, M=M, K=K) * np.float32(seed + 1))
        y = torch.empty((M, N), dtype=torch.float32)            # pageable: copies run synchronously
        q8.q8_linear_host(a, qw, s_w, None, y, chunk_rows=200, workspace=ws)
        outs.append((a, y))
    torch.cuda.synchronize()
    for a, y in outs:
        ref = device_layer(q8, a, qw, s_w, None, True)
        np.testing.assert_array_equal(y.numpy().view(np.int32), ref.numpy().view(np.int32))


def test_k_zero_gives_zeros_and_empty_shapes_do_nothing(q8):
    qw = torch.empty((8, 0), dtype=torch.int8, device="cuda")
    s_w = torch.ones(8, device="cuda")
    y = torch.full((5, 8), 7.0).pin_memory()
    q8.q8_linear_host(torch.empty((5, 0)), qw, s_w, None, y)
    torch.cuda.synchronize()
    assert float(y.abs().sum()) == 0.0
    y0 = torch.full((0, 8), 1.0)
    q8.q8_linear_host(torch.empty((0, 16)), torch.zeros((8, 16), dtype=torch.int8, device="cuda"), s_w, None, y0)


def test_too_small_workspace_is_rejected_before_anything_runs(q8):
    M, N, K = 64, 64, 64
    qw = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    s_w = torch.ones(N, device="cuda")
    a = torch.zeros((M, K)).pin_memory()
    y = torch.full((M, N), 3.0).pin_memory()
    small = torch.empty(q8.q8_linear_host_workspace(M, N, K) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(q8.Q8Error):
        q8.q8_linear_host(a, qw, s_w, None, y, workspace=small)
    torch.cuda.synchronize()
    assert float(y.min()) == 3.0


def test_full_size_host_layer_as_the_bench_times_it(q8):
    # the prefill16k layer (8192 x 16384 tokens, 8192 channels) with the default slicing that
    # bench.py's e2e figure uses: bit-identical to the device path on every output
    wl = workloads.WORKLOADS["prefill16k"]
    a = torch.from_numpy(workloads.make_activations(wl))
    w = torch.from_numpy(workloads.make_weights(wl)).cuda()
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    del w
    y = q8.q8_linear_host(pinned(a), qw, s_w, None)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    ref = device_layer(q8, a, qw, s_w, None, True)
    np.testing.assert_array_equal(y.numpy().view(np.int32), ref.numpy().view(np.int32))
