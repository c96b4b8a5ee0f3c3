"""Seeded random ragged shapes through every GEMM kernel that takes them.

Integer results (int8 and int4 weights) are compared with the oracle's int64 GEMM bit for
bit; block-scaled results use codes in [-3, 3] and exponents within four binades of a row
base, where every partial sum is exact in fp32, so they too must match the oracle's exactly
rounded sum bit for bit. A kernel that does not take a shape rejects it (Q8Error) and is
skipped for that shape; every shape runs on at least the CTA-pair kernel. The workspace forms
(the activation codes copied once as fp16 values for the pair kernel) run on the same shapes.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

INT8_KERNELS = ("tcgen05_pair", "tcgen05", "mma_s8", "skinny", "decode", "decode_tc")


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


def shapes(seed, count):
    rng = np.random.default_rng(seed)
    for _ in range(count):
        M = int(rng.choice([1, 2, 7, 15, 16, 17, 33, 64, 100, 255, 256, 257, 300, 513]))
        N = int(rng.integers(1, 700))
        K = int(rng.integers(1, 200)) * 32
        yield rng, M, N, K


def run_kernels(q8, fn, kernels):
    """{kernel: result} for the kernels that take the shape."""
    out = {}
    for k in kernels:
        try:
            out[k] = fn(k)
        except q8.Q8Error:
            continue
        assert q8.q8_device_error() == 0
    assert "tcgen05_pair" in out
    return out


@pytest.mark.parametrize("seed", [101, 202])
def test_random_shapes_int8_and_int4_weights(q8, seed):
    for rng, M, N, K in shapes(seed, 20):
        qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
        qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
        want = oracle.gemm_acc(qa, qw, threads=8)
        got = run_kernels(q8, lambda k: q8.q8_gemm_s32(dev(qa), dev(qw), kernel=k).cpu().numpy(), INT8_KERNELS)
        for k, acc in got.items():
            np.testing.assert_array_equal(acc.astype(np.int64), want, err_msg=f"int8 {k} {M}x{N}x{K}")
        q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
        want4 = oracle.gemm_acc(qa, q4, threads=8)
        packed = dev(oracle.pack_int4(q4))
        got4 = run_kernels(q8, lambda k: q8.q8_gemm_w4a8_s32(dev(qa), packed, kernel=k).cpu().numpy(),
                           ("tcgen05_pair", "decode"))
        for k, acc in got4.items():
            np.testing.assert_array_equal(acc.astype(np.int64), want4, err_msg=f"int4 {k} {M}x{N}x{K}")
        # the workspace forms with unit scales: y = fl(acc), rounded once like the oracle's int64 sums
        ws = torch.empty(2 * M * K, dtype=torch.uint8, device="cuda")
        ones_m, ones_n = dev(np.ones(M, np.float32)), dev(np.ones(N, np.float32))
        y8 = q8.q8_gemm_dequant(dev(qa), ones_m, None, dev(qw), ones_n, workspace=ws).cpu().numpy()
        y4 = q8.q8_gemm_w4a8(dev(qa), ones_m, None, packed, ones_n, workspace=ws).cpu().numpy()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y8, want.astype(np.float32), err_msg=f"int8 workspace {M}x{N}x{K}")
        np.testing.assert_array_equal(y4, want4.astype(np.float32), err_msg=f"int4 workspace {M}x{N}x{K}")


@pytest.mark.parametrize("seed", [303])
def test_random_shapes_block_scaled_weights(q8, seed):
    for rng, M, N, K in shapes(seed, 20):
        G = 32 if K % 128 else int(rng.choice([32, 128]))
        qa = rng.integers(-3, 4, (M, K), dtype=np.int8)
        q = rng.integers(-3, 4, (N, K), dtype=np.int8)
        e = rng.integers(103, 133, (N, 1)) + rng.integers(0, 4, (N, K // G))
        sf = np.zeros(((K // G + 3) // 4, N), np.uint32)
        for g in range(K // G):
            sf[g // 4] |= e[:, g].astype(np.uint32) << np.uint32(8 * (g % 4))
        t_ref, _ = oracle.gemm_mx(qa, q, sf, G, threads=8)
        ones = dev(np.ones(M, np.float32))
        got = run_kernels(q8, lambda k: q8.q8_gemm_mx(dev(qa), ones, dev(q), dev(sf.view(np.int32)), G,
                                                       kernel=k).cpu().numpy(), ("tcgen05_pair", "decode"))
        for k, t in got.items():
            np.testing.assert_array_equal(t.view(np.int32), t_ref.view(np.int32), err_msg=f"mx {k} G{G} {M}x{N}x{K}")
        ws = torch.empty(2 * M * K, dtype=torch.uint8, device="cuda")
        t = q8.q8_gemm_mx(dev(qa), ones, dev(q), dev(sf.view(np.int32)), G, workspace=ws).cpu().numpy()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(t.view(np.int32), t_ref.view(np.int32), err_msg=f"mx workspace G{G} {M}x{N}x{K}")


@pytest.mark.parametrize("seed", [404])
def test_random_shapes_fp32_layer_with_the_default_kernel(q8, seed):
    # the fp32 epilogue (asymmetric tokens, per-channel weights) on whatever kernel the pick and the
    # K split choose for the shape, straight after the activation quantizer on the same stream
    for rng, M, N, K in shapes(seed, 16):
        a = rng.standard_normal((M, K), dtype=np.float32)
        qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
        sw = (rng.random(N, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
        qa, sa, za = q8.q8_quantize_act(dev(a), per_row=True, symmetric=False)
        y = q8.q8_gemm_dequant(qa, sa, za, dev(qw), dev(sw), q8.q8_colsum(dev(qw))).cpu().numpy()
        assert q8.q8_device_error() == 0
        y_ref, st = oracle.linear_codes(qa.cpu().numpy(), sa.cpu().numpy(), za.cpu().numpy(), qw, sw, True, True,
                                        threads=8)
        assert st == oracle.OK
        np.testing.assert_array_equal(y.view(np.int32), y_ref.view(np.int32), err_msg=f"{M}x{N}x{K}")
        # the layer in one call with a workspace (quantizer writing the fp16 copy, pair kernel on it)
        ws = torch.empty(max(16, q8.q8_gemm_workspace(M, N, K)), dtype=torch.uint8, device="cuda")
        y_ws = q8.q8_linear(dev(a), dev(qw), dev(sw), q8.q8_colsum(dev(qw)), symmetric=False, workspace=ws)
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(y_ws.cpu().numpy().view(np.int32), y_ref.view(np.int32),
                                      err_msg=f"linear workspace {M}x{N}x{K}")
