"""The int4 and block-scaled weight layers with a caller workspace (q8_gemm_w4a8_ws, q8_gemm_mx_ws).

The activation codes are written once into the workspace as fp16 values, each group of four K
stored as K 0, 2, 1, 3 (the order in which the CTA-pair kernel converts the weight codes), and the
kernel loads them by TMA instead of converting them per output tile. The tensor core then sees the
same operands in the same order as on the direct path, so y must equal the direct path's bit for
bit: for int4 weights the exact INT32 sums of the TileLang tutorial's int4 GEMM example (ch. 27,
2.4 int8 / int4), for block-scaled weights (ch. 27, 2.3 MX / E8M0 block scales) the same fp32
tensor-core sums, which the direct path's tests hold to the accumulation bound. Both are also
checked against the oracle here.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gates
from tests.test_gpu_mx import accumulation_gate, block_weights, words

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


def pair_order(qa):
    """The codes [M, K] with each group of four K as K 0, 2, 1, 3."""
    M, K = qa.shape
    return qa.reshape(M, K // 4, 4)[:, :, [0, 2, 1, 3]].reshape(M, K)


def workspace(M, K):
    # stale contents: the call overwrites what it uses
    return torch.full((2 * M * K,), 0x55, dtype=torch.uint8, device="cuda")


W4_CASES = [
    # M, N, K, symmetric activations
    (200, 264, 1088, True),       # ragged M and N, 17 k-blocks (no even K split): whole tiles
    (513, 777, 3104, False),      # zero points and column sums, ragged everything
    (2048, 2048, 4096, True),     # one wave of 64 whole tiles
    (2344, 2056, 2048, True),     # 90 ragged tiles: two waves, the last wave's 14 tiles in 4 K slices
    (256, 256, 32, True),         # one k-block
    (300, 520, 16416, False),     # K past one exact 16384-K chunk
]


@pytest.mark.parametrize("M,N,K,sym", W4_CASES)
def test_w4a8_workspace_equals_the_direct_layer_and_the_oracle(q8, M, N, K, sym):
    wl = workloads.WORKLOADS["prefill2k" if sym else "relu4k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    q4, s4 = oracle.quantize_int4(w)
    qw4 = dev(oracle.pack_int4(q4))
    if sym:
        qa, sa = oracle.quantize_sym(a, per_row=True)
        za, cs = None, None
    else:
        qa, sa, za = oracle.quantize_asym(a, per_row=True)
        cs = dev(oracle.colsum(q4).astype(np.int32))
    args = (dev(qa), dev(sa), None if za is None else dev(za), qw4, dev(s4))
    ws = workspace(M, K)
    y_direct = q8.q8_gemm_w4a8(*args, colsum=cs)
    for _ in range(2):
        y_ws = q8.q8_gemm_w4a8(*args, colsum=cs, workspace=ws)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(host(y_ws).view(np.int32), host(y_direct).view(np.int32))
    ref, st = oracle.linear_codes(qa, sa, za, q4, s4, True, True, threads=8)
    assert st == oracle.OK
    assert int(gates.ulp_distance(host(y_ws), ref).max()) <= 2
    # the workspace holds the codes as fp16 values, in pair order
    np.testing.assert_array_equal(host(ws.view(torch.float16)[:M * K].view(M, K)).astype(np.int32),
                                  pair_order(qa).astype(np.int32))
    # bf16 output through the same path
    yb = q8.q8_gemm_w4a8(*args, colsum=cs, out_dtype=torch.bfloat16, workspace=ws)
    np.testing.assert_array_equal(host(yb.view(torch.int16)).view(np.uint16), oracle.to_bf16(host(y_ws)))


def test_w4a8_workspace_largest_products_at_a_large_k(q8):
    # |a n| at its maxima on every k over four exact 16384-K chunks; unit scales give y = fl(acc)
    M, N, K = 256, 256, 65536
    rng = np.random.default_rng(K)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
    qa[0, :], qa[1, :], qa[2, :] = -128, 127, -128
    q4[0, :], q4[1, :], q4[2, :] = 7, -8, -8
    ones_m, ones_n = dev(np.ones(M, np.float32)), dev(np.ones(N, np.float32))
    y = q8.q8_gemm_w4a8(dev(qa), ones_m, None, dev(oracle.pack_int4(q4)), ones_n, workspace=workspace(M, K))
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    want = oracle.gemm_acc(qa, q4, threads=8)
    assert want[0, 0] == -128 * 7 * K and want[2, 2] == 1024 * K
    np.testing.assert_array_equal(host(y), want.astype(np.float32))


def test_w4a8_workspace_too_small_or_decode_shape_is_not_used(q8):
    M, N, K = 16, 1024, 4096                  # decode kernel: the workspace stays untouched
    rng = np.random.default_rng(3)
    qa = dev(rng.integers(-128, 128, (M, K), dtype=np.int8))
    q4 = dev(oracle.pack_int4(rng.integers(-8, 8, (N, K), dtype=np.int8)))
    sa, s4 = dev(np.ones(M, np.float32)), dev(np.ones(N, np.float32))
    ws = workspace(M, K)
    y = q8.q8_gemm_w4a8(qa, sa, None, q4, s4, workspace=ws)
    np.testing.assert_array_equal(host(y), host(q8.q8_gemm_w4a8(qa, sa, None, q4, s4)))
    assert bool((ws == 0x55).all())
    M = 300                                   # pair kernel, one byte short: the direct path
    qa = dev(rng.integers(-128, 128, (M, K), dtype=np.int8))
    sa = dev(np.ones(M, np.float32))
    short = torch.full((2 * M * K - 1,), 0x55, dtype=torch.uint8, device="cuda")
    y = q8.q8_gemm_w4a8(qa, sa, None, q4, s4, workspace=short)
    np.testing.assert_array_equal(host(y), host(q8.q8_gemm_w4a8(qa, sa, None, q4, s4)))
    assert bool((short == 0x55).all())
    assert q8.q8_device_error() == 0


MX_CASES = [(200, 264, 1088, 32), (513, 777, 4096, 128), (2048, 1024, 4096, 32), (300, 520, 512, 128),
            (2344, 2056, 512, 32)]   # 90 ragged tiles: two waves (whole tiles)


@pytest.mark.parametrize("M,N,K,G", MX_CASES)
def test_mx_workspace_equals_the_direct_layer_and_the_accumulation_bound(q8, M, N, K, G):
    wl = workloads.WORKLOADS["prefill2k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=K + G)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    d = dict(qw=dev(q), sf=dev(words(sf)), group=G)
    ws = workspace(M, K)
    ones = dev(np.ones(M, np.float32))
    t_direct = q8.q8_gemm_mx(dev(qa), ones, **d)
    for _ in range(2):
        t_ws = q8.q8_gemm_mx(dev(qa), ones, workspace=ws, **d)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(host(t_ws).view(np.int32), host(t_direct).view(np.int32))
    t_ref, absum = oracle.gemm_mx(qa, q, sf, G, threads=8)
    accumulation_gate(host(t_ws), t_ref, absum, qa, q, sf, G)
    np.testing.assert_array_equal(host(ws.view(torch.float16)[:M * K].view(M, K)).astype(np.int32),
                                  pair_order(qa).astype(np.int32))
    # the scaled layer and its epilogue variants through the same path
    bias = workloads.gaussian((N,), 11) * np.float32(0.1)
    y = host(q8.q8_gemm_mx(dev(qa), dev(sa), bias=dev(bias), workspace=ws, **d))
    np.testing.assert_array_equal(y, host(q8.q8_gemm_mx(dev(qa), dev(sa), bias=dev(bias), **d)))
    yb = q8.q8_gemm_mx(dev(qa), dev(sa), bias=dev(bias), out_dtype=torch.bfloat16, workspace=ws, **d)
    np.testing.assert_array_equal(host(yb.view(torch.int16)).view(np.uint16), oracle.to_bf16(y))


def test_mx_workspace_large_scales_take_the_scaled_conversion(q8):
    # exponents above 132 in some rows take the converters' second form ((1152 + q) s / 16, times 16)
    M, N, K, G = 260, 264, 1024, 32
    rng = np.random.default_rng(5)
    qa = rng.integers(-3, 4, (M, K), dtype=np.int8)
    q = rng.integers(-3, 4, (N, K), dtype=np.int8)
    e = rng.integers(127, 137, (N, 1)) + np.zeros((1, K // G), np.int64)
    e[::3] = 103 + rng.integers(0, 4, (e[::3].shape[0], K // G))
    from tests.test_gpu_mx import sf_from_exponents
    sf = sf_from_exponents(e)
    t_ref, _ = oracle.gemm_mx(qa, q, sf, G, threads=8)
    ones = dev(np.ones(M, np.float32))
    t = host(q8.q8_gemm_mx(dev(qa), ones, dev(q), dev(words(sf)), G, workspace=workspace(M, K)))
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(t.view(np.int32), t_ref.view(np.int32))


@pytest.mark.parametrize("ws", [False, True])
def test_mx_scale_words_by_tma_and_by_loads_agree(q8, ws):
    # N % 4 == 0 and a 16-byte aligned scale array: the pair kernel stages the scale words by TMA;
    # the same words 4 bytes past a 16-byte boundary take the converters' own loads
    M, N, K, G = 300, 520, 2048, 32
    wl = workloads.WORKLOADS["prefill2k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=9)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    sf_words = words(sf)
    aligned = dev(sf_words)
    assert aligned.data_ptr() % 16 == 0
    shifted_store = torch.zeros(sf_words.size + 4, dtype=torch.int32, device="cuda")
    shifted = shifted_store[1:1 + sf_words.size].view(sf_words.shape)
    shifted.copy_(aligned)
    assert shifted.data_ptr() % 16 == 4
    extra = {"workspace": workspace(M, K)} if ws else {}
    t1 = host(q8.q8_gemm_mx(dev(qa), dev(np.ones(M, np.float32)), dev(q), aligned, G, **extra))
    t2 = host(q8.q8_gemm_mx(dev(qa), dev(np.ones(M, np.float32)), dev(q), shifted, G, **extra))
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(t1.view(np.int32), t2.view(np.int32))
    t_ref, absum = oracle.gemm_mx(qa, q, sf, G, threads=8)
    accumulation_gate(t1, t_ref, absum, qa, q, sf, G)


def _ulp(a, b):
    return int(gates.ulp_distance(a, b).max()) if a.size else 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "prefill16k"])
def test_w4a8_full_size(q8, name):
    """The measured int4 configurations at full size: the weights' codes and scales in full; the
    decode layer at every output; the prefill layer (direct and with the workspace, bit-identical)
    on 16 whole rows, 16 whole columns and 3000 sampled outputs."""
    wl = workloads.WORKLOADS[name]
    a = workloads.make_activations(wl)
    w = workloads.make_weights(wl)
    rq4, rs4 = oracle.quantize_int4(w)
    qw4, s4 = q8.q8_quantize_weight_int4(dev(w))
    del w
    np.testing.assert_array_equal(host(qw4), oracle.pack_int4(rq4))
    np.testing.assert_array_equal(host(s4), rs4)
    rqa, rsa = oracle.quantize_sym(a, True)
    qa, sa, _ = q8.q8_quantize_act(dev(a))
    del a
    np.testing.assert_array_equal(host(qa), rqa)
    y = q8.q8_gemm_w4a8(qa, sa, None, qw4, s4)
    threads = oracle.max_threads()
    if name == "decode":
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        ry, st = oracle.linear_codes(rqa, rsa, None, rq4, rs4, True, True, threads=threads)
        assert st == oracle.OK
        assert _ulp(host(y), ry) <= 2
        return
    y_ws = q8.q8_gemm_w4a8(qa, sa, None, qw4, s4, workspace=workspace(wl.M, wl.K))
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    assert torch.equal(y_ws.view(torch.int32), y.view(torch.int32))
    yh = host(y)
    rng = np.random.default_rng(wl.seed + 23)
    rows = np.unique(np.concatenate([rng.integers(0, wl.M, 14), [0, wl.M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, wl.N, 14), [0, wl.N - 1]]))
    ry_r, st = oracle.linear_codes(rqa[rows], rsa[rows], None, rq4, rs4, True, True, threads=threads)
    assert st == oracle.OK
    assert _ulp(yh[rows], ry_r) <= 2
    ry_c, st = oracle.linear_codes(rqa, rsa, None, rq4[cols], rs4[cols], True, True, threads=threads)
    assert st == oracle.OK
    assert _ulp(yh[:, cols], ry_c) <= 2
    ms = rng.integers(0, wl.M, 3000)
    ns = rng.integers(0, wl.N, 3000)
    ry_s, _, st = oracle.linear_codes_at(rqa, rsa, None, rq4, rs4, ms, ns, True, True)
    assert st == oracle.OK
    assert _ulp(yh[ms, ns], ry_s) <= 2
