"""GPU parity of the block-scaled (MX-style) int8 weight path against the oracle.

TileLang tutorial ch. 27 (low-precision quantization), 2.3 MX / block-scaled. The
weight quantizer is integer / exponent work and must be bit-identical (codes and
scale words). The GEMM dequantizes each weight to the fp16 value q * s (exact) and
the tensor core sums the exact products in fp32 over the whole K, so the result
equals the oracle's exactly rounded sum only where every partial sum is an fp32
value: those designed cases are compared bit for bit (they also pin the scale
layout: byte order, group-major words, the group of every K chunk). Elsewhere the
gate follows the kernel's summation: the accumulator takes one fp32 rounding per
16-wide MMA step j (at most 2 ulp, 2^-22 relative: allowing truncation and the
alignment of the step's 16 exact products), so with P_j the exact running sum after
step j, |T - T_exact| <= 2^-22 (sum_j |P_j| + sum_k |p_k|), plus one rounding of T
and of y. The running sums are exact int64 fixed-point sums (every product
q a 2^(e - 127) is an integer multiple of 2^-24 below 2^23).
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


def words(sf_np):
    return np.ascontiguousarray(sf_np).view(np.int32)


def block_weights(N, K, G, seed):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02)
    mag = np.exp(rng.uniform(np.log(2.0 ** -8), 0.0, size=(N, K // G))).astype(np.float32)
    return (w.reshape(N, K // G, G) * mag[:, :, None]).reshape(N, K).astype(np.float32)


def sf_from_exponents(e):
    """Scale words [ceil(groups / 4), N] from exponents e [N, groups] (byte g % 4 of word g / 4)."""
    N, groups = e.shape
    sf = np.zeros(((groups + 3) // 4, N), np.uint32)
    for g in range(groups):
        sf[g // 4] |= (e[:, g].astype(np.uint32) << np.uint32(8 * (g % 4)))
    return sf


def unit_scales(M):
    return dev(np.ones(M, np.float32))


@pytest.mark.parametrize("N,K,G", [(64, 256, 32), (300, 4128, 32), (17, 8192, 128), (1000, 2048, 128)])
def test_quantize_weight_mx_bit_exact(q8, N, K, G):
    w = block_weights(N, K, G, seed=N + K)
    w[N // 2] = 0.0                                          # zero groups: e = 103, codes 0
    w[N // 3, :G] *= np.float32(1e9)                         # a saturating group: e = 136, codes +-127
    qw, sf = q8.q8_quantize_weight_mx(dev(w), G)
    q_ref, sf_ref = oracle.quantize_weight_mx(w, G)
    np.testing.assert_array_equal(host(qw), q_ref)
    np.testing.assert_array_equal(host(sf), words(sf_ref))


EXACT_CASES = [(300, 520, 512, 32), (16, 264, 1024, 128), (513, 256, 2048, 32), (1, 72, 512, 128)]


@pytest.mark.parametrize("M,N,K,G", EXACT_CASES)
def test_block_scales_applied_exactly_where_fp32_sums_are_exact(q8, M, N, K, G):
    # codes in [-3, 3] and exponents spread over 4 binades per row: every partial sum is a
    # multiple of the row's smallest scale below 2^24 of it, so any summation order is exact
    rng = np.random.default_rng(M * 31 + K)
    qa = rng.integers(-3, 4, (M, K), dtype=np.int8)
    q = rng.integers(-3, 4, (N, K), dtype=np.int8)
    base = rng.integers(103, 133, (N, 1))
    e = base + rng.integers(0, 4, (N, K // G))
    sf = sf_from_exponents(e)
    t_ref, _ = oracle.gemm_mx(qa, q, sf, G, threads=8)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G))
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(t.view(np.int32), t_ref.view(np.int32))


def test_equal_scales_give_the_scaled_integer_product(q8):
    # one exponent per row and |acc| < 2^24 (K = 1024): T = 2^(e - 127) * acc exactly
    M, N, K, G = 256, 256, 1024, 32
    rng = np.random.default_rng(77)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    q = rng.integers(-127, 128, (N, K), dtype=np.int8)
    e = np.repeat(rng.integers(103, 137, (N, 1)), K // G, axis=1)
    sf = sf_from_exponents(e)
    acc = qa.astype(np.int64) @ q.astype(np.int64).T
    want = (acc.astype(np.float64) * np.exp2(e[:, 0] - 127.0)[None, :]).astype(np.float32)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G))
    np.testing.assert_array_equal(t, want)


def running_sums(qa, q, sf, G):
    """(sum_j |P_j|, T_exact) per output as float64 from exact int64 sums: P_j is the exact sum of the
    products of the first j 16-wide K steps, in units of 2^-24 (q a 2^(e - 103), e >= 103: integers
    below 2^47, sums of up to 2^16 of them below 2^63)."""
    M, K = qa.shape
    N = q.shape[0]
    groups = K // G
    e = np.zeros((N, groups), np.int64)
    for g in range(groups):
        e[:, g] = (sf[g // 4].astype(np.int64) >> (8 * (g % 4))) & 0xFF
    wq = q.astype(np.int64) * np.left_shift(np.int64(1), np.repeat(e - 103, G, axis=1))   # [N, K]
    a = qa.astype(np.int64)
    run = np.zeros((M, N), np.int64)
    tot = np.zeros((M, N), np.float64)
    for k0 in range(0, K, 16):
        run += a[:, k0:k0 + 16] @ wq[:, k0:k0 + 16].T
        tot += np.abs(run).astype(np.float64)
    return tot * 2.0 ** -24, run.astype(np.float64) * 2.0 ** -24


def decode_tree_sums(qa, q, sf, G):
    """sum over the nodes of the decode kernel's summation tree of |exact node value| (units of
    2^-24, as float64): warp w (of 16) runs an fp32 partial over the 16-wide pieces
    [512 s + 32 w + 16 h, + 16) in the order s, h; warps 8 .. 15 are added onto warps 0 .. 7;
    the eight sums are added in warp order."""
    M, K = qa.shape
    N = q.shape[0]
    groups = K // G
    e = np.zeros((N, groups), np.int64)
    for g in range(groups):
        e[:, g] = (sf[g // 4].astype(np.int64) >> (8 * (g % 4))) & 0xFF
    wq = q.astype(np.int64) * np.left_shift(np.int64(1), np.repeat(e - 103, G, axis=1))
    a = qa.astype(np.int64)
    tot = np.zeros((M, N), np.float64)
    part = []
    for w in range(16):
        run = np.zeros((M, N), np.int64)
        for s0 in range(0, K, 512):
            for h in range(2):
                k0 = s0 + 32 * w + 16 * h
                if k0 >= K:
                    continue
                run += a[:, k0:k0 + 16] @ wq[:, k0:k0 + 16].T
                tot += np.abs(run)
        part.append(run)
    comb = [part[w] + part[w + 8] for w in range(8)]
    for c in comb:
        tot += np.abs(c)
    r = comb[0].copy()
    for w in range(1, 8):
        r += comb[w]
        tot += np.abs(r)
    return tot * 2.0 ** -24, r.astype(np.float64) * 2.0 ** -24


def accumulation_gate(t, t_ref, absum, qa, q, sf, G, order="pair"):
    """|T - T_exact| <= 2^-22 (sum of |exact partial sums| along the kernel's summation order +
    sum_k |p_k|) + one rounding of T. order: "pair" (the tensor-core kernel: K steps in sequence)
    or "decode" (the warp-MMA decode kernel's tree)."""
    sum_p, t_exact = running_sums(qa, q, sf, G) if order == "pair" else decode_tree_sums(qa, q, sf, G)
    assert np.array_equal(t_exact.astype(np.float32), t_ref)   # the oracle's T is the exact sum, rounded once
    bound = 2.0 ** -22 * (sum_p + absum) + np.abs(t_ref) * 2.0 ** -23
    err = np.abs(t.astype(np.float64) - t_ref.astype(np.float64))
    assert np.all(err <= bound)
    return err, bound


@pytest.mark.parametrize("M,N,K,G", [(200, 264, 1088, 32), (513, 777, 4096, 128), (16, 1000, 8192, 32)])
def test_layer_within_the_accumulation_bound(q8, M, N, K, G):
    wl = workloads.WORKLOADS["prefill2k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=K)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    t_ref, absum = oracle.gemm_mx(qa, q, sf, G, threads=8)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G))
    assert q8.q8_device_error() == 0
    _, tbound = accumulation_gate(t, t_ref, absum, qa, q, sf, G)
    y = host(q8.q8_gemm_mx(dev(qa), dev(sa), dev(q), dev(words(sf)), G))
    y_ref = oracle.linear_mx(qa, sa, q, sf, G)
    # y = fl(T * s_a): the same bound scaled by s_a, plus one rounding of y
    bound = sa[:, None] * tbound + np.abs(y_ref) * 2.0 ** -23
    assert np.all(np.abs(y.astype(np.float64) - y_ref) <= bound)
    # deterministic: the same bits again
    y2 = host(q8.q8_gemm_mx(dev(qa), dev(sa), dev(q), dev(words(sf)), G))
    np.testing.assert_array_equal(y.view(np.int32), y2.view(np.int32))


def test_epilogue_variants_follow_the_fp32_result(q8):
    M, N, K, G = 300, 272, 2048, 32
    wl = workloads.WORKLOADS["prefill2k"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=5)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    bias = workloads.gaussian((N,), 13) * np.float32(0.1)
    d = dict(qa=dev(qa), s_a=dev(sa), qw=dev(q), sf=dev(words(sf)), group=G)
    y0 = host(q8.q8_gemm_mx(**d))
    yb = host(q8.q8_gemm_mx(bias=dev(bias), **d))
    np.testing.assert_array_equal(yb, (y0 + bias[None, :]).astype(np.float32))
    y16 = host(q8.q8_gemm_mx(bias=dev(bias), out_dtype=torch.bfloat16, **d).view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(y16, oracle.to_bf16(yb))
    s_out = float(np.float32(np.abs(yb).max() / np.float32(100.0)))
    y8 = host(q8.q8_gemm_mx(bias=dev(bias), out_dtype=torch.int8, out_scale=s_out, **d))
    np.testing.assert_array_equal(y8, oracle.quantize_static(yb, s_out))
    yt = host(q8.q8_gemm_mx(d["qa"], dev(sa[:1].copy()), d["qw"], d["sf"], G))   # per-tensor s_a
    t = host(q8.q8_gemm_mx(d["qa"], unit_scales(M), d["qw"], d["sf"], G))
    np.testing.assert_array_equal(yt, (t * sa[0]).astype(np.float32))


def test_k_zero_and_empty(q8):
    bias = workloads.gaussian((8,), 3)
    z = torch.empty((3, 0), dtype=torch.int8, device="cuda")
    w = torch.empty((8, 0), dtype=torch.int8, device="cuda")
    sf = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    y = host(q8.q8_gemm_mx(z, torch.ones(3, device="cuda"), w, sf, 32, bias=dev(bias)))
    np.testing.assert_array_equal(y, np.broadcast_to(bias, (3, 8)))


def test_full_size_sampled_outputs(q8):
    # the measured configuration: prefill16k activations, block-scaled weights (G = 32); the
    # oracle quantizes the sampled rows of the same floats itself (per-token and per-group
    # quantization act row by row)
    wl = workloads.WORKLOADS["prefill16k"]
    M, N, K, G = wl.M, wl.N, wl.K, 32
    a_np = workloads.make_activations(wl)
    w_np = block_weights(N, K, G, seed=16)
    qa, sa, _ = q8.q8_quantize_act(dev(a_np))
    qw, sf = q8.q8_quantize_weight_mx(dev(w_np), G)
    y = q8.q8_gemm_mx(qa, sa, qw, sf, G)
    t = q8.q8_gemm_mx(qa, torch.ones(M, device="cuda"), qw, sf, G)
    # the workspace form the bench also times: the same bits
    t_ws = q8.q8_gemm_mx(qa, torch.ones(M, device="cuda"), qw, sf, G,
                         workspace=torch.empty(2 * M * K, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    assert torch.equal(t_ws.view(torch.int32), t.view(torch.int32))
    del t_ws
    rng = np.random.default_rng(0)
    ms = np.unique(np.concatenate([rng.integers(0, M, 40), [0, M - 1]]))
    ns = np.unique(np.concatenate([rng.integers(0, N, 40), [0, N - 1]]))
    qa_s, sa_s = oracle.quantize_sym(a_np[ms], per_row=True)
    qw_s, sf_s = oracle.quantize_weight_mx(w_np[ns], G)
    np.testing.assert_array_equal(host(qa)[ms], qa_s)
    np.testing.assert_array_equal(host(qw)[ns], qw_s)
    np.testing.assert_array_equal(host(sf)[:, ns], words(sf_s))
    t_ref, absum = oracle.gemm_mx(qa_s, qw_s, sf_s, G, threads=8)
    t_s = host(t)[np.ix_(ms, ns)]
    accumulation_gate(t_s, t_ref, absum, qa_s, qw_s, sf_s, G)
    np.testing.assert_array_equal(host(y)[np.ix_(ms, ns)], (t_s * sa_s[:, None]).astype(np.float32))


DECODE_EXACT = [(16, 264, 1024, 128), (1, 72, 512, 128), (7, 200, 2080, 32), (16, 4096, 8192, 32), (3, 68, 32, 32)]


@pytest.mark.parametrize("M,N,K,G", DECODE_EXACT)
@pytest.mark.parametrize("kernel", ["decode", "tcgen05_pair"])
def test_decode_shapes_exact_where_fp32_sums_are_exact(q8, M, N, K, G, kernel):
    # both kernels that take M <= 16, on the designed exact cases (ragged N, K tails of 16 and
    # of 32 past a 256-K stage, every token count's padding)
    rng = np.random.default_rng(M * 7 + N + K)
    qa = rng.integers(-3, 4, (M, K), dtype=np.int8)
    q = rng.integers(-3, 4, (N, K), dtype=np.int8)
    base = rng.integers(103, 133, (N, 1))
    e = base + rng.integers(0, 4, (N, K // G))
    sf = sf_from_exponents(e)
    t_ref, _ = oracle.gemm_mx(qa, q, sf, G, threads=8)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G, kernel=kernel))
    assert q8.q8_device_error() == 0
    np.testing.assert_array_equal(t.view(np.int32), t_ref.view(np.int32))


@pytest.mark.parametrize("M,N,K,G", [(16, 1000, 8192, 32), (5, 520, 4096, 128), (16, 2048, 16384, 32)])
def test_decode_kernel_within_the_accumulation_bound(q8, M, N, K, G):
    wl = workloads.WORKLOADS["decode"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=K + 1)
    w[1, :G] *= np.float32(3e6)                              # one group with s > 32 (e = 133 .. 136)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    assert ((sf[0, 1] & 0xFF) > 132)
    t_ref, absum = oracle.gemm_mx(qa, q, sf, G, threads=8)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G, kernel="decode"))
    assert q8.q8_device_error() == 0
    accumulation_gate(t, t_ref, absum, qa, q, sf, G, order="decode")
    y = host(q8.q8_gemm_mx(dev(qa), dev(sa), dev(q), dev(words(sf)), G, kernel="decode"))
    np.testing.assert_array_equal(y, (t * sa[:, None]).astype(np.float32))
    y2 = host(q8.q8_gemm_mx(dev(qa), dev(sa), dev(q), dev(words(sf)), G))   # auto picks the decode kernel
    np.testing.assert_array_equal(y.view(np.int32), y2.view(np.int32))


def test_decode_kernel_epilogue_variants(q8):
    M, N, K, G = 11, 264, 2048, 32
    wl = workloads.WORKLOADS["decode"]
    a = workloads.make_activations(wl, M=M, K=K)
    w = block_weights(N, K, G, seed=9)
    qa, sa = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    bias = workloads.gaussian((N,), 21) * np.float32(0.1)
    d = dict(qa=dev(qa), s_a=dev(sa), qw=dev(q), sf=dev(words(sf)), group=G, kernel="decode")
    y0 = host(q8.q8_gemm_mx(**d))
    yb = host(q8.q8_gemm_mx(bias=dev(bias), **d))
    np.testing.assert_array_equal(yb, (y0 + bias[None, :]).astype(np.float32))
    y16 = host(q8.q8_gemm_mx(bias=dev(bias), out_dtype=torch.bfloat16, **d).view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(y16, oracle.to_bf16(yb))
    s_out = float(np.float32(np.abs(yb).max() / np.float32(100.0)))
    y8 = host(q8.q8_gemm_mx(bias=dev(bias), out_dtype=torch.int8, out_scale=s_out, **d))
    np.testing.assert_array_equal(y8, oracle.quantize_static(yb, s_out))
    yt = host(q8.q8_gemm_mx(d["qa"], dev(sa[:1].copy()), d["qw"], d["sf"], G, kernel="decode"))   # per-tensor s_a
    t = host(q8.q8_gemm_mx(d["qa"], unit_scales(M), d["qw"], d["sf"], G, kernel="decode"))
    np.testing.assert_array_equal(yt, (t * sa[0]).astype(np.float32))


def test_decode_kernel_rejects_what_it_cannot_take(q8):
    qa = torch.zeros((17, 64), dtype=torch.int8, device="cuda")   # M > 16
    qw = torch.zeros((8, 64), dtype=torch.int8, device="cuda")
    sf = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(q8.Q8Error):
        q8.q8_gemm_mx(qa, torch.ones(17, device="cuda"), qw, sf, 32, kernel="decode")
    qw6 = torch.zeros((6, 64), dtype=torch.int8, device="cuda")   # N % 4 != 0: the pair kernel takes it
    sf6 = torch.zeros((1, 6), dtype=torch.int32, device="cuda")
    with pytest.raises(q8.Q8Error):
        q8.q8_gemm_mx(qa[:4], torch.ones(4, device="cuda"), qw6, sf6, 32, kernel="decode")
    y = q8.q8_gemm_mx(qa[:4], torch.ones(4, device="cuda"), qw6, sf6, 32)
    torch.cuda.synchronize()
    assert float(y.abs().sum()) == 0.0


def test_decode_full_size_sampled_outputs(q8):
    # the decode workload (16 x 8192 tokens x 28672 rows) with block-scaled weights, G = 32
    wl = workloads.WORKLOADS["decode"]
    M, N, K, G = wl.M, wl.N, wl.K, 32
    a_np = workloads.make_activations(wl)
    w_np = block_weights(N, K, G, seed=4)
    qa, sa, _ = q8.q8_quantize_act(dev(a_np))
    qw, sf = q8.q8_quantize_weight_mx(dev(w_np), G)
    t = q8.q8_gemm_mx(qa, torch.ones(M, device="cuda"), qw, sf, G)
    y = q8.q8_gemm_mx(qa, sa, qw, sf, G)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    rng = np.random.default_rng(1)
    ns = np.unique(np.concatenate([rng.integers(0, N, 300), [0, N - 1]]))
    qa_s, sa_s = oracle.quantize_sym(a_np, per_row=True)
    qw_s, sf_s = oracle.quantize_weight_mx(w_np[ns], G)
    np.testing.assert_array_equal(host(qa), qa_s)
    np.testing.assert_array_equal(host(qw)[ns], qw_s)
    np.testing.assert_array_equal(host(sf)[:, ns], words(sf_s))
    t_ref, absum = oracle.gemm_mx(qa_s, qw_s, sf_s, G, threads=8)
    t_s = host(t)[:, ns]
    accumulation_gate(t_s, t_ref, absum, qa_s, qw_s, sf_s, G, order="decode")
    np.testing.assert_array_equal(host(y)[:, ns], (t_s * sa_s[:, None]).astype(np.float32))


def ulps_from(t, exact):
    """|t - exact| in units of the fp32 ulp of the exact value."""
    ex = np.abs(exact.astype(np.float64))
    ulp = np.exp2(np.floor(np.log2(np.maximum(ex, 2.0 ** -126))) - 23)
    return np.abs(t.astype(np.float64) - exact.astype(np.float64)) / ulp


@pytest.mark.parametrize("name,M,N,K,G", [("decode", 16, 2048, 8192, 32), ("prefill16k", 272, 264, 16384, 32),
                                         ("prefill16k", 272, 264, 16384, 128)])
def test_observed_error_of_the_tensor_core_sum(q8, name, M, N, K, G, capsys):
    """The observed error of T against the exactly rounded sum, in ulp of T, on the bench's
    statistics (activations of the workload, weights drawn like the bench's with E8M0 groups):
    reported, and held to the derived bound and to a small typical error."""
    wl = workloads.WORKLOADS[name]
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    qa, _ = oracle.quantize_sym(a, per_row=True)
    q, sf = oracle.quantize_weight_mx(w, G)
    t_ref, absum = oracle.gemm_mx(qa, q, sf, G, threads=8)
    t = host(q8.q8_gemm_mx(dev(qa), unit_scales(M), dev(q), dev(words(sf)), G))
    assert q8.q8_device_error() == 0
    err, bound = accumulation_gate(t, t_ref, absum, qa, q, sf, G, order="decode" if M <= 16 else "pair")
    u = ulps_from(t, t_ref)
    with capsys.disabled():
        print(f"\n[block-scaled T error] {name} M={M} N={N} K={K} G={G}: max {u.max():.1f} ulp, median "
              f"{np.median(u):.2f} ulp, exact {100 * np.mean(u == 0):.1f} %, max err / bound "
              f"{(err / bound).max():.3f}")
    assert np.median(u) <= 2.0
