"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer results (codes, zero points, column sums, INT32 accumulators) and the
fp32 scales must be bit-identical; y must be within 2 ulp (the kernels use the
oracle's operation order, so 0 ulp is expected). Inputs are seeded, synthetic
and shaped like the workloads in workloads.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gates

pytestmark = pytest.mark.gpu

KERNELS = ("tcgen05", "tcgen05_pair", "mma_s8", "skinny", "decode", "decode_tc")


def runs(kernel, M):
    """Whether the kernel accepts M rows (the decode kernel takes M <= 16)."""
    return not kernel.startswith("decode") or M <= 16


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


def assert_no_device_error(q8):
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0


def max_ulp(a, b):
    return int(gates.ulp_distance(a, b).max()) if a.size else 0


# ---------------------------------------------------------------- quantizers

QUANT_CASES = [
    # (M, K, per_row, symmetric, maker)
    (16, 256, False, True, "tiny"),
    (512, 2048, True, True, "prefill2k"),
    (2048, 4096, True, False, "relu4k"),
    (16, 8192, True, True, "decode"),
    (64, 16384, True, True, "prefill16k"),
    (37, 528, True, False, "prefill2k"),       # ragged K per thread block
    (5, 40000, True, True, "prefill2k"),       # rows longer than the register budget
    (3, 40000, True, False, "relu4k"),
    (300, 48, False, False, "relu4k"),         # per-tensor asymmetric (one-CTA kernel)
    (1, 16, True, True, "tiny"),
    (7, 1040, False, True, "prefill2k"),
    (32, 1024, False, True, "prefill2k"),      # per-tensor, exactly 8192 float4: the one-CTA kernel
    (33, 1008, False, True, "prefill2k"),      # per-tensor, 8316 float4: range, parameter and code kernels
    (512, 2048, False, False, "relu4k"),       # per-tensor asymmetric over the grid
]


@pytest.mark.parametrize("M,K,per_row,sym,name", QUANT_CASES)
def test_quantize_act_bit_exact(q8, M, K, per_row, sym, name):
    a = workloads.make_activations(workloads.WORKLOADS[name], M=M, K=K)
    a[M // 2] = 0.0                                     # an all-zero row (padding token)
    if M > 2:
        a[1] = -np.abs(a[1])                            # a non-positive row
    qa, s_a, z_a = q8.q8_quantize_act(dev(a), per_row=per_row, symmetric=sym)
    if sym:
        rq, rs = oracle.quantize_sym(a, per_row)
    else:
        rq, rs, rz = oracle.quantize_asym(a, per_row)
        np.testing.assert_array_equal(host(z_a), rz)
    np.testing.assert_array_equal(host(s_a), rs)
    np.testing.assert_array_equal(host(qa), rq)


def test_rounding_ties_on_gpu(q8):
    x = np.array([[127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -1.5, -127.0] + [0.0] * 7,
                  [0.881577730178833, 0.7115095853805542] + [0.0] * 14,
                  [3.754473924636841, 0.10346975177526474] + [0.0] * 14], np.float32)
    qa, s_a, _ = q8.q8_quantize_act(dev(x), per_row=True)
    q = host(qa)
    assert q[0, :9].tolist() == [127, 2, 4, -2, 0, 2, 0, -2, -127]
    assert q[1, 1] == 102 and q[2, 1] == 4


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("N,K", [(128, 256), (2048, 2048), (1000, 4112)])
def test_quantize_weight_and_colsum_bit_exact(q8, per_row, N, K):
    w = workloads.make_weights(workloads.WORKLOADS["prefill2k"], N=N, K=K)
    qw, s_w = q8.q8_quantize_weight(dev(w), per_row=per_row)
    cs = q8.q8_colsum(qw)
    rq, rs = oracle.quantize_sym(w, per_row)
    np.testing.assert_array_equal(host(s_w), rs)
    np.testing.assert_array_equal(host(qw), rq)
    np.testing.assert_array_equal(host(cs).astype(np.int64), oracle.colsum(rq))


def test_colsum_extreme_codes(q8):
    qw = np.full((9, 131056), -128, np.int8)
    qw[3] = 127
    cs = q8.q8_colsum(dev(qw))
    np.testing.assert_array_equal(host(cs).astype(np.int64), oracle.colsum(qw))


# ---------------------------------------------------------------- integer GEMM

GEMM_SHAPES = [
    (1, 1, 16), (16, 128, 256), (128, 256, 1024), (200, 264, 1088), (129, 257, 1040),
    (300, 520, 2064), (17, 1000, 4096), (256, 512, 3072), (64, 96, 48),
    (16, 28672, 8192), (5, 1000, 1040), (16, 65, 16), (11, 4100, 3200),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_s32_bit_exact(q8, kernel, M, N, K):
    qa = workloads.random_codes((M, K), seed=M * 7 + K)
    qw = workloads.random_codes((N, K), seed=N * 11 + K)
    if not runs(kernel, M):
        with pytest.raises(q8.Q8Error) as ex:
            q8.q8_gemm_s32(dev(qa), dev(qw), kernel=kernel)
        assert ex.value.status == q8.Q8_ERR_UNSUPPORTED
        return
    acc = q8.q8_gemm_s32(dev(qa), dev(qw), kernel=kernel)
    assert_no_device_error(q8)
    np.testing.assert_array_equal(host(acc).astype(np.int64), oracle.gemm_acc(qa, qw, threads=8))


@pytest.mark.parametrize("M,N,K,reps", [(1024, 1024, 4096, 10), (2048, 2048, 8192, 4)])
def test_gemm_s32_repeatable_under_load(q8, M, N, K, reps):
    """Many tiles per CTA and deep K: every repetition must be bit-exact. Pipeline races
    (a staging slot refilled before its reads completed) show up here as whole tile rows
    whose k-block was replaced by a later one."""
    qa = workloads.random_codes((M, K), seed=M * 7 + K)
    qw = workloads.random_codes((N, K), seed=N * 11 + K)
    ref = oracle.gemm_acc(qa, qw, threads=16)
    da, dw = dev(qa), dev(qw)
    for _ in range(reps):
        for kernel in ("tcgen05", "tcgen05_pair"):
            acc = host(q8.q8_gemm_s32(da, dw, kernel=kernel)).astype(np.int64)
            assert_no_device_error(q8)
            np.testing.assert_array_equal(acc, ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_gemm_s32_extreme_codes(q8, kernel):
    """-128 * -128 products everywhere: every fp32 chunk sum sits exactly on 2^24."""
    M, N, K = (16 if kernel.startswith("decode") else 160), 300, 16384
    qa = np.full((M, K), -128, np.int8)
    qw = np.full((N, K), -128, np.int8)
    qw[1::2] = 127
    acc = host(q8.q8_gemm_s32(dev(qa), dev(qw), kernel=kernel)).astype(np.int64)
    assert_no_device_error(q8)
    expect = np.where(np.arange(N) % 2 == 0, K * 16384, -K * 128 * 127)
    np.testing.assert_array_equal(acc, np.broadcast_to(expect, (M, N)))


def test_decode_largest_k_extreme_codes(q8):
    """The decode kernel offsets weight codes by 128: at the largest K its int32 tile sums of
    a (w + 128) pass 2^31 and wrap, and the result must still be exact."""
    M, N, K = 16, 72, 131056
    rng = np.random.default_rng(K)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-128, 128, (N, K), dtype=np.int8)
    qa[0], qa[1] = -128, 127
    qw[0], qw[1], qw[2] = 127, -128, 127
    acc = host(q8.q8_gemm_s32(dev(qa), dev(qw), kernel="decode")).astype(np.int64)
    assert_no_device_error(q8)
    want = oracle.gemm_acc(qa, qw, threads=8)
    assert want[0, 0] == -128 * 127 * K and want[0, 1] == 16384 * K and want[1, 2] == 127 * 127 * K
    np.testing.assert_array_equal(acc, want)


@pytest.mark.parametrize("kernel", KERNELS)
def test_gemm_s32_small_terms_next_to_large_partial_sums(q8, kernel):
    """Each 1024-deep chunk first climbs to ~2^24 with -128*-128 products, then adds +-1
    and +-127 terms: an accumulator that kept fewer than 24 significant bits would drop them."""
    M, N, K = (16 if kernel.startswith("decode") else 130), 260, 4096
    rng = np.random.Generator(np.random.PCG64(5))
    qa = np.zeros((M, K), np.int8)
    qw = np.zeros((N, K), np.int8)
    for c0 in range(0, K, 1024):
        big = 1000
        qa[:, c0:c0 + big] = -128
        qw[:, c0:c0 + big] = -128
        qa[:, c0 + big:c0 + 1024] = rng.integers(-128, 128, size=(M, 1024 - big))
        qw[:, c0 + big:c0 + 1024] = rng.choice(np.array([-1, 1, 127, -127], np.int8), size=(N, 1024 - big))
    acc = host(q8.q8_gemm_s32(dev(qa), dev(qw), kernel=kernel)).astype(np.int64)
    assert_no_device_error(q8)
    np.testing.assert_array_equal(acc, oracle.gemm_acc(qa, qw, threads=8))


# ---------------------------------------------------------------- GEMM + epilogue

LAYER_CASES = [
    # name, M, N, K, act_per_row, act_sym, w_per_row
    ("tiny", 16, 128, 256, False, True, False),
    ("decode", 7, 3000, 2064, True, False, True),
    ("prefill2k", 200, 264, 1088, True, True, True),
    ("relu4k", 333, 520, 2048, True, False, True),
    ("decode", 16, 1000, 8192, True, True, True),
    ("relu4k", 129, 256, 1040, False, False, True),
    ("prefill2k", 64, 300, 528, True, True, False),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name,M,N,K,apr,asym_is_sym,wpr", LAYER_CASES)
def test_linear_layer_matches_oracle(q8, kernel, name, M, N, K, apr, asym_is_sym, wpr):
    if not runs(kernel, M):
        pytest.skip("the decode kernel takes M <= 16")
    wl = workloads.WORKLOADS[name]
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    ref = oracle.linear(a, w, apr, asym_is_sym, wpr, threads=8)
    assert ref["status"] == oracle.OK
    qw, s_w = q8.q8_quantize_weight(dev(w), per_row=wpr)
    cs = q8.q8_colsum(qw)
    qa, s_a, z_a = q8.q8_quantize_act(dev(a), per_row=apr, symmetric=asym_is_sym)
    y = host(q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, cs, kernel=kernel))
    assert_no_device_error(q8)
    np.testing.assert_array_equal(host(qa), ref["qa"])
    assert max_ulp(y, ref["y"]) <= 2
    # and the layer still honours the page's per-column gate against fp64
    if wpr:
        err = np.abs(y - gates.reference_fp64(a, w))
        assert gates.first_violation(err, gates.column_gate_atol(a, w, apr)) is None


@pytest.mark.parametrize("kernel", KERNELS)
def test_epilogue_with_random_scales_and_zero_points(q8, kernel):
    M, N, K = (13 if kernel.startswith("decode") else 150), 280, 1536
    qa = workloads.random_codes((M, K), seed=40)
    qw = workloads.random_codes((N, K), seed=41, lo=-127)
    sa = workloads.random_scales(M, seed=42)
    sw = workloads.random_scales(N, seed=43)
    za = workloads.random_zero_points(M, seed=44)
    cs = oracle.colsum(qw).astype(np.int32)
    y = host(q8.q8_gemm_dequant(dev(qa), dev(sa), dev(za), dev(qw), dev(sw), dev(cs), kernel=kernel))
    ry, st = oracle.linear_codes(qa, sa, za, qw, sw, True, True, threads=8)
    assert st == oracle.OK
    assert max_ulp(y, ry) <= 2


def test_empty_problems(q8):
    z = torch.zeros(0, 32, dtype=torch.int8, device="cuda")
    w = torch.zeros(8, 32, dtype=torch.int8, device="cuda")
    s = torch.ones(8, dtype=torch.float32, device="cuda")
    y = q8.q8_gemm_dequant(z, torch.ones(1, device="cuda"), None, w, s)
    assert y.shape == (0, 8)
    qa0 = torch.zeros(4, 0, dtype=torch.int8, device="cuda")
    qw0 = torch.zeros(8, 0, dtype=torch.int8, device="cuda")
    y0 = q8.q8_gemm_dequant(qa0, torch.ones(4, device="cuda"), None, qw0, s)
    assert torch.count_nonzero(y0).item() == 0 and not torch.signbit(y0).any()
    qa, s_a, _ = q8.q8_quantize_act(torch.zeros(3, 0, device="cuda"))
    assert torch.all(s_a == torch.tensor(np.float32(np.float32(1e-8) / np.float32(127)), device="cuda"))


def test_launch_counter_counts_our_kernels(q8):
    before = q8.q8_launch_count()
    a = torch.randn(64, 256, device="cuda")
    qa, s_a, _ = q8.q8_quantize_act(a)
    qw, s_w = q8.q8_quantize_weight(torch.randn(128, 256, device="cuda"))
    q8.q8_gemm_dequant(qa, s_a, None, qw, s_w, kernel="tcgen05")
    assert q8.q8_launch_count() - before == 3


# ---------------------------------------------------------------- full-size workloads

FULL = ["tiny", "prefill2k", "relu4k", "decode", "prefill16k"]


def _sample_pairs(M, N, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    ms = np.concatenate([rng.integers(0, M, count), [0, M - 1, 0, M - 1, min(127, M - 1), min(128, M - 1)]])
    ns = np.concatenate([rng.integers(0, N, count), [0, N - 1, N - 1, 0, min(255, N - 1), min(256, N - 1)]])
    return ms.astype(np.int64), ns.astype(np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(q8, name):
    """The bench's launch configuration (kernel chosen by q8_gemm_pick, the layer's workspace where
    the shape takes one) at the workload's full size: every code, scale and zero point bit-exact;
    y and the INT32 accumulators compared with the threaded oracle at every output, except for the
    large prefill (1.1e12 multiply-adds), where they are compared on 16 whole rows, 16 whole columns
    and 3000 sampled outputs; the layer with and without the workspace bit-identical, and (the
    bench's step) with the quantizer writing the codes' fp16 copy itself."""
    wl = workloads.WORKLOADS[name]
    a = workloads.make_activations(wl)
    w = workloads.make_weights(wl)
    apr, wpr = wl.act_granularity == "row", wl.w_granularity == "row"
    if wl.act_symmetric:
        (rqa, rsa), rza = oracle.quantize_sym(a, apr), None
    else:
        rqa, rsa, rza = oracle.quantize_asym(a, apr)
    rqw, rsw = oracle.quantize_sym(w, wpr)
    a_d, w_d = dev(a), dev(w)
    del a
    qw, s_w = q8.q8_quantize_weight(w_d, per_row=wpr)
    del w_d
    cs = q8.q8_colsum(qw)
    qa, s_a, z_a = q8.q8_quantize_act(a_d, per_row=apr, symmetric=wl.act_symmetric)
    nws = q8.q8_gemm_workspace(wl.M, wl.N, wl.K)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda") if nws else None
    y = q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, cs, workspace=ws)
    y_direct = q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, cs)
    acc = q8.q8_gemm_s32(qa, qw)
    assert_no_device_error(q8)
    assert torch.equal(y.view(torch.int32), y_direct.view(torch.int32))
    del y_direct
    if ws is not None:   # the bench's step: the quantizer writes the fp16 copy, the pair kernel reads it
        ws16 = ws.view(torch.float16)[:wl.M * wl.K].view(wl.M, wl.K)
        ws.fill_(0x55)
        qa2, _, s_a2, z_a2 = q8.q8_quantize_act_dual(a_d, per_row=apr, symmetric=wl.act_symmetric, qa16=ws16)
        y_step = q8.q8_gemm_f16a(ws16, s_a2, z_a2, qw, s_w, cs)
        assert_no_device_error(q8)
        assert torch.equal(qa2, qa) and torch.equal(s_a2.view(torch.int32), s_a.view(torch.int32))
        assert torch.equal(y_step.view(torch.int32), y.view(torch.int32))
        del y_step, qa2
    np.testing.assert_array_equal(host(s_a), rsa)
    np.testing.assert_array_equal(host(qa), rqa)
    if rza is not None:
        np.testing.assert_array_equal(host(z_a), rza)
    np.testing.assert_array_equal(host(s_w), rsw)
    np.testing.assert_array_equal(host(qw), rqw)
    np.testing.assert_array_equal(host(cs).astype(np.int64), oracle.colsum(rqw))
    if name != "prefill16k":
        threads = oracle.max_threads()
        ry, st = oracle.linear_codes(rqa, rsa, rza, rqw, rsw, apr, wpr, threads=threads)
        assert st == oracle.OK
        assert max_ulp(host(y), ry) <= 2
        np.testing.assert_array_equal(host(acc).astype(np.int64), oracle.gemm_acc(rqa, rqw, threads=threads))
        return
    ms, ns = _sample_pairs(wl.M, wl.N, 3000, seed=wl.seed)
    ry, racc, st = oracle.linear_codes_at(rqa, rsa, rza, rqw, rsw, ms, ns, apr, wpr)
    assert st == oracle.OK
    yt, acct = torch.as_tensor(ms).cuda(), torch.as_tensor(ns).cuda()
    np.testing.assert_array_equal(host(acc[yt, acct]).astype(np.int64), racc)
    assert max_ulp(host(y[yt, acct]), ry) <= 2
    # whole rows (every N-tile) and whole columns (every M-tile)
    rng = np.random.default_rng(wl.seed + 17)
    rows = np.unique(np.concatenate([rng.integers(0, wl.M, 14), [0, wl.M - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, wl.N, 14), [0, wl.N - 1]]))
    threads = oracle.max_threads()
    ry_r, st = oracle.linear_codes(rqa[rows], rsa[rows] if apr else rsa, None, rqw, rsw, apr, wpr, threads=threads)
    assert st == oracle.OK
    yh, acch = host(y), host(acc)
    assert max_ulp(yh[rows], ry_r) <= 2
    np.testing.assert_array_equal(acch[rows].astype(np.int64), oracle.gemm_acc(rqa[rows], rqw, threads=threads))
    ry_c, st = oracle.linear_codes(rqa, rsa, None, rqw[cols], rsw[cols] if wpr else rsw, apr, wpr, threads=threads)
    assert st == oracle.OK
    assert max_ulp(yh[:, cols], ry_c) <= 2
    np.testing.assert_array_equal(acch[:, cols].astype(np.int64), oracle.gemm_acc(rqa, rqw[cols], threads=threads))


@pytest.mark.slow
def test_full_size_worst_case_codes(q8):
    """Large prefill shape with raw codes at the int8 extremes: every acc equals the closed
    form, K * (-128) * (-127), the accumulator bound of Day 98."""
    wl = workloads.WORKLOADS["prefill16k"]
    qa = torch.full((wl.M, wl.K), -128, dtype=torch.int8, device="cuda")
    qw = torch.full((wl.N, wl.K), -127, dtype=torch.int8, device="cuda")
    acc = q8.q8_gemm_s32(qa, qw)
    assert_no_device_error(q8)
    assert torch.all(acc == wl.K * 16256).item()
    assert wl.K * 16256 == 266338304


@pytest.mark.parametrize("kernel", ["tcgen05_pair", "tcgen05", "mma_s8"])
def test_prefill_kernels_at_the_largest_k(q8, kernel):
    """K = 131056, the largest symmetric K the API takes: -128 * -128 on every k brings the INT32
    accumulator to 16384 * 131056 = 2^31 - 2^18 through 128 exact fp32 chunks (tensor-core
    kernels); other rows mix in +127 and random codes."""
    M, N, K = 130, 260, 131056
    rng = np.random.default_rng(11)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-128, 128, (N, K), dtype=np.int8)
    qa[0] = -128
    qw[0] = -128
    qw[1] = 127
    acc = host(q8.q8_gemm_s32(dev(qa), dev(qw), kernel=kernel)).astype(np.int64)
    assert_no_device_error(q8)
    want = oracle.gemm_acc(qa, qw, threads=8)
    assert want[0, 0] == 16384 * K and want[0, 1] == -128 * 127 * K
    np.testing.assert_array_equal(acc, want)


# Shapes whose pair-kernel grid would leave most clusters idle: the kernel then splits K into
# 2, 4 or 8 slices whose INT32 partial sums are added by TMA reduce-add (into y's storage for fp32
# output, followed by the in-place epilogue). (M, N, K, expected slices on 76 resident pairs.)
SPLIT_CASES = [(300, 520, 4096, 8), (512, 2048, 2048, 4), (16, 1024, 8192, 8), (257, 2052, 1024, 2)]


@pytest.mark.parametrize("M,N,K,_slices", SPLIT_CASES)
def test_k_split_pair_kernel_is_exact(q8, M, N, K, _slices):
    rng = np.random.default_rng(M + N + K)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    want = oracle.gemm_acc(qa, qw, threads=8)
    acc = host(q8.q8_gemm_s32(dev(qa), dev(qw), kernel="tcgen05_pair")).astype(np.int64)
    assert_no_device_error(q8)
    np.testing.assert_array_equal(acc, want)
    # the fp32 layer with asymmetric activations (zero points, column sums), and with a bias
    sa = (rng.random(M, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    sw = (rng.random(N, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    za = rng.integers(-128, 128, M, dtype=np.int32)
    cs = q8.q8_colsum(dev(qw))
    y = host(q8.q8_gemm_dequant(dev(qa), dev(sa), dev(za), dev(qw), dev(sw), cs, kernel="tcgen05_pair"))
    assert_no_device_error(q8)
    y_ref, st = oracle.linear_codes(qa, sa, za, qw, sw, True, True, threads=8)
    assert st == oracle.OK
    np.testing.assert_array_equal(y.view(np.int32), y_ref.view(np.int32))
    bias = rng.standard_normal(N, dtype=np.float32)
    yb = host(q8.q8_gemm_epilogue(dev(qa), dev(sa), dev(za), dev(qw), dev(sw), cs, bias=dev(bias),
                                  kernel="tcgen05_pair"))
    assert_no_device_error(q8)
    yb_ref, st = oracle.linear_codes_bias(qa, sa, za, qw, sw, bias, True, True, threads=8)
    np.testing.assert_array_equal(yb.view(np.int32), yb_ref.view(np.int32))


@pytest.mark.parametrize("apr,wpr", [(False, False), (True, False), (False, True)])
def test_k_split_with_per_tensor_scales_and_int4_weights(q8, apr, wpr):
    # 512 x 2048 x 2048 splits K in 4 on the pair kernel: per-tensor activation and weight scales
    # through the in-place epilogue, and the same split with packed int4 weights
    M, N, K = 512, 2048, 2048
    rng = np.random.default_rng(17 + 2 * apr + wpr)
    qa = rng.integers(-128, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    sa = (rng.random(M if apr else 1, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    sw = (rng.random(N if wpr else 1, dtype=np.float32) + np.float32(0.5)) * np.float32(1e-2)
    za = rng.integers(-128, 128, M if apr else 1, dtype=np.int32)
    y = host(q8.q8_gemm_dequant(dev(qa), dev(sa), dev(za), dev(qw), dev(sw), q8.q8_colsum(dev(qw)),
                                kernel="tcgen05_pair"))
    assert_no_device_error(q8)
    y_ref, st = oracle.linear_codes(qa, sa, za, qw, sw, apr, wpr, threads=8)
    assert st == oracle.OK
    np.testing.assert_array_equal(y.view(np.int32), y_ref.view(np.int32))
    q4 = rng.integers(-8, 8, (N, K), dtype=np.int8)
    acc4 = host(q8.q8_gemm_w4a8_s32(dev(qa), dev(oracle.pack_int4(q4)), kernel="tcgen05_pair")).astype(np.int64)
    assert_no_device_error(q8)
    np.testing.assert_array_equal(acc4, oracle.gemm_acc(qa, q4, threads=8))


@pytest.mark.parametrize("symmetric", [True, False])
@pytest.mark.parametrize("per_row", [True, False])
def test_codes_next_to_half_integer_quotients(q8, symmetric, per_row):
    """Values whose quotient x / s lies on a half-integer or within a few ulp of one (and farther
    out) under random scales: the quantizer multiplies by the row's reciprocal and falls back to the
    IEEE quotient near half-integers, so every code must still equal the oracle's (IEEE division,
    round half to even)."""
    rng = np.random.default_rng(99 + 2 * symmetric + per_row)
    rows, cols = 64, 1024
    x = np.zeros((rows, cols), np.float32)
    offsets = np.array([0.0, 1e-7, -1e-7, 6e-6, -6e-6, 3e-5, -3e-5, 6.2e-5, -6.2e-5, 2e-4, -2e-4, 0.25],
                       np.float64)
    for r in range(rows):
        amax = np.float32(np.exp(rng.uniform(np.log(1e-3), np.log(1e3))))
        s = np.float32(amax / np.float32(127.0)) if symmetric else np.float32(amax / np.float32(255.0))
        k = rng.integers(-126, 126, cols - 2)
        q = (k + 0.5 + rng.choice(offsets, cols - 2)) * np.float64(s)
        if not symmetric:
            q = np.abs(q)                         # one-signed row: lo = 0, codes span 0 .. 255
        x[r, 2:] = np.clip(q, -amax, amax).astype(np.float32)
        x[r, 0] = amax
        x[r, 1] = -amax if symmetric else 0.0
    if symmetric:
        qa, sa, _ = q8.q8_quantize_act(dev(x), per_row=per_row)
        q_ref, s_ref = oracle.quantize_sym(x, per_row)
    else:
        qa, sa, za = q8.q8_quantize_act(dev(x), per_row=per_row, symmetric=False)
        q_ref, s_ref, z_ref = oracle.quantize_asym(x, per_row)
        np.testing.assert_array_equal(host(za), z_ref)
    np.testing.assert_array_equal(host(sa), s_ref)
    np.testing.assert_array_equal(host(qa), q_ref)
