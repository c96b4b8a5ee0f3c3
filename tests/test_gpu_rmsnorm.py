"""GPU parity of the fused RMSNorm + per-token quantization (q8_rmsnorm_quantize_act)
against the oracle ("Activation Quantization Architecture", Fusion pseudocode).

Reading shared by both sides: the sum of squares of a row is the exact sum rounded
once to fp32; everything after it is fp32 IEEE arithmetic in the order written. The
oracle forms the sum in long double, the kernel with error-free pair arithmetic, so
both round to the same fp32 value unless the exact sum lies on (within 2^-36 of) a
midpoint between two fp32 values, where either neighbour is a correct rounding. Rows
away from a midpoint must match bit for bit (codes and scales); a flagged row may
differ by one code step and a few ulp of scale.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gates

pytestmark = pytest.mark.gpu

EPS = 1e-6


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


def compare(qa, s_a, ref):
    # every row with a nonzero maximum has a code of magnitude exactly 127 (its maximum element,
    # whose value the code pass must see exactly as the range pass did)
    live = np.abs(ref["qa"]).max(axis=1) > 0 if ref["qa"].size else np.zeros(0, bool)
    if live.any():
        assert np.all(np.abs(qa[live].astype(np.int32)).max(axis=1) == 127)
    flag = gates.near_f32_midpoint(ref["sumsq"])
    ok = ~flag
    np.testing.assert_array_equal(s_a[ok], ref["sa"][ok])
    np.testing.assert_array_equal(qa[ok], ref["qa"][ok])
    if flag.any():
        assert int(gates.ulp_distance(s_a[flag], ref["sa"][flag]).max()) <= 4
        assert int(np.abs(qa[flag].astype(np.int32) - ref["qa"][flag]).max()) <= 1
    return int(flag.sum())


CASES = [
    # (M, K, workload the activations are shaped like): K spans every kernel tier
    (16, 256, "tiny"),
    (512, 2048, "prefill2k"),
    (33, 4112, "prefill2k"),      # 1028 float4 per row: two per thread
    (16, 8192, "decode"),
    (40, 8208, "relu4k"),         # four per thread
    (64, 16384, "prefill16k"),    # four per thread, 1024 threads
    (9, 20000, "prefill2k"),      # eight per thread
    (5, 40000, "prefill2k"),      # longer than the register budget: three sweeps
    (1, 16, "tiny"),
]


@pytest.mark.parametrize("M,K,name", CASES)
def test_rmsnorm_quantize_matches_oracle(q8, M, K, name):
    a = workloads.make_activations(workloads.WORKLOADS[name], M=M, K=K)
    if M > 2:
        a[M // 2] = 0.0                                  # a padding token: rms = sqrt(eps)
        a[1] *= np.float32(1e-3)                         # a row where eps is not negligible
    gamma = workloads.make_norm_weights(K, seed=M + K)
    qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), EPS)
    torch.cuda.synchronize()
    compare(host(qa), host(s_a), oracle.rmsnorm_quantize(a, gamma, EPS))


def test_rmsnorm_quantize_full_size(q8):
    # the measured configuration (the prefill16k activations, gamma seed 4, eps 1e-6): every row
    wl = workloads.WORKLOADS["prefill16k"]
    a = workloads.make_activations(wl)
    gamma = workloads.make_norm_weights(wl.K, seed=4)
    qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), EPS)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    compare(host(qa), host(s_a), oracle.rmsnorm_quantize(a, gamma, EPS))


def test_rmsnorm_constant_rows_exact(q8):
    # closed form: a row of c gives y = sign(c) gamma exactly when eps is negligible
    K = 512
    gamma = workloads.make_norm_weights(K, seed=9)
    a = np.stack([np.full(K, c, np.float32) for c in (3.0, -0.75, 12.0, 1.0)])
    qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), 1e-30)
    ref_q, ref_s = oracle.quantize_sym(np.sign(a) * gamma[None, :], per_row=True)
    np.testing.assert_array_equal(host(qa), ref_q)
    np.testing.assert_array_equal(host(s_a), ref_s)


def test_fused_then_gemm_matches_oracle_layer(q8):
    wl = workloads.WORKLOADS["prefill2k"]
    M, N, K = 300, 264, 2048
    a = workloads.make_activations(wl, M=M, K=K)
    w = workloads.make_weights(wl, N=N, K=K)
    gamma = workloads.make_norm_weights(K, seed=1)
    qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), EPS)
    qw, s_w = q8.q8_quantize_weight(dev(w), per_row=True)
    y = q8.q8_gemm_dequant(qa, s_a, None, qw, s_w)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_quantize(a, gamma, EPS)
    assert not gates.near_f32_midpoint(ref["sumsq"]).any()
    rqw, rsw = oracle.quantize_sym(w, per_row=True)
    ry, st = oracle.linear_codes(ref["qa"], ref["sa"], None, rqw, rsw, a_per_row=True, w_per_row=True)
    assert st == oracle.OK
    yi = host(y).view(np.int32).astype(np.int64)
    ri = ry.view(np.int32).astype(np.int64)
    assert np.max(np.abs(yi - ri)) <= 2


def test_rmsnorm_empty(q8):
    a = torch.empty((0, 64), dtype=torch.float32, device="cuda")
    g = torch.ones(64, dtype=torch.float32, device="cuda")
    qa, s_a = q8.q8_rmsnorm_quantize_act(a, g, EPS)
    assert qa.shape == (0, 64) and s_a.shape == (0,)


def test_rmsnorm_quotient_paths(q8):
    """Rows that take each path of the division x / rms: Markstein's corrected quotient (rms in
    [2^-60, 2^60], |x| >= 2^-60), the IEEE quotient for elements below 2^-60 (subnormal ones
    included) and for whole rows whose rms lies outside [2^-60, 2^60]; and signed zeros."""
    rng = np.random.default_rng(11)
    K = 4096
    rows = []
    mag = np.exp2(rng.uniform(-40.0, 40.0, K)) * rng.choice([-1.0, 1.0], K)   # quotients of every exponent
    rows.append(mag.astype(np.float32))
    r = rng.standard_normal(K).astype(np.float32)
    r[::7] = (rng.standard_normal(K)[::7] * 2.0 ** -70).astype(np.float32)      # tiny elements: IEEE path
    r[3], r[5] = np.float32(2.0 ** -60), np.nextafter(np.float32(2.0 ** -60), np.float32(0))
    r[11:13] = np.float32(1e-40)                                                # subnormal inputs
    rows.append(r)
    z = rng.standard_normal(K).astype(np.float32)
    z[::3] = np.float32(-0.0)
    z[1::3] = np.float32(0.0)
    rows.append(z)
    rows.append((rng.standard_normal(K) * 1e-3).astype(np.float32))
    a = np.stack(rows)
    gamma = workloads.make_norm_weights(K, seed=5)
    qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), EPS)
    torch.cuda.synchronize()
    compare(host(qa), host(s_a), oracle.rmsnorm_quantize(a, gamma, EPS))
    # whole rows with rms below 2^-60 and above 2^60 (values k * 2^-61 and k * 2^61 with short
    # mantissas, so every square and sum is exact and nothing under- or overflows)
    ks = rng.choice(np.array([1.0, 0.5, 0.75, 1.25, -1.0, -0.5, -0.75, -1.25]), size=(2, 64))
    for scale, Kx in ((2.0 ** -61, 64), (2.0 ** 61, 16)):
        b = np.stack([(ks[0, :Kx] * scale), rng.standard_normal(Kx)]).astype(np.float32)
        g = workloads.make_norm_weights(Kx, seed=Kx)
        qb, sb = q8.q8_rmsnorm_quantize_act(dev(b), dev(g), 1e-45)
        torch.cuda.synchronize()
        ref = oracle.rmsnorm_quantize(b, g, 1e-45)
        rms0 = np.sqrt(np.float64(ref["sumsq"][0]) / Kx)
        assert (rms0 < 2.0 ** -60) if scale < 1 else (rms0 > 2.0 ** 60)
        compare(host(qb), host(sb), ref)


@pytest.mark.parametrize("M,K", [(460, 4112), (320, 16384)])
def test_streaming_kernel_rows_with_every_path(q8, M, K):
    """Enough rows (>= two per SM) for the streaming kernel, with a ragged K (the general form) and
    with K = 16384 (512 threads of eight float4, no bounds checks): random rows, zero rows, rows
    with tiny elements (IEEE path), huge-range rows and eps-dominated rows, in an order that puts
    each kind into every shared-memory buffer slot."""
    rng = np.random.default_rng(21 + K)
    a = workloads.make_activations(workloads.WORKLOADS["prefill2k"], M=M, K=K)
    for r in range(0, M, 7):
        kind = (r // 7) % 5
        if kind == 0:
            a[r] = 0.0
        elif kind == 1:
            a[r, ::5] = (rng.standard_normal(K)[::5] * 2.0 ** -72).astype(np.float32)
        elif kind == 2:
            a[r] = (np.exp2(rng.uniform(-30.0, 30.0, K)) * rng.choice([-1.0, 1.0], K)).astype(np.float32)
        elif kind == 3:
            a[r] *= np.float32(1e-4)               # eps (1e-6) dominates the mean of squares
        else:
            a[r, ::3] = np.float32(-0.0)
    gamma = workloads.make_norm_weights(K, seed=3)
    for _ in range(2):
        qa, s_a = q8.q8_rmsnorm_quantize_act(dev(a), dev(gamma), EPS)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        compare(host(qa), host(s_a), oracle.rmsnorm_quantize(a, gamma, EPS))
