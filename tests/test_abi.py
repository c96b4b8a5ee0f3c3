"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU. These
calls never launch a kernel (validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8.h")


@pytest.fixture(scope="module")
def lib():
    from int8_quantized_gemm_gb300 import build
    build.build()
    import int8_quantized_gemm_gb300 as q8
    return q8.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\*?\s+\**(q8_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q8_quantize_act", "q8_quantize_weight", "q8_colsum", "q8_gemm_dequant",
                     "q8_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in q8.h but not exported"


def test_status_strings(lib):
    for s in range(5):
        assert lib.q8_status_string(s)
    assert lib.q8_status_string(99) == b"unknown status"


P = ctypes.c_void_p
FAKE = P(0x10000)          # 16-byte aligned, never dereferenced: validation fails first
MISALIGNED = P(0x10004)


def gemm(lib, qa=FAKE, sa=FAKE, za=None, ga=1, qw=FAKE, sw=FAKE, gw=1, cs=None, M=8, N=8, K=16,
         y=FAKE, kernel=0):
    return lib.q8_gemm_dequant_ex(qa, sa, za, ga, qw, sw, gw, cs, M, N, K, y, kernel, None)


def test_gemm_rejects_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    assert gemm(lib, qa=None) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, y=None) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, sa=None) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, M=-1) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, ga=7) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, kernel=9) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, qa=MISALIGNED) == q8.Q8_ERR_INVALID_ARG
    assert gemm(lib, za=FAKE, cs=None) == q8.Q8_ERR_INVALID_ARG     # asymmetric A needs colsum
    assert gemm(lib, K=24) == q8.Q8_ERR_UNSUPPORTED                # K % 16
    assert gemm(lib, K=131072) == q8.Q8_ERR_UNSUPPORTED            # 128*128*K would leave int32
    assert gemm(lib, K=65808, za=FAKE, cs=FAKE) == q8.Q8_ERR_UNSUPPORTED
    # empty problems are valid and launch nothing
    before = lib.q8_launch_count()
    assert gemm(lib, M=0) == q8.Q8_OK
    assert gemm(lib, N=0) == q8.Q8_OK
    assert lib.q8_launch_count() == before


def test_rmsnorm_quantize_rejects_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    f = lambda a, g, M, K, eps, qa, sa: lib.q8_rmsnorm_quantize_act(a, g, M, K, ctypes.c_float(eps), qa, sa, None)
    assert f(FAKE, FAKE, 0, 32, 1e-6, FAKE, FAKE) == q8.Q8_OK                       # empty: nothing enqueued
    assert f(FAKE, FAKE, 4, 32, 0.0, FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG           # eps must be > 0
    assert f(FAKE, FAKE, 4, 32, float("inf"), FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 32, float("nan"), FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG
    assert f(FAKE, FAKE, -1, 32, 1e-6, FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 0, 1e-6, FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG           # mean over no elements
    assert f(FAKE, None, 4, 32, 1e-6, FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG          # gamma required
    assert f(FAKE, MISALIGNED, 4, 32, 1e-6, FAKE, FAKE) == q8.Q8_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 24, 1e-6, FAKE, FAKE) == q8.Q8_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 4, (1 << 24) + 16, 1e-6, FAKE, FAKE) == q8.Q8_ERR_UNSUPPORTED


def test_epilogue_variant_rejects_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8

    def f(out_type=0, out=FAKE, scale=0.0, bias=None, K=16):
        return lib.q8_gemm_epilogue_ex(FAKE, FAKE, None, 1, FAKE, FAKE, 1, None, bias, 8, 8, K, out_type, out,
                                       ctypes.c_float(scale), 0, None)
    assert f(out_type=3) == q8.Q8_ERR_INVALID_ARG                  # unknown output type
    assert f(out_type=2, scale=0.0) == q8.Q8_ERR_INVALID_ARG       # int8 output needs a scale > 0
    assert f(out_type=2, scale=float("inf")) == q8.Q8_ERR_INVALID_ARG
    assert f(out=None) == q8.Q8_ERR_INVALID_ARG
    assert f(out=MISALIGNED) == q8.Q8_ERR_INVALID_ARG
    assert f(bias=P(0x10002)) == q8.Q8_ERR_INVALID_ARG            # bias must be 4-byte aligned
    assert f(K=24) == q8.Q8_ERR_UNSUPPORTED


def test_block_scaled_entries_reject_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8

    def g(group=32, K=64, kernel=0, sf=FAKE, sa=FAKE, out=FAKE, M=8, N=8):
        return lib.q8_gemm_mx_ex(FAKE, sa, 1, FAKE, sf, group, None, M, N, K, 0, out, ctypes.c_float(0.0),
                                 kernel, None)
    assert g(group=64) == q8.Q8_ERR_INVALID_ARG                   # the granularity is 32 or 128
    assert g(group=0) == q8.Q8_ERR_INVALID_ARG
    assert g(K=48) == q8.Q8_ERR_UNSUPPORTED                       # K % group
    assert g(group=128, K=192) == q8.Q8_ERR_UNSUPPORTED
    assert g(kernel=q8.KERNELS["mma_s8"]) == q8.Q8_ERR_UNSUPPORTED      # pair or decode kernels only
    assert g(sf=None) == q8.Q8_ERR_INVALID_ARG
    assert g(sf=P(0x10002)) == q8.Q8_ERR_INVALID_ARG
    assert g(sa=None) == q8.Q8_ERR_INVALID_ARG
    assert g(out=None) == q8.Q8_ERR_INVALID_ARG
    before = lib.q8_launch_count()
    assert g(M=0) == q8.Q8_OK and g(N=0) == q8.Q8_OK
    assert lib.q8_launch_count() == before
    w = lambda N, K, group, qw=FAKE, sf=FAKE: lib.q8_quantize_weight_mx(FAKE, N, K, group, qw, sf, None)
    assert w(4, 64, 16) == q8.Q8_ERR_INVALID_ARG
    assert w(4, 96, 64) == q8.Q8_ERR_INVALID_ARG
    assert w(4, 160, 128) == q8.Q8_ERR_UNSUPPORTED
    assert w(4, 64, 32, sf=None) == q8.Q8_ERR_INVALID_ARG
    assert w(4, 64, 32, qw=MISALIGNED) == q8.Q8_ERR_INVALID_ARG
    assert w(-1, 64, 32) == q8.Q8_ERR_INVALID_ARG
    assert w(0, 64, 32) == q8.Q8_OK


def test_fp16_code_entries_reject_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    q = lib.q8_quantize_act_f16
    assert q(FAKE, 4, 32, 1, 0, FAKE, FAKE, FAKE, None) == q8.Q8_ERR_INVALID_ARG   # z_a given for symmetric
    assert q(FAKE, 4, 32, 1, 1, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG   # z_a missing for asymmetric
    assert q(FAKE, 4, 32, 1, 0, None, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG   # codes required
    assert q(FAKE, 4, 32, 1, 0, MISALIGNED, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG
    assert q(FAKE, 4, 24, 1, 0, FAKE, FAKE, None, None) == q8.Q8_ERR_UNSUPPORTED
    assert q(FAKE, 0, 32, 1, 0, FAKE, FAKE, None, None) == q8.Q8_OK

    def g(qa=FAKE, sa=FAKE, za=None, cs=None, out=FAKE, out_type=0, K=16, M=8, N=8):
        return lib.q8_gemm_f16a_ex(qa, sa, za, 1, FAKE, FAKE, 1, cs, None, M, N, K, out_type, out,
                                   ctypes.c_float(0.0), None)
    assert g(qa=None) == q8.Q8_ERR_INVALID_ARG
    assert g(qa=MISALIGNED) == q8.Q8_ERR_INVALID_ARG
    assert g(sa=None) == q8.Q8_ERR_INVALID_ARG
    assert g(out=None) == q8.Q8_ERR_INVALID_ARG
    assert g(za=FAKE) == q8.Q8_ERR_INVALID_ARG                    # asymmetric A needs colsum
    assert g(out_type=2) == q8.Q8_ERR_INVALID_ARG                 # int8 output needs a scale
    assert g(K=24) == q8.Q8_ERR_UNSUPPORTED
    assert g(K=131072) == q8.Q8_ERR_UNSUPPORTED
    before = lib.q8_launch_count()
    assert g(M=0) == q8.Q8_OK and g(N=0) == q8.Q8_OK
    assert lib.q8_launch_count() == before
    s32 = lib.q8_gemm_f16a_s32
    assert s32(FAKE, FAKE, 8, 8, 16, None, None) == q8.Q8_ERR_INVALID_ARG
    assert s32(FAKE, FAKE, 8, 8, 16, MISALIGNED, None) == q8.Q8_ERR_INVALID_ARG
    assert s32(FAKE, FAKE, 8, 8, 40, FAKE, None) == q8.Q8_ERR_UNSUPPORTED


def test_k_limits_are_the_int32_bounds():
    # 128*128*K < 2^31 for raw codes; 255*128*K < 2^31 with a zero point.
    assert 128 * 128 * 131056 < 2 ** 31 <= 128 * 128 * (131056 + 16)
    assert 255 * 128 * 65792 < 2 ** 31 <= 255 * 128 * (65792 + 16)


def test_quantize_rejects_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    q = lib.q8_quantize_act
    assert q(FAKE, 4, 32, 1, 0, FAKE, FAKE, FAKE, None) == q8.Q8_ERR_INVALID_ARG   # z_a given for symmetric
    assert q(FAKE, 4, 32, 1, 1, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG   # z_a missing for asymmetric
    assert q(FAKE, 4, 32, 1, 2, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG   # bad symmetry
    assert q(FAKE, 4, 32, 5, 0, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG   # bad granularity
    assert q(None, 4, 32, 1, 0, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG
    assert q(FAKE, 4, 24, 1, 0, FAKE, FAKE, None, None) == q8.Q8_ERR_UNSUPPORTED
    assert q(MISALIGNED, 4, 32, 1, 0, FAKE, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG
    assert q(FAKE, 0, 32, 1, 0, FAKE, FAKE, None, None) == q8.Q8_OK
    w = lib.q8_quantize_weight
    assert w(FAKE, 4, 32, 1, None, FAKE, None) == q8.Q8_ERR_INVALID_ARG
    assert w(FAKE, 4, 40, 1, FAKE, FAKE, None) == q8.Q8_ERR_UNSUPPORTED
    assert lib.q8_colsum(FAKE, 4, 32, None, None) == q8.Q8_ERR_INVALID_ARG
    assert lib.q8_colsum(FAKE, 4, 20, FAKE, None) == q8.Q8_ERR_UNSUPPORTED


def test_kernel_pick_is_a_concrete_kernel(lib):
    import int8_quantized_gemm_gb300 as q8
    for shape in ((16, 28672, 8192), (8192, 8192, 16384), (1, 1, 16), (513, 100, 48)):
        assert q8.q8_gemm_pick(*shape) in ("tcgen05", "tcgen05_pair", "mma_s8", "skinny", "decode")
    assert q8.q8_gemm_pick(16, 28672, 8192) == "decode"
    assert q8.q8_gemm_pick(8192, 8192, 16384) == "tcgen05_pair"
    assert q8.q8_gemm_pick(2048, 4096, 4096) == "tcgen05_pair"
    assert q8.q8_gemm_pick(17, 4096, 4096) == "tcgen05_pair"
    assert q8.q8_gemm_pick(300, 1000, 1024) == "tcgen05_pair"
    assert q8.q8_gemm_pick(100, 2048, 2048) == "skinny"


def test_gemm_workspace_sizes(lib):
    import int8_quantized_gemm_gb300 as q8
    # an fp16 copy of the activation codes for shapes on the CTA-pair kernel, nothing otherwise
    assert q8.q8_gemm_workspace(8192, 8192, 16384) == 2 * 8192 * 16384
    assert q8.q8_gemm_workspace(2048, 4096, 4096) == 2 * 2048 * 4096
    assert q8.q8_gemm_workspace(16, 28672, 8192) == 0          # decode kernel
    assert q8.q8_gemm_workspace(100, 2048, 2048) == 0          # small layer: mma.sync kernel
    assert q8.q8_gemm_workspace(300, 1000, 1000) == 0          # K % 16
    assert q8.q8_gemm_workspace(0, 8, 64) == 0
    # a misaligned workspace is refused before anything is enqueued
    st = lib.q8_gemm_dequant_ws(FAKE, FAKE, None, 1, FAKE, FAKE, 1, None, 512, 512, 512, FAKE, MISALIGNED, 1 << 20,
                                None)
    assert st == q8.Q8_ERR_INVALID_ARG


def test_workspace_entries_reject_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    f32 = ctypes.c_float(0.0)
    big = 1 << 30
    # int4 and block-scaled GEMMs with a misaligned workspace; a group size the format does not have
    assert lib.q8_gemm_w4a8_ws(FAKE, FAKE, None, 1, FAKE, FAKE, None, None, 512, 512, 512, 0, FAKE, f32,
                               MISALIGNED, big, None) == q8.Q8_ERR_INVALID_ARG
    assert lib.q8_gemm_mx_ws(FAKE, FAKE, 1, FAKE, FAKE, 32, None, 512, 512, 512, 0, FAKE, f32,
                             MISALIGNED, big, None) == q8.Q8_ERR_INVALID_ARG
    assert lib.q8_gemm_mx_ws(FAKE, FAKE, 1, FAKE, FAKE, 64, None, 512, 512, 512, 0, FAKE, f32,
                             FAKE, big, None) == q8.Q8_ERR_INVALID_ARG
    # the layer with a workspace: a misaligned workspace, a symmetry that is not an enum value
    assert lib.q8_linear_ws(FAKE, 512, 512, 1, 0, FAKE, FAKE, None, FAKE, FAKE, 1, None, 512, FAKE,
                            MISALIGNED, big, None) == q8.Q8_ERR_INVALID_ARG
    assert q8.q8_gemm_workspace(512, 512, 512) > 0
    assert lib.q8_linear_ws(FAKE, 512, 512, 1, 7, FAKE, FAKE, None, FAKE, FAKE, 1, None, 512, FAKE,
                            FAKE, big, None) == q8.Q8_ERR_INVALID_ARG
    # the dual quantizer: no fp16 output, a misaligned one, a zero point without asymmetry
    assert lib.q8_quantize_act_dual(FAKE, 8, 64, 1, 0, FAKE, None, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG
    assert lib.q8_quantize_act_dual(FAKE, 8, 64, 1, 0, FAKE, MISALIGNED, FAKE, None, None) == q8.Q8_ERR_INVALID_ARG
    assert lib.q8_quantize_act_dual(FAKE, 8, 64, 1, 0, FAKE, FAKE, FAKE, FAKE, None) == q8.Q8_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    import int8_quantized_gemm_gb300 as q8
    with pytest.raises(ValueError):
        q8.q8_quantize_act(torch.zeros(4, 32))


def test_host_layer_rejects_bad_arguments(lib):
    import int8_quantized_gemm_gb300 as q8
    ws_need = lib.q8_linear_host_workspace(64, 32, 64, 0)
    assert ws_need > 0 and lib.q8_linear_host_workspace(0, 32, 64, 0) == 0
    assert lib.q8_linear_host_workspace(1000, 32, 64, 1) < lib.q8_linear_host_workspace(1000, 32, 64, 0)

    def h(M=64, K=64, N=32, sym=0, a=FAKE, qw=FAKE, sw=FAKE, cs=None, y=FAKE, chunk=0, ws=P(0x100000), wsb=None):
        return lib.q8_linear_host(a, M, K, sym, qw, sw, 1, cs, N, y, chunk, ws, ws_need if wsb is None else wsb,
                                  None)
    assert h(wsb=ws_need - 1) == q8.Q8_ERR_INVALID_ARG            # workspace too small
    assert h(ws=P(0x100010)) == q8.Q8_ERR_INVALID_ARG             # not 256-byte aligned
    assert h(ws=None) == q8.Q8_ERR_INVALID_ARG
    assert h(K=24) == q8.Q8_ERR_UNSUPPORTED                        # K % 16
    assert h(sym=1) == q8.Q8_ERR_INVALID_ARG                       # asymmetric needs column sums
    assert h(sym=7) == q8.Q8_ERR_INVALID_ARG
    assert h(y=None) == q8.Q8_ERR_INVALID_ARG
    assert h(a=None) == q8.Q8_ERR_INVALID_ARG
    assert h(qw=MISALIGNED) == q8.Q8_ERR_INVALID_ARG
    assert h(M=-1) == q8.Q8_ERR_INVALID_ARG and h(chunk=-2) == q8.Q8_ERR_INVALID_ARG
    before = lib.q8_launch_count()
    assert h(M=0) == q8.Q8_OK and h(N=0) == q8.Q8_OK               # nothing to do
    assert lib.q8_launch_count() == before
