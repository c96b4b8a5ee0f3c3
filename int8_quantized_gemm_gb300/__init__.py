"""GB300 W8A8 quantized linear layer: Python binding of the C ABI in include/q8.h.

Argument marshalling only: every step of the path runs in the CUDA kernels of
libq8.so. PyTorch supplies device memory and the current stream. There is no
CPU fallback; if the library is missing or a call fails, an exception says so.

  q8_quantize_act(a, per_row=True, symmetric=True)   -> qa, s_a, z_a
  q8_rmsnorm_quantize_act(a, gamma, eps)             -> qa, s_a   (fused RMSNorm + per-token quantize)
  q8_quantize_weight(w, per_row=True)                 -> qw, s_w
  q8_colsum(qw)                                       -> colsum
  q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum)      -> y
  q8_gemm_epilogue(qa, s_a, z_a, qw, s_w, colsum, bias, out_dtype, out_scale) -> y (+bias; fp32/bf16/int8)
  q8_gemm_s32(qa, qw)                                 -> acc (raw INT32 accumulators)
  q8_quantize_weight_int4(w) -> qw4, s_w;  q8_colsum_int4(qw4, K);  q8_gemm_w4a8(qa, s_a, z_a, qw4, s_w, ...)
  q8_quantize_weight_mx(w, group) -> qw, sf;  q8_gemm_mx(qa, s_a, qw, sf, group, ...)   (block-scaled weights)
  q8_linear(a, qw, s_w, colsum)                       -> y   (quantize A, then GEMM)
  q8_linear_host(a_host, qw, s_w, colsum, y_host)      (host buffers; copies overlapped with the device work)
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "Q8Error", "load", "q8_quantize_act", "q8_rmsnorm_quantize_act", "q8_quantize_weight", "q8_colsum", "q8_gemm_dequant",
    "q8_gemm_epilogue", "q8_gemm_s32", "q8_linear", "q8_quantize_weight_int4", "q8_colsum_int4", "q8_gemm_w4a8",
    "q8_gemm_w4a8_s32", "q8_quantize_weight_mx", "q8_gemm_mx", "q8_quantize_act_f16", "q8_quantize_act_dual", "q8_gemm_f16a", "q8_gemm_f16a_s32", "q8_linear_host", "q8_linear_host_workspace", "q8_gemm_workspace", "q8_gemm_pick", "q8_launch_count", "q8_device_error",
    "q8_selftest_wait_timeout", "KERNELS",
]

LIB_PATH = _build.LIB
Q8_OK, Q8_ERR_INVALID_ARG, Q8_ERR_UNSUPPORTED, Q8_ERR_CUDA, Q8_ERR_TIMEOUT = range(5)
Q8_PER_TENSOR, Q8_PER_ROW = 0, 1
Q8_SYMMETRIC, Q8_ASYMMETRIC = 0, 1
KERNELS = {"auto": 0, "tcgen05": 1, "mma_s8": 2, "skinny": 3, "decode": 4, "decode_tc": 5, "tcgen05_pair": 6}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}

_lib = None


class Q8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libq8.so (built in-tree by build.py). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libq8.so is not built ({path}); run int8_quantized_gemm_gb300.build.build()")
    lib = ctypes.CDLL(path)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.q8_quantize_act.argtypes = [p, i64, i64, i32, i32, p, p, p, p]
    lib.q8_rmsnorm_quantize_act.argtypes = [p, p, i64, i64, ctypes.c_float, p, p, p]
    lib.q8_quantize_weight.argtypes = [p, i64, i64, i32, p, p, p]
    lib.q8_colsum.argtypes = [p, i64, i64, p, p]
    lib.q8_gemm_dequant.argtypes = [p, p, p, i32, p, p, i32, p, i64, i64, i64, p, p]
    lib.q8_gemm_dequant_ex.argtypes = [p, p, p, i32, p, p, i32, p, i64, i64, i64, p, i32, p]
    lib.q8_gemm_dequant_ws.argtypes = [p, p, p, i32, p, p, i32, p, i64, i64, i64, p, p, ctypes.c_size_t, p]
    lib.q8_gemm_workspace.argtypes = [i64, i64, i64]
    lib.q8_gemm_workspace.restype = ctypes.c_size_t
    lib.q8_gemm_epilogue_ex.argtypes = [p, p, p, i32, p, p, i32, p, p, i64, i64, i64, i32, p, ctypes.c_float, i32, p]
    lib.q8_gemm_s32_ex.argtypes = [p, p, i64, i64, i64, p, i32, p]
    lib.q8_quantize_act_f16.argtypes = [p, i64, i64, i32, i32, p, p, p, p]
    lib.q8_gemm_f16a_ex.argtypes = [p, p, p, i32, p, p, i32, p, p, i64, i64, i64, i32, p, ctypes.c_float, p]
    lib.q8_gemm_f16a_s32.argtypes = [p, p, i64, i64, i64, p, p]
    lib.q8_quantize_weight_int4.argtypes = [p, i64, i64, p, p, p]
    lib.q8_colsum_int4.argtypes = [p, i64, i64, p, p]
    lib.q8_gemm_w4a8_ex.argtypes = [p, p, p, i32, p, p, p, p, i64, i64, i64, i32, p, ctypes.c_float, i32, p]
    lib.q8_gemm_w4a8_s32_ex.argtypes = [p, p, i64, i64, i64, p, i32, p]
    lib.q8_quantize_weight_mx.argtypes = [p, i64, i64, i32, p, p, p]
    lib.q8_gemm_mx_ex.argtypes = [p, p, i32, p, p, i32, p, i64, i64, i64, i32, p, ctypes.c_float, i32, p]
    lib.q8_gemm_w4a8_ws.argtypes = [p, p, p, i32, p, p, p, p, i64, i64, i64, i32, p, ctypes.c_float, p,
                                    ctypes.c_size_t, p]
    lib.q8_gemm_mx_ws.argtypes = [p, p, i32, p, p, i32, p, i64, i64, i64, i32, p, ctypes.c_float, p,
                                  ctypes.c_size_t, p]
    lib.q8_linear.argtypes = [p, i64, i64, i32, i32, p, p, p, p, p, i32, p, i64, p, p]
    lib.q8_linear_ws.argtypes = [p, i64, i64, i32, i32, p, p, p, p, p, i32, p, i64, p, p, ctypes.c_size_t, p]
    lib.q8_quantize_act_dual.argtypes = [p, i64, i64, i32, i32, p, p, p, p, p]
    lib.q8_selftest_wait_timeout.argtypes = [i32, p, p, i64, i64, i64, p, i64, p]
    lib.q8_linear_host_workspace.argtypes = [i64, i64, i64, i64]
    lib.q8_linear_host_workspace.restype = ctypes.c_size_t
    lib.q8_linear_host.argtypes = [p, i64, i64, i32, p, p, i32, p, i64, p, i64, p, ctypes.c_size_t, p]
    lib.q8_gemm_pick.argtypes = [i64, i64, i64]
    lib.q8_status_string.argtypes = [i32]
    lib.q8_status_string.restype = ctypes.c_char_p
    lib.q8_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.q8_launch_count.argtypes = []
    lib.q8_launch_count.restype = ctypes.c_uint64
    for name in ("q8_quantize_act", "q8_rmsnorm_quantize_act", "q8_quantize_weight", "q8_colsum", "q8_gemm_dequant",
                 "q8_gemm_dequant_ex", "q8_gemm_dequant_ws", "q8_gemm_epilogue_ex", "q8_gemm_s32_ex", "q8_quantize_weight_int4",
                 "q8_colsum_int4", "q8_gemm_w4a8_ex", "q8_gemm_w4a8_s32_ex", "q8_quantize_weight_mx", "q8_gemm_mx_ex",
                 "q8_gemm_w4a8_ws", "q8_gemm_mx_ws", "q8_linear_ws", "q8_quantize_act_dual",
                 "q8_linear", "q8_linear_host", "q8_gemm_pick", "q8_device_error", "q8_selftest_wait_timeout"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().q8_status_string(status).decode()


def _check(status: int, what: str):
    if status != Q8_OK:
        raise Q8Error(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, ndim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def q8_quantize_act(a: torch.Tensor, per_row: bool = True, symmetric: bool = True, qa=None, s_a=None,
                    z_a=None, stream=None):
    """Dynamic activation quantization of fp32 a[M, K]; returns (qa int8, s_a fp32, z_a int32 or None)."""
    _need(a, torch.float32, "a", 2)
    M, K = a.shape
    n = M if per_row else 1
    qa = torch.empty((M, K), dtype=torch.int8, device=a.device) if qa is None else qa
    s_a = torch.empty(n, dtype=torch.float32, device=a.device) if s_a is None else s_a
    if not symmetric and z_a is None:
        z_a = torch.empty(n, dtype=torch.int32, device=a.device)
    if symmetric:
        z_a = None
    _check(load().q8_quantize_act(_ptr(a), M, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR,
                                  Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qa), _ptr(s_a),
                                  _ptr(z_a), _stream(stream)), "q8_quantize_act")
    return qa, s_a, z_a


def q8_rmsnorm_quantize_act(a: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, qa=None, s_a=None,
                            stream=None):
    """Fused RMSNorm (weights gamma[K], eps under the root) + per-token symmetric quantization
    of fp32 a[M, K]; returns (qa int8 [M, K], s_a fp32 [M])."""
    _need(a, torch.float32, "a", 2)
    _need(gamma, torch.float32, "gamma", 1)
    M, K = a.shape
    if gamma.numel() != K:
        raise ValueError("gamma must have K entries")
    qa = torch.empty((M, K), dtype=torch.int8, device=a.device) if qa is None else qa
    s_a = torch.empty(M, dtype=torch.float32, device=a.device) if s_a is None else s_a
    _check(load().q8_rmsnorm_quantize_act(_ptr(a), _ptr(gamma), M, K, ctypes.c_float(eps), _ptr(qa), _ptr(s_a),
                                          _stream(stream)), "q8_rmsnorm_quantize_act")
    return qa, s_a


def q8_quantize_weight(w: torch.Tensor, per_row: bool = True, qw=None, s_w=None, stream=None):
    """Symmetric quantization of fp32 W[N, K] (K-major); returns (qw int8, s_w fp32)."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device) if qw is None else qw
    s_w = torch.empty(N if per_row else 1, dtype=torch.float32, device=w.device) if s_w is None else s_w
    _check(load().q8_quantize_weight(_ptr(w), N, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR, _ptr(qw),
                                     _ptr(s_w), _stream(stream)), "q8_quantize_weight")
    return qw, s_w


def q8_colsum(qw: torch.Tensor, out=None, stream=None):
    _need(qw, torch.int8, "qw", 2)
    N, K = qw.shape
    out = torch.empty(N, dtype=torch.int32, device=qw.device) if out is None else out
    _check(load().q8_colsum(_ptr(qw), N, K, _ptr(out), _stream(stream)), "q8_colsum")
    return out


def q8_gemm_workspace(M: int, N: int, K: int) -> int:
    """Device workspace bytes q8_gemm_dequant(..., workspace=) can use for this shape (0: none)."""
    return int(load().q8_gemm_workspace(M, N, K))


def q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum=None, y=None, kernel: str = "auto", workspace=None,
                    stream=None):
    """y[M, N] = (acc - z_a*colsum) * (s_a * s_w) from int8 codes; per-row scales are inferred
    from the lengths of s_a (M entries) and s_w (N entries). workspace: an optional device tensor of
    at least q8_gemm_workspace(M, N, K) bytes (kernel "auto" only; q8_gemm_dequant_ws)."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw, torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qa and qw disagree on K")
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    ga = Q8_PER_ROW if (s_a.numel() == M and M != 1) else Q8_PER_TENSOR
    gw = Q8_PER_ROW if (s_w.numel() == N and N != 1) else Q8_PER_TENSOR
    if s_a.numel() not in (1, M) or s_w.numel() not in (1, N):
        raise ValueError("s_a must have 1 or M entries and s_w 1 or N entries")
    if z_a is not None:
        _need(z_a, torch.int32, "z_a", 1)
        if z_a.numel() != s_a.numel():
            raise ValueError("z_a must have as many entries as s_a")
        if colsum is None:
            raise ValueError("an asymmetric A needs the weight column sums")
        _need(colsum, torch.int32, "colsum", 1)
    y = torch.empty((M, N), dtype=torch.float32, device=qa.device) if y is None else y
    _need(y, torch.float32, "y", 2)
    if workspace is not None:
        if kernel != "auto":
            raise ValueError("a workspace goes with the automatic kernel choice")
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        _check(load().q8_gemm_dequant_ws(_ptr(qa), _ptr(s_a), _ptr(z_a), ga, _ptr(qw), _ptr(s_w), gw,
                                         _ptr(colsum if z_a is not None else None), M, N, K, _ptr(y),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)), "q8_gemm_dequant_ws")
        return y
    _check(load().q8_gemm_dequant_ex(_ptr(qa), _ptr(s_a), _ptr(z_a), ga, _ptr(qw), _ptr(s_w), gw,
                                     _ptr(colsum if z_a is not None else None), M, N, K, _ptr(y),
                                     KERNELS[kernel], _stream(stream)), "q8_gemm_dequant")
    return y


OUT_TYPES = {torch.float32: 0, torch.bfloat16: 1, torch.int8: 2}


def _epilogue_args(qa, qa_dtype, s_a, z_a, qw, s_w, colsum, bias, out_dtype, out_scale, out):
    """Checks of the epilogue entries; returns (M, N, K, ga, gw, out)."""
    _need(qa, qa_dtype, "qa", 2)
    _need(qw, torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qa and qw disagree on K")
    if out_dtype not in OUT_TYPES:
        raise TypeError("out_dtype must be torch.float32, torch.bfloat16 or torch.int8")
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    if s_a.numel() not in (1, M) or s_w.numel() not in (1, N):
        raise ValueError("s_a must have 1 or M entries and s_w 1 or N entries")
    ga = Q8_PER_ROW if (s_a.numel() == M and M != 1) else Q8_PER_TENSOR
    gw = Q8_PER_ROW if (s_w.numel() == N and N != 1) else Q8_PER_TENSOR
    if z_a is not None:
        _need(z_a, torch.int32, "z_a", 1)
        if colsum is None:
            raise ValueError("an asymmetric A needs the weight column sums")
        _need(colsum, torch.int32, "colsum", 1)
    if bias is not None:
        _need(bias, torch.float32, "bias", 1)
        if bias.numel() != N:
            raise ValueError("bias must have N entries")
    if out_dtype == torch.int8 and out_scale is None:
        raise ValueError("int8 output needs out_scale")
    out = torch.empty((M, N), dtype=out_dtype, device=qa.device) if out is None else out
    _need(out, out_dtype, "out", 2)
    return M, N, K, ga, gw, out


def q8_quantize_act_f16(a: torch.Tensor, per_row: bool = True, symmetric: bool = True, qa16=None, s_a=None,
                        z_a=None, stream=None):
    """q8_quantize_act with the codes written as fp16 values; returns (qa16 float16, s_a, z_a or None)."""
    _need(a, torch.float32, "a", 2)
    M, K = a.shape
    n = M if per_row else 1
    qa16 = torch.empty((M, K), dtype=torch.float16, device=a.device) if qa16 is None else qa16
    _need(qa16, torch.float16, "qa16", 2)
    s_a = torch.empty(n, dtype=torch.float32, device=a.device) if s_a is None else s_a
    if not symmetric and z_a is None:
        z_a = torch.empty(n, dtype=torch.int32, device=a.device)
    if symmetric:
        z_a = None
    _check(load().q8_quantize_act_f16(_ptr(a), M, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR,
                                      Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qa16), _ptr(s_a),
                                      _ptr(z_a), _stream(stream)), "q8_quantize_act_f16")
    return qa16, s_a, z_a


def q8_quantize_act_dual(a: torch.Tensor, per_row: bool = True, symmetric: bool = True, qa=None, qa16=None,
                         s_a=None, z_a=None, stream=None):
    """q8_quantize_act that also writes the codes as fp16 values (for q8_gemm_f16a); returns
    (qa int8, qa16 float16, s_a, z_a or None)."""
    _need(a, torch.float32, "a", 2)
    M, K = a.shape
    n = M if per_row else 1
    qa = torch.empty((M, K), dtype=torch.int8, device=a.device) if qa is None else qa
    qa16 = torch.empty((M, K), dtype=torch.float16, device=a.device) if qa16 is None else qa16
    _need(qa16, torch.float16, "qa16", 2)
    s_a = torch.empty(n, dtype=torch.float32, device=a.device) if s_a is None else s_a
    if not symmetric and z_a is None:
        z_a = torch.empty(n, dtype=torch.int32, device=a.device)
    if symmetric:
        z_a = None
    _check(load().q8_quantize_act_dual(_ptr(a), M, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR,
                                       Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qa), _ptr(qa16), _ptr(s_a),
                                       _ptr(z_a), _stream(stream)), "q8_quantize_act_dual")
    return qa, qa16, s_a, z_a


def q8_gemm_f16a(qa16, s_a, z_a, qw, s_w, colsum=None, bias=None, out_dtype=torch.float32, out_scale=None,
                 out=None, stream=None):
    """q8_gemm_epilogue on fp16-valued activation codes (from q8_quantize_act_f16)."""
    M, N, K, ga, gw, out = _epilogue_args(qa16, torch.float16, s_a, z_a, qw, s_w, colsum, bias, out_dtype,
                                          out_scale, out)
    _check(load().q8_gemm_f16a_ex(_ptr(qa16), _ptr(s_a), _ptr(z_a), ga, _ptr(qw), _ptr(s_w), gw,
                                  _ptr(colsum if z_a is not None else None), _ptr(bias), M, N, K,
                                  OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0),
                                  _stream(stream)), "q8_gemm_f16a")
    return out


def q8_gemm_f16a_s32(qa16, qw, out=None, stream=None):
    """Raw INT32 accumulators of q8_gemm_f16a."""
    _need(qa16, torch.float16, "qa16", 2)
    _need(qw, torch.int8, "qw", 2)
    M, K = qa16.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qa16 and qw disagree on K")
    out = torch.empty((M, N), dtype=torch.int32, device=qa16.device) if out is None else out
    _need(out, torch.int32, "out", 2)
    _check(load().q8_gemm_f16a_s32(_ptr(qa16), _ptr(qw), M, N, K, _ptr(out), _stream(stream)), "q8_gemm_f16a_s32")
    return out


def q8_gemm_epilogue(qa, s_a, z_a, qw, s_w, colsum=None, bias=None, out_dtype=torch.float32, out_scale=None,
                     out=None, kernel: str = "auto", stream=None):
    """Quantized linear layer with the epilogue variants: y = (acc - z_a*colsum) * (s_a*s_w) + bias,
    written as fp32, bf16, or int8 codes with the static output scale out_scale."""
    M, N, K, ga, gw, out = _epilogue_args(qa, torch.int8, s_a, z_a, qw, s_w, colsum, bias, out_dtype, out_scale,
                                          out)
    _check(load().q8_gemm_epilogue_ex(_ptr(qa), _ptr(s_a), _ptr(z_a), ga, _ptr(qw), _ptr(s_w), gw,
                                      _ptr(colsum if z_a is not None else None), _ptr(bias), M, N, K,
                                      OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0),
                                      KERNELS[kernel], _stream(stream)), "q8_gemm_epilogue")
    return out


def q8_quantize_weight_int4(w: torch.Tensor, qw4=None, s_w=None, stream=None):
    """Per-channel symmetric int4 codes of fp32 W[N, K], packed two per byte: (qw4 uint8 [N, K/2], s_w [N])."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    qw4 = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device) if qw4 is None else qw4
    s_w = torch.empty(N, dtype=torch.float32, device=w.device) if s_w is None else s_w
    _check(load().q8_quantize_weight_int4(_ptr(w), N, K, _ptr(qw4), _ptr(s_w), _stream(stream)),
           "q8_quantize_weight_int4")
    return qw4, s_w


def q8_colsum_int4(qw4: torch.Tensor, K: int, out=None, stream=None):
    _need(qw4, torch.uint8, "qw4", 2)
    N = qw4.shape[0]
    if qw4.shape[1] * 2 != K:
        raise ValueError("qw4 must be [N, K / 2]")
    out = torch.empty(N, dtype=torch.int32, device=qw4.device) if out is None else out
    _check(load().q8_colsum_int4(_ptr(qw4), N, K, _ptr(out), _stream(stream)), "q8_colsum_int4")
    return out


def _ws_args(workspace, kernel):
    if kernel != "auto":
        raise ValueError("a workspace goes with the automatic kernel choice")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def q8_gemm_w4a8(qa, s_a, z_a, qw4, s_w, colsum=None, bias=None, out_dtype=torch.float32, out_scale=None,
                 out=None, kernel: str = "auto", workspace=None, stream=None):
    """W4A8 linear layer: int8 activations x packed int4 weights, epilogue as q8_gemm_epilogue.
    workspace: an optional device tensor of at least 2 M K bytes for the fp16 copy of the codes
    (kernel "auto" only; q8_gemm_w4a8_ws)."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw4, torch.uint8, "qw4", 2)
    M, K = qa.shape
    N = qw4.shape[0]
    if qw4.shape[1] * 2 != K:
        raise ValueError("qw4 must be [N, K / 2]")
    if out_dtype not in OUT_TYPES:
        raise TypeError("out_dtype must be torch.float32, torch.bfloat16 or torch.int8")
    _need(s_a, torch.float32, "s_a", 1)
    _need(s_w, torch.float32, "s_w", 1)
    if s_a.numel() not in (1, M) or s_w.numel() != N:
        raise ValueError("s_a must have 1 or M entries and s_w N entries")
    ga = Q8_PER_ROW if (s_a.numel() == M and M != 1) else Q8_PER_TENSOR
    if z_a is not None:
        _need(z_a, torch.int32, "z_a", 1)
        if colsum is None:
            raise ValueError("an asymmetric A needs the weight column sums")
        _need(colsum, torch.int32, "colsum", 1)
    if bias is not None:
        _need(bias, torch.float32, "bias", 1)
    if out_dtype == torch.int8 and out_scale is None:
        raise ValueError("int8 output needs out_scale")
    out = torch.empty((M, N), dtype=out_dtype, device=qa.device) if out is None else out
    _need(out, out_dtype, "out", 2)
    if workspace is not None:
        wp, wb = _ws_args(workspace, kernel)
        _check(load().q8_gemm_w4a8_ws(_ptr(qa), _ptr(s_a), _ptr(z_a), ga, _ptr(qw4), _ptr(s_w),
                                      _ptr(colsum if z_a is not None else None), _ptr(bias), M, N, K,
                                      OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0), wp, wb,
                                      _stream(stream)), "q8_gemm_w4a8_ws")
        return out
    _check(load().q8_gemm_w4a8_ex(_ptr(qa), _ptr(s_a), _ptr(z_a), ga, _ptr(qw4), _ptr(s_w),
                                  _ptr(colsum if z_a is not None else None), _ptr(bias), M, N, K,
                                  OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0),
                                  KERNELS[kernel], _stream(stream)), "q8_gemm_w4a8")
    return out


def q8_gemm_w4a8_s32(qa, qw4, out=None, kernel: str = "auto", stream=None):
    """Raw INT32 accumulators of int8 qa x packed int4 qw4 (diagnostic export)."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw4, torch.uint8, "qw4", 2)
    M, K = qa.shape
    N = qw4.shape[0]
    out = torch.empty((M, N), dtype=torch.int32, device=qa.device) if out is None else out
    _need(out, torch.int32, "out", 2)
    _check(load().q8_gemm_w4a8_s32_ex(_ptr(qa), _ptr(qw4), M, N, K, _ptr(out), KERNELS[kernel], _stream(stream)),
           "q8_gemm_w4a8_s32")
    return out


def q8_gemm_s32(qa, qw, out=None, kernel: str = "auto", stream=None):
    """Raw INT32 accumulators acc[M, N] = qa . qw^T (diagnostic export of the integer GEMM)."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw, torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    out = torch.empty((M, N), dtype=torch.int32, device=qa.device) if out is None else out
    _need(out, torch.int32, "out", 2)
    _check(load().q8_gemm_s32_ex(_ptr(qa), _ptr(qw), M, N, K, _ptr(out), KERNELS[kernel], _stream(stream)),
           "q8_gemm_s32")
    return out


def q8_linear(a, qw, s_w, colsum=None, per_row: bool = True, symmetric: bool = True, kernel: str = "auto",
              qa=None, s_a=None, z_a=None, y=None, workspace=None, stream=None):
    """Whole W8A8 layer on fp32 activations: dynamic quantization of a, then the GEMM + epilogue
    (one C call, q8_linear, for kernel="auto"; an explicit kernel runs the two calls). workspace:
    an optional device tensor of at least q8_gemm_workspace(M, N, K) bytes (q8_linear_ws: the
    quantizer also writes the codes as fp16 values there for the CTA-pair kernel). Returns y."""
    if kernel != "auto":
        qa, s_a, z_a = q8_quantize_act(a, per_row=per_row, symmetric=symmetric, qa=qa, s_a=s_a, z_a=z_a,
                                       stream=stream)
        return q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum, kernel=kernel, y=y, stream=stream)
    _need(a, torch.float32, "a", 2)
    _need(qw, torch.int8, "qw", 2)
    _need(s_w, torch.float32, "s_w", 1)
    M, K = a.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qw must be [N, K] with the K of a")
    n = M if per_row else 1
    qa = torch.empty((M, K), dtype=torch.int8, device=a.device) if qa is None else qa
    s_a = torch.empty(n, dtype=torch.float32, device=a.device) if s_a is None else s_a
    if symmetric:
        z_a = None
    elif z_a is None:
        z_a = torch.empty(n, dtype=torch.int32, device=a.device)
    if not symmetric and colsum is None:
        raise ValueError("asymmetric activations need colsum")
    y = torch.empty((M, N), dtype=torch.float32, device=a.device) if y is None else y
    _need(y, torch.float32, "y", 2)
    gw = Q8_PER_ROW if (s_w.numel() == N and N != 1) else Q8_PER_TENSOR
    if workspace is not None:
        wp, wb = _ws_args(workspace, kernel)
        _check(load().q8_linear_ws(_ptr(a), M, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR,
                                   Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qa), _ptr(s_a), _ptr(z_a),
                                   _ptr(qw), _ptr(s_w), gw, _ptr(colsum if not symmetric else None), N, _ptr(y), wp,
                                   wb, _stream(stream)), "q8_linear_ws")
        return y
    _check(load().q8_linear(_ptr(a), M, K, Q8_PER_ROW if per_row else Q8_PER_TENSOR,
                            Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qa), _ptr(s_a), _ptr(z_a), _ptr(qw),
                            _ptr(s_w), gw, _ptr(colsum if not symmetric else None), N, _ptr(y), _stream(stream)),
           "q8_linear")
    return y


def q8_linear_host_workspace(M: int, N: int, K: int, chunk_rows: int = 0) -> int:
    """Device workspace bytes that q8_linear_host needs."""
    return int(load().q8_linear_host_workspace(M, N, K, chunk_rows))


def q8_linear_host(a_host, qw, s_w, colsum=None, y_host=None, symmetric: bool = True, chunk_rows: int = 0,
                   workspace=None, stream=None):
    """Whole layer on host buffers: a_host fp32 [M, K] (CPU, pinned for overlap) -> y_host fp32 [M, N] (CPU),
    per-token quantization on the device. The result is in y_host once `stream` (default: the current
    stream) has completed."""
    if a_host.device.type != "cpu" or a_host.dtype != torch.float32 or a_host.dim() != 2 or not a_host.is_contiguous():
        raise ValueError("a_host must be a contiguous fp32 [M, K] CPU tensor")
    _need(qw, torch.int8, "qw", 2)
    M, K = a_host.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qw must be [N, K]")
    _need(s_w, torch.float32, "s_w", 1)
    gw = Q8_PER_ROW if (s_w.numel() == N and N != 1) else Q8_PER_TENSOR
    if y_host is None:
        y_host = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    if y_host.device.type != "cpu" or y_host.dtype != torch.float32 or tuple(y_host.shape) != (M, N) \
            or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous fp32 [M, N] CPU tensor")
    need = q8_linear_host_workspace(M, N, K, chunk_rows)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=qw.device)
    _check(load().q8_linear_host(_ptr(a_host), M, K, Q8_SYMMETRIC if symmetric else Q8_ASYMMETRIC, _ptr(qw),
                                 _ptr(s_w), gw, _ptr(colsum), N, _ptr(y_host), chunk_rows, _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "q8_linear_host")
    return y_host


def q8_gemm_pick(M: int, N: int, K: int) -> str:
    return KERNEL_NAMES[load().q8_gemm_pick(M, N, K)]


def q8_launch_count() -> int:
    return int(load().q8_launch_count())


def q8_selftest_wait_timeout(qa, qw, kernel: str = "decode", wait_cycles: int = 1 << 24, stream=None):
    """Self-test of the bounded device waits: runs `kernel` ("decode" or "tcgen05") with its loads
    withheld so that its first wait runs out after wait_cycles; read the result with q8_device_error()."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw, torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    acc = torch.zeros((M, N), dtype=torch.int32, device=qa.device)
    _check(load().q8_selftest_wait_timeout(KERNELS[kernel], _ptr(qa), _ptr(qw), M, N, K, _ptr(acc), wait_cycles,
                                           _stream(stream)), "q8_selftest_wait_timeout")
    return acc


def q8_device_error() -> int:
    """Device error word of the tensor-core kernel (0 = every bounded wait completed); resets it."""
    code = ctypes.c_uint32(0)
    st = load().q8_device_error(ctypes.byref(code))
    if st not in (Q8_OK, Q8_ERR_TIMEOUT):
        _check(st, "q8_device_error")
    return int(code.value)


def q8_quantize_weight_mx(w: torch.Tensor, group: int = 32, qw=None, sf=None, stream=None):
    """Block-scaled int8 codes of fp32 W[N, K]: (qw int8 [N, K], sf [ceil(K / group / 4), N] E8M0 scale
    words, held as int32 bit patterns: byte b of word w is group 4w + b)."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    words = (K // group + 3) // 4
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device) if qw is None else qw
    sf = torch.empty((words, N), dtype=torch.int32, device=w.device) if sf is None else sf
    _check(load().q8_quantize_weight_mx(_ptr(w), N, K, group, _ptr(qw), _ptr(sf), _stream(stream)),
           "q8_quantize_weight_mx")
    return qw, sf


def q8_gemm_mx(qa, s_a, qw, sf, group: int = 32, bias=None, out_dtype=torch.float32, out_scale=None, out=None,
               kernel: str = "auto", workspace=None, stream=None):
    """Linear layer with block-scaled int8 weights: y = fl(T * s_a) (+ bias), T = sum_k qa * q * s.
    workspace: as q8_gemm_w4a8 (q8_gemm_mx_ws)."""
    _need(qa, torch.int8, "qa", 2)
    _need(qw, torch.int8, "qw", 2)
    _need(sf, torch.int32, "sf", 2)
    M, K = qa.shape
    N = qw.shape[0]
    if qw.shape[1] != K or sf.shape[1] != N:
        raise ValueError("qw must be [N, K] and sf [words, N]")
    if out_dtype not in OUT_TYPES:
        raise TypeError("out_dtype must be torch.float32, torch.bfloat16 or torch.int8")
    _need(s_a, torch.float32, "s_a", 1)
    if s_a.numel() not in (1, M):
        raise ValueError("s_a must have 1 or M entries")
    ga = Q8_PER_ROW if (s_a.numel() == M and M != 1) else Q8_PER_TENSOR
    if bias is not None:
        _need(bias, torch.float32, "bias", 1)
    if out_dtype == torch.int8 and out_scale is None:
        raise ValueError("int8 output needs out_scale")
    out = torch.empty((M, N), dtype=out_dtype, device=qa.device) if out is None else out
    _need(out, out_dtype, "out", 2)
    if workspace is not None:
        wp, wb = _ws_args(workspace, kernel)
        _check(load().q8_gemm_mx_ws(_ptr(qa), _ptr(s_a), ga, _ptr(qw), _ptr(sf), group, _ptr(bias), M, N, K,
                                    OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0), wp, wb,
                                    _stream(stream)), "q8_gemm_mx_ws")
        return out
    _check(load().q8_gemm_mx_ex(_ptr(qa), _ptr(s_a), ga, _ptr(qw), _ptr(sf), group, _ptr(bias), M, N, K,
                                OUT_TYPES[out_dtype], _ptr(out), ctypes.c_float(out_scale or 0.0), KERNELS[kernel],
                                _stream(stream)), "q8_gemm_mx")
    return out
