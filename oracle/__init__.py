"""CPU oracle for the W8A8 quantized linear layer -- TEST INFRASTRUCTURE.

Plain, slow, obviously correct: a C file (q8_oracle.c, built with gcc
-O2 -ffp-contract=off) wrapped with ctypes over numpy arrays. It shares no
code with the CUDA library and never imports it. Only tests/, the smoke check
and bench.py's CPU-baseline leg may call it; the product path never does.

Every function follows a passage of the pages (cited in q8_oracle.c):
  quantize_sym / quantize_asym   "100 Days of GPU, Day 98" (What a scale
                                 actually promises); "Write Int8 Quantized
                                 Kernel" step 1; "Activation Quantization
                                 Architecture" (The quantizer itself; numpy
                                 reference; Fusion pseudocode for the guard)
  colsum                         Day 98 (zero-point paragraph after the kernel)
  gemm_acc                       Day 98 (accumulate loop); "Activation
                                 Quantization Architecture" (The integer GEMM)
  linear_codes / linear_codes_at Day 98 (epilogue listing)
  rmsnorm / rmsnorm_quantize     "Activation Quantization Architecture" (Fusion:
                                 the fused norm-and-quantize pseudocode)
  quantize_int4, pack_int4,      TileLang tutorial ch. 27 (2.4 int8 / int4; the int4
  unpack_int4                    GEMM example's packing and sign extension)
  linear_codes_bias, to_bf16,    "Activation Quantization Architecture" (Fusion:
  quantize_static                the epilogue adds the bias, writes bf16, or
                                 quantizes the output for the next GEMM)
  quantize_weight_mx, gemm_mx,   TileLang tutorial ch. 27 (2.3 MX / block-scaled:
  linear_mx, e8m0_ceil           block granularity + E8M0, the scale-word packing)
All of them are pinned by tests/test_oracle_pins.py and tests/test_oracle_rmsnorm.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libq8oracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_ARG, INT32_OVERFLOW = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile q8_oracle.c with gcc (OpenMP if available). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
            "-shared", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.q8o_quantize_sym.argtypes = [p, i64, i64, i32, p, p]
        lib.q8o_quantize_sym.restype = i32
        lib.q8o_quantize_asym.argtypes = [p, i64, i64, i32, p, p, p]
        lib.q8o_quantize_asym.restype = i32
        lib.q8o_colsum.argtypes = [p, i64, i64, p]
        lib.q8o_colsum.restype = None
        lib.q8o_dot.argtypes = [p, p, i64]
        lib.q8o_dot.restype = i64
        lib.q8o_gemm_acc.argtypes = [p, p, i64, i64, i64, p, i32]
        lib.q8o_gemm_acc.restype = None
        lib.q8o_linear_codes.argtypes = [p, p, p, i32, p, p, i32, i64, i64, i64, p, i32]
        lib.q8o_linear_codes.restype = i32
        lib.q8o_linear_codes_at.argtypes = [p, p, p, i32, p, p, i32, i64, p, p, i64, p, p]
        lib.q8o_linear_codes_at.restype = i32
        lib.q8o_sym_scale.argtypes = [ctypes.c_float]
        lib.q8o_sym_scale.restype = ctypes.c_float
        lib.q8o_rmsnorm.argtypes = [p, p, i64, i64, ctypes.c_float, p, p]
        lib.q8o_quantize_int4.argtypes = [p, i64, i64, p, p]
        lib.q8o_quantize_int4.restype = i32
        lib.q8o_pack_int4.argtypes = [p, i64, i64, p]
        lib.q8o_pack_int4.restype = i32
        lib.q8o_unpack_int4.argtypes = [p, i64, i64, p]
        lib.q8o_unpack_int4.restype = i32
        lib.q8o_linear_codes_bias.argtypes = [p, p, p, i32, p, p, i32, p, i64, i64, i64, p, i32]
        lib.q8o_linear_codes_bias.restype = i32
        lib.q8o_to_bf16.argtypes = [p, i64, p]
        lib.q8o_to_bf16.restype = None
        lib.q8o_quantize_static.argtypes = [p, i64, ctypes.c_float, p]
        lib.q8o_quantize_static.restype = None
        lib.q8o_rmsnorm.restype = i32
        lib.q8o_e8m0_ceil.argtypes = [ctypes.c_float]
        lib.q8o_e8m0_ceil.restype = i32
        lib.q8o_quantize_weight_mx.argtypes = [p, i64, i64, i32, p, p]
        lib.q8o_quantize_weight_mx.restype = i32
        lib.q8o_gemm_mx.argtypes = [p, p, p, i64, i64, i64, i32, p, p, i32]
        lib.q8o_gemm_mx.restype = i32
        lib.q8o_linear_mx.argtypes = [p, p, i32, p, p, p, i64, i64, i64, i32, p, i32]
        lib.q8o_linear_mx.restype = i32
        lib.q8o_openmp_max_threads.argtypes = []
        lib.q8o_openmp_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().q8o_openmp_max_threads())


def quantize_sym(x: np.ndarray, per_row: bool):
    """Symmetric int8 codes of a 2-D fp32 array; returns (q int8, s fp32[rows or 1])."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.int8)
    s = np.empty(rows if per_row else 1, np.float32)
    st = _load().q8o_quantize_sym(_ptr(x), rows, cols, int(per_row), _ptr(q), _ptr(s))
    assert st == OK
    return q, s


def quantize_asym(x: np.ndarray, per_row: bool):
    """Asymmetric int8 codes; returns (q int8, s fp32, z int32) with s, z [rows or 1]."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.int8)
    n = rows if per_row else 1
    s = np.empty(n, np.float32)
    z = np.empty(n, np.int32)
    st = _load().q8o_quantize_asym(_ptr(x), rows, cols, int(per_row), _ptr(q), _ptr(s), _ptr(z))
    assert st == OK
    return q, s, z


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float):
    """RMSNorm rows of fp32 x with weights gamma; returns (y fp32, exact sum of squares per row
    as float64). The sum is exact and rounded once to fp32 (see q8o_rmsnorm)."""
    x = _c(x, np.float32)
    gamma = _c(gamma, np.float32)
    rows, cols = x.shape
    assert gamma.shape == (cols,)
    y = np.empty((rows, cols), np.float32)
    sumsq = np.empty(rows, np.float64)
    st = _load().q8o_rmsnorm(_ptr(x), _ptr(gamma), rows, cols, ctypes.c_float(eps), _ptr(y), _ptr(sumsq))
    assert st == OK
    return y, sumsq


def rmsnorm_quantize(x: np.ndarray, gamma: np.ndarray, eps: float) -> dict:
    """Fused RMSNorm + per-token symmetric quantization: qa int8, sa fp32 [rows], plus the
    normalised rows y and the per-row sums of squares."""
    y, sumsq = rmsnorm(x, gamma, eps)
    qa, sa = quantize_sym(y, per_row=True)
    return {"qa": qa, "sa": sa, "y": y, "sumsq": sumsq}


def sym_scale(amax: float) -> np.float32:
    return np.float32(_load().q8o_sym_scale(ctypes.c_float(amax)))


def colsum(qw: np.ndarray) -> np.ndarray:
    """int64 column sums of a K-major W[N, K] of codes."""
    qw = _c(qw, np.int8)
    N, K = qw.shape
    out = np.empty(N, np.int64)
    _load().q8o_colsum(_ptr(qw), N, K, _ptr(out))
    return out


def dot(a: np.ndarray, b: np.ndarray) -> int:
    a = _c(a, np.int8)
    b = _c(b, np.int8)
    assert a.shape == b.shape and a.ndim == 1
    return int(_load().q8o_dot(_ptr(a), _ptr(b), a.shape[0]))


def gemm_acc(qa: np.ndarray, qw: np.ndarray, threads: int = 1) -> np.ndarray:
    """int64 acc[M, N] = qa[M, K] . qw[N, K]^T."""
    qa = _c(qa, np.int8)
    qw = _c(qw, np.int8)
    M, K = qa.shape
    N, K2 = qw.shape
    assert K == K2
    acc = np.empty((M, N), np.int64)
    _load().q8o_gemm_acc(_ptr(qa), _ptr(qw), M, N, K, _ptr(acc), threads)
    return acc


def linear_codes(qa, sa, za, qw, sw, a_per_row: bool, w_per_row: bool, threads: int = 1):
    """fp32 y[M, N] from codes and scales; returns (y, status)."""
    qa = _c(qa, np.int8)
    qw = _c(qw, np.int8)
    sa = _c(sa, np.float32)
    sw = _c(sw, np.float32)
    za = None if za is None else _c(za, np.int32)
    M, K = qa.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.float32)
    st = _load().q8o_linear_codes(_ptr(qa), _ptr(sa), _ptr(za), int(a_per_row),
                                  _ptr(qw), _ptr(sw), int(w_per_row), M, N, K, _ptr(y), threads)
    return y, st


def linear_codes_bias(qa, sa, za, qw, sw, bias, a_per_row: bool, w_per_row: bool, threads: int = 1):
    """fp32 y[M, N] from codes and scales plus bias[N] (None: no bias); returns (y, status)."""
    qa = _c(qa, np.int8)
    qw = _c(qw, np.int8)
    sa = _c(sa, np.float32)
    sw = _c(sw, np.float32)
    za = None if za is None else _c(za, np.int32)
    bias = None if bias is None else _c(bias, np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.float32)
    st = _load().q8o_linear_codes_bias(_ptr(qa), _ptr(sa), _ptr(za), int(a_per_row), _ptr(qw), _ptr(sw),
                                       int(w_per_row), _ptr(bias), M, N, K, _ptr(y), threads)
    return y, st


def quantize_int4(w: np.ndarray):
    """Per-row symmetric int4 codes (one per int8 element, in [-8, 7]) and scales s = absmax / 7."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols), np.int8)
    s = np.empty(rows, np.float32)
    assert _load().q8o_quantize_int4(_ptr(w), rows, cols, _ptr(q), _ptr(s)) == OK
    return q, s


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Two int4 codes per byte along each row, low nibble first: uint8 [rows, cols / 2]."""
    q = _c(q, np.int8)
    rows, cols = q.shape
    out = np.empty((rows, cols // 2), np.uint8)
    assert _load().q8o_pack_int4(_ptr(q), rows, cols, _ptr(out)) == OK
    return out


def unpack_int4(packed: np.ndarray, cols: int) -> np.ndarray:
    """Inverse of pack_int4, sign-extending each nibble."""
    packed = _c(packed, np.uint8)
    rows = packed.shape[0]
    out = np.empty((rows, cols), np.int8)
    assert _load().q8o_unpack_int4(_ptr(packed), rows, cols, _ptr(out)) == OK
    return out


def e8m0_ceil(x: float) -> int:
    """E8M0 byte of x rounded up to a power of two (clamped to 103 .. 136)."""
    return int(_load().q8o_e8m0_ceil(ctypes.c_float(x)))


def mx_words(K: int, G: int) -> int:
    """32-bit scale words per weight row: four E8M0 bytes per word."""
    return (K // G + 3) // 4


def quantize_weight_mx(w: np.ndarray, G: int):
    """Block-scaled int8 weights: codes int8 [N, K] and E8M0 scale words uint32
    [ceil(K / G / 4), N] (byte b of word w is group 4w + b; group-major)."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.int8)
    sf = np.empty((mx_words(K, G), N), np.uint32)
    assert _load().q8o_quantize_weight_mx(_ptr(w), N, K, G, _ptr(q), _ptr(sf)) == OK
    return q, sf


def gemm_mx(qa: np.ndarray, q: np.ndarray, sf: np.ndarray, G: int, threads: int = 1):
    """T = sum_k qa * q * s exactly, rounded once to fp32 [M, N]; and sum_k |qa * q * s| (fp64)."""
    qa, q, sf = _c(qa, np.int8), _c(q, np.int8), _c(sf, np.uint32)
    M, K = qa.shape
    N = q.shape[0]
    t = np.empty((M, N), np.float32)
    absum = np.empty((M, N), np.float64)
    assert _load().q8o_gemm_mx(_ptr(qa), _ptr(q), _ptr(sf), M, N, K, G, _ptr(t), _ptr(absum), threads) == OK
    return t, absum


def linear_mx(qa, sa, q, sf, G: int, bias=None, a_per_row: bool = True, threads: int = 1) -> np.ndarray:
    """Block-scaled layer: y = fl(T * s_a[m]) (+ bias[n])."""
    qa, q, sf = _c(qa, np.int8), _c(q, np.int8), _c(sf, np.uint32)
    sa = _c(np.atleast_1d(sa), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    M, K = qa.shape
    N = q.shape[0]
    y = np.empty((M, N), np.float32)
    assert _load().q8o_linear_mx(_ptr(qa), _ptr(sa), 1 if a_per_row else 0, _ptr(q), _ptr(sf), _ptr(b),
                                 M, N, K, G, _ptr(y), threads) == OK
    return y


def to_bf16(y: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, round-to-nearest-even."""
    y = _c(y, np.float32)
    out = np.empty(y.shape, np.uint16)
    _load().q8o_to_bf16(_ptr(y), y.size, _ptr(out))
    return out


def quantize_static(y: np.ndarray, s_out: float) -> np.ndarray:
    """int8 codes clamp(rint(y / s_out), -127, 127) with a fixed output scale."""
    y = _c(y, np.float32)
    q = np.empty(y.shape, np.int8)
    _load().q8o_quantize_static(_ptr(y), y.size, ctypes.c_float(s_out), _ptr(q))
    return q


def linear_codes_at(qa, sa, za, qw, sw, ms, ns, a_per_row: bool, w_per_row: bool):
    """y and int64 acc at the (ms[i], ns[i]) pairs only; returns (y, acc, status)."""
    qa = _c(qa, np.int8)
    qw = _c(qw, np.int8)
    sa = _c(sa, np.float32)
    sw = _c(sw, np.float32)
    za = None if za is None else _c(za, np.int32)
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    K = qa.shape[1]
    y = np.empty(ms.size, np.float32)
    acc = np.empty(ms.size, np.int64)
    st = _load().q8o_linear_codes_at(_ptr(qa), _ptr(sa), _ptr(za), int(a_per_row), _ptr(qw), _ptr(sw),
                                     int(w_per_row), K, _ptr(ms), _ptr(ns), ms.size, _ptr(y), _ptr(acc))
    return y, acc, st


def linear(a: np.ndarray, w: np.ndarray, act_per_row: bool, act_symmetric: bool,
           w_per_row: bool, threads: int = 1):
    """Whole layer from fp32 A[M, K] and W[N, K]: quantize both, integer GEMM, epilogue.

    Returns a dict with qa, sa, za (None if symmetric), qw, sw, colsum, y, status.
    """
    if act_symmetric:
        qa, sa = quantize_sym(a, act_per_row)
        za = None
    else:
        qa, sa, za = quantize_asym(a, act_per_row)
    qw, sw = quantize_sym(w, w_per_row)
    M, N = a.shape[0], w.shape[0]
    y = np.empty((M, N), np.float32)
    lib = _load()
    st = lib.q8o_linear_codes(_ptr(qa), _ptr(sa), _ptr(za), int(act_per_row), _ptr(qw), _ptr(sw),
                              int(w_per_row), M, N, a.shape[1], _ptr(y), threads)
    return dict(qa=qa, sa=sa, za=za, qw=qw, sw=sw, colsum=colsum(qw), y=y, status=st)
