"""Seeded synthetic inputs for the W8A8 quantized linear layer.

This module only draws random floats and integer codes with the shapes and
statistics of the five workloads below. It holds none of the method's
arithmetic (no scales, no rounding, no integer products), so both the CPU
oracle and the CUDA path can take their inputs from here without sharing any
step of the computation.

Workloads (shapes follow the pages: A is [M, K] tokens x features; the weight
matrix is drawn per output channel n and stored K-major as W[N, K], which is
the layout "Write Int8 Quantized Kernel" (Common failure modes) gives for an
(N, K) weight with per-channel scales of shape (N,)):

  tiny      A [16, 256]     N(0,1), channel 7 scaled x30;
            W [128, 256]    row n ~ N(0, sigma_n), sigma_n log-uniform [1/64, 1];
            per-tensor symmetric A and W (seed 0)
  prefill2k A [512, 2048]   N(0,1), 4 fixed outlier channels at +-60, token 0 x20;
            W [2048, 2048]  row std 0.02 * log-uniform [1/64, 1];
            per-token symmetric A, per-channel symmetric W
  relu4k    A [2048, 4096]  max(0, N(0,1)) (ReLU output);
            W [4096, 4096]  row std 0.02 * log-uniform [1/64, 1];
            per-token asymmetric A, per-channel symmetric W
  decode    A [16, 8192]    N(0,1), 8 outlier channels at +-40;
            W [28672, 8192] row std 0.02 * log-uniform [1/16, 1];
            per-token symmetric A, per-channel symmetric W
  prefill16k A [8192, 16384] N(0,1), 16 outlier channels at +-60;
            W [8192, 16384] row std 0.02 * log-uniform [1/64, 1];
            per-token symmetric A, per-channel symmetric W

Outlier channels replace the entries of a channel with +-amplitude, keeping
the sign of the underlying N(0,1) draw; the channel indices are drawn once
from the seeded generator and are the same for every token ("fixed").
Seeds: workload index (tiny=0, prefill2k=1, relu4k=2, decode=3, prefill16k=4).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    act_granularity: str      # "tensor" | "row"  (row = per token)
    act_symmetric: bool
    w_granularity: str        # "tensor" | "row"  (row = per output channel)
    seed: int
    a_kind: str               # "gauss" | "relu"
    a_outlier_channels: int
    a_outlier_amp: float      # replace value with +-amp (0: none)
    a_channel_scale: tuple    # ((channel, factor), ...) multiplicative channel gains
    a_token0_gain: float
    w_std: float
    w_lu_lo: float            # log-uniform lower bound of the per-channel gain


WORKLOADS = {
    "tiny": Workload("tiny", 16, 128, 256, "tensor", True, "tensor", 0,
                     "gauss", 0, 0.0, ((7, 30.0),), 1.0, 1.0, 1.0 / 64),
    "prefill2k": Workload("prefill2k", 512, 2048, 2048, "row", True, "row", 1,
                          "gauss", 4, 60.0, (), 20.0, 0.02, 1.0 / 64),
    "relu4k": Workload("relu4k", 2048, 4096, 4096, "row", False, "row", 2,
                       "relu", 0, 0.0, (), 1.0, 0.02, 1.0 / 64),
    "decode": Workload("decode", 16, 28672, 8192, "row", True, "row", 3,
                       "gauss", 8, 40.0, (), 1.0, 0.02, 1.0 / 16),
    "prefill16k": Workload("prefill16k", 8192, 8192, 16384, "row", True, "row", 4,
                           "gauss", 16, 60.0, (), 1.0, 0.02, 1.0 / 64),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def make_activations(wl: Workload, M: int | None = None, K: int | None = None) -> np.ndarray:
    """fp32 [M, K] activations with the workload's statistics (C-contiguous)."""
    M = wl.M if M is None else M
    K = wl.K if K is None else K
    rng = _rng(wl.seed, 1)
    a = rng.standard_normal((M, K), dtype=np.float32)
    if wl.a_kind == "relu":
        np.maximum(a, 0.0, out=a)
    for ch, gain in wl.a_channel_scale:
        if ch < K:
            a[:, ch] *= np.float32(gain)
    if wl.a_outlier_channels and wl.a_outlier_amp:
        chans = _rng(wl.seed, 2).choice(K, size=min(wl.a_outlier_channels, K), replace=False)
        for ch in chans:
            col = a[:, ch]
            a[:, ch] = np.where(col < 0, -wl.a_outlier_amp, wl.a_outlier_amp).astype(np.float32)
    if wl.a_token0_gain != 1.0 and M > 0:
        a[0, :] *= np.float32(wl.a_token0_gain)
    return np.ascontiguousarray(a)


def make_weights(wl: Workload, N: int | None = None, K: int | None = None) -> np.ndarray:
    """fp32 W[N, K]: output channel n is a row with std w_std * LU[w_lu_lo, 1]."""
    N = wl.N if N is None else N
    K = wl.K if K is None else K
    rng = _rng(wl.seed, 3)
    gains = np.exp(rng.uniform(np.log(wl.w_lu_lo), 0.0, size=N)).astype(np.float32)
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= (np.float32(wl.w_std) * gains)[:, None]
    return np.ascontiguousarray(w)


def random_codes(shape, seed: int, lo: int = -128, hi: int = 127) -> np.ndarray:
    """Uniform int8 codes in [lo, hi] (for GEMM-only cases)."""
    return _rng(seed, 7).integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)


def random_scales(n: int, seed: int, lo: float = 1e-3, hi: float = 1.0) -> np.ndarray:
    """Positive fp32 scales drawn log-uniform in [lo, hi]."""
    r = _rng(seed, 8).uniform(np.log(lo), np.log(hi), size=n)
    return np.exp(r).astype(np.float32)


def random_zero_points(n: int, seed: int) -> np.ndarray:
    return _rng(seed, 9).integers(-128, 128, size=n, dtype=np.int64).astype(np.int32)


def gaussian(shape, seed: int, std: float = 1.0) -> np.ndarray:
    return (_rng(seed, 10).standard_normal(shape, dtype=np.float32) * np.float32(std))


def uniform01(shape, seed: int) -> np.ndarray:
    return _rng(seed, 11).random(shape, dtype=np.float32)


def make_norm_weights(K: int, seed: int = 0) -> np.ndarray:
    """fp32 gamma[K] of an RMSNorm in front of the layer: 1 + 0.1 N(0, 1) per channel."""
    return (np.float32(1.0) + np.float32(0.1) * _rng(seed, 12).standard_normal(K, dtype=np.float32)).astype(np.float32)
