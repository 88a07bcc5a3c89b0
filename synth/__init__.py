"""Seeded synthetic inputs for the PTQ1_0 tests and the benchmark.

Holds random-number generation and storage rounding only (see ``gen.c``); no
step of the ternary matmul, the rotation or the feed-forward block lives here.
Both the CPU oracle and the CUDA library are fed the arrays it returns.

Workload shapes (synthetic stand-ins for the projections of a 27B hybrid
model; the pages measure whole models only):

* tiny matvec      M=1, N=K=1024, one rotation block, seed 0
* decode gate/up   M in {1, 4}, K=5120, N=17408, seed 1
* decode down      M in {1, 8}, K=17408, N=5120, trits P(0)=0.4, seed 2
* prefill          M in {128, 512, 2048}, K=5120, N=17408, bf16 x, seed 3
* feed-forward     64 layers, H=5120, I=17408, M in {1, 256}, seed 4
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libptq_synth.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-Werror", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.syn_trits_uniform.argtypes = [_U64, _U64, _P, _I64]
        L.syn_trits_sparse.argtypes = [_U64, _U64, ctypes.c_double, _P, _I64]
        L.syn_signs.argtypes = [_U64, _U64, _P, _I64]
        L.syn_normal_f64.argtypes = [_U64, _U64, _P, _I64]
        L.syn_normal_f32.argtypes = [_U64, _U64, _P, _I64]
        L.syn_normal_bf16.argtypes = [_U64, _U64, _P, _I64]
        L.syn_abs_normal_f16.argtypes = [_U64, _U64, ctypes.c_double, _P, _I64]
        L.syn_token_ids.argtypes = [_U64, _U64, _I64, _P, _I64]
        for f in ("syn_trits_uniform", "syn_trits_sparse", "syn_signs", "syn_normal_f64",
                  "syn_normal_f32", "syn_normal_bf16", "syn_abs_normal_f16", "syn_token_ids"):
            getattr(L, f).restype = None
        L.syn_half_bits.argtypes = [ctypes.c_double]
        L.syn_half_bits.restype = ctypes.c_uint16
        L.syn_bf16_bits.argtypes = [ctypes.c_float]
        L.syn_bf16_bits.restype = ctypes.c_uint16
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def trits_uniform(seed: int, stream: int, shape, out=None) -> np.ndarray:
    a = np.empty(shape, np.int8) if out is None else out
    lib().syn_trits_uniform(seed, stream, _p(a), a.size)
    return a


def trits_sparse(seed: int, stream: int, shape, p_zero: float, out=None) -> np.ndarray:
    a = np.empty(shape, np.int8) if out is None else out
    lib().syn_trits_sparse(seed, stream, float(p_zero), _p(a), a.size)
    return a


def signs(seed: int, stream: int, n: int) -> np.ndarray:
    a = np.empty(n, np.int8)
    lib().syn_signs(seed, stream, _p(a), n)
    return a


def normal_f64(seed: int, stream: int, shape) -> np.ndarray:
    a = np.empty(shape, np.float64)
    lib().syn_normal_f64(seed, stream, _p(a), a.size)
    return a


def normal_f32(seed: int, stream: int, shape) -> np.ndarray:
    a = np.empty(shape, np.float32)
    lib().syn_normal_f32(seed, stream, _p(a), a.size)
    return a


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws."""
    a = np.empty(shape, np.uint16)
    lib().syn_normal_bf16(seed, stream, _p(a), a.size)
    return a


def scales_f16(seed: int, stream: int, shape, sigma: float = 0.02, out=None) -> np.ndarray:
    """fp16 bit patterns (uint16) of sigma * |N(0,1)|."""
    a = np.empty(shape, np.uint16) if out is None else out
    lib().syn_abs_normal_f16(seed, stream, float(sigma), _p(a), a.size)
    return a


def token_ids(seed: int, stream: int, n: int, V: int) -> np.ndarray:
    """n int32 token ids, uniform over [0, V)."""
    a = np.empty(n, np.int32)
    lib().syn_token_ids(seed, stream, int(V), _p(a), n)
    return a


def half_bits(v: float) -> int:
    return int(lib().syn_half_bits(float(v)))


def bf16_bits(v: float) -> int:
    return int(lib().syn_bf16_bits(float(v)))


# ---- workload recipes ------------------------------------------------------
# Streams: 0 trits, 1 scales, 2 activations, 3 signs (first rotation),
# 4 signs (second rotation), 5 second activation factor; per-layer streams of
# the feed-forward workload are offset by 16 * layer.

@dataclass
class Matvec:
    trits: np.ndarray      # N x K int8
    scales: np.ndarray     # N x K/128 uint16 (fp16 bits)
    x: np.ndarray          # M x K float32, or uint16 (bf16 bits)
    signs: np.ndarray      # K int8


def weights(seed: int, N: int, K: int, p_zero: float | None = None, stream_base: int = 0):
    """Trits (uniform, or P(0)=p_zero and P(+-1) equal) and fp16 scales."""
    if p_zero is None:
        t = trits_uniform(seed, stream_base + 0, (N, K))
    else:
        t = trits_sparse(seed, stream_base + 0, (N, K), p_zero)
    s = scales_f16(seed, stream_base + 1, (N, K // 128))
    return t, s


def gaussian_matvec(seed: int, M: int, N: int, K: int, dtype: str = "f32",
                    p_zero: float | None = None) -> Matvec:
    """Weights as above; x ~ N(0,1) as fp32 or bf16; one sign per element.

    A rotated N(0, I) vector is again N(0, I) (the rotation is orthogonal), so
    pre-rotated Gaussian activations are drawn as plain Gaussians.
    """
    t, s = weights(seed, N, K, p_zero)
    x = normal_f32(seed, 2, (M, K)) if dtype == "f32" else normal_bf16(seed, 2, (M, K))
    return Matvec(t, s, x, signs(seed, 3, K))


def gated_pair(seed: int, M: int, K: int):
    """The two N(0,1) factors (a, b) of the decode-down activations."""
    return normal_f64(seed, 2, (M, K)), normal_f64(seed, 5, (M, K))


@dataclass
class FfnLayer:
    wgu_trits: np.ndarray   # 2I x H
    wgu_scales: np.ndarray  # 2I x H/128
    wd_trits: np.ndarray    # H x I
    wd_scales: np.ndarray   # H x I/128
    signs_in: np.ndarray    # H
    signs_mid: np.ndarray   # I


def ffn_layer(seed: int, layer: int, H: int, I: int) -> FfnLayer:
    """Weights and signs of one feed-forward layer (streams offset by 16 * layer)."""
    base = 16 * layer
    t_gu, s_gu = weights(seed, 2 * I, H, stream_base=base + 0)
    t_d, s_d = weights(seed, H, I, stream_base=base + 8)
    return FfnLayer(t_gu, s_gu, t_d, s_d, signs(seed, base + 4, H), signs(seed, base + 5, I))


def ffn_input(seed: int, layer: int, M: int, H: int, dtype: str = "f32") -> np.ndarray:
    base = 16 * layer
    return normal_f32(seed, base + 6, (M, H)) if dtype == "f32" else normal_bf16(seed, base + 6, (M, H))


def norm_gain(seed: int, layer: int, H: int) -> np.ndarray:
    """RMSNorm gains of one layer, fp32: 1 + 0.1 N(0, 1) (stream 16 * layer + 7)."""
    return (1.0 + 0.1 * normal_f64(seed, 16 * layer + 7, (H,))).astype(np.float32)
