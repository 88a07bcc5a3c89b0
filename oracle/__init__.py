"""CPU oracle for the PTQ1_0 ternary matmul and the signed Walsh-Hadamard
rotation -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does.  The
arithmetic lives in ``ptq_oracle.c`` (plain C, fp64); this module only builds
it with gcc and marshals numpy arrays through ctypes.

Sources: "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", sections
"What Bonsai is", "What Ferrox does with it" and "Speed, and where it goes".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ptq_oracle.c")
_LIB = os.path.join(_HERE, "libptq_oracle.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "ptq_oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
             "-Wall", "-Wextra", "-Werror", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_half_to_double.restype = ctypes.c_double
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        for name in ("orc_decode_f16", "orc_decode_bf16", "orc_decode_f32"):
            getattr(L, name).argtypes = [_P, _P, _I64]
            getattr(L, name).restype = None
        L.orc_peel_digit.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.orc_peel_digit.restype = ctypes.c_int
        L.orc_pack.argtypes = [_P, _P, _I64, _I64]
        L.orc_pack.restype = ctypes.c_int
        L.orc_unpack.argtypes = [_P, _P, _I64, _I64]
        L.orc_unpack.restype = ctypes.c_int
        for name in ("orc_fwht_def", "orc_fwht_fast"):
            getattr(L, name).argtypes = [_P, _P, _P, _I64, _I64]
            getattr(L, name).restype = None
        L.orc_pq2_pack.argtypes = [_P, _P, _I64, _I64]
        L.orc_pq2_pack.restype = ctypes.c_int
        L.orc_pq2_unpack.argtypes = [_P, _P, _I64, _I64]
        L.orc_pq2_unpack.restype = ctypes.c_int
        L.orc_pq2_matmul.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64]
        L.orc_pq2_matmul.restype = None
        L.orc_pq2_matmul_rows.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64]
        L.orc_pq2_matmul_rows.restype = None
        L.orc_unrotate_def.argtypes = [_P, _P, _P, _I64, _I64]
        L.orc_unrotate_def.restype = None
        L.orc_embed.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64]
        L.orc_embed.restype = None
        L.orc_embed_ptq1.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64]
        L.orc_embed_ptq1.restype = ctypes.c_int
        L.orc_matmul.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64]
        L.orc_matmul.restype = None
        L.orc_matmul_rows.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64]
        L.orc_matmul_rows.restype = None
        L.orc_swiglu.argtypes = [_P, _P, _P, _I64]
        L.orc_swiglu.restype = None
        L.orc_ffn.argtypes = [_P] * 8 + [_I64] * 3
        L.orc_ffn.restype = ctypes.c_int
        L.orc_ffn_stack.argtypes = [_P] * 7 + [_I64, ctypes.c_double, _P, _I64, _I64, _I64]
        L.orc_ffn_stack.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = None
        L.orc_get_threads.argtypes = []
        L.orc_get_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def half_to_double(bits: int) -> float:
    return float(lib().orc_half_to_double(int(bits)))


def decode_f16(bits: np.ndarray) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().orc_decode_f16(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().orc_decode_bf16(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_f32(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.float64)
    lib().orc_decode_f32(_ptr(x), _ptr(out), x.size)
    return out


def peel_digit(byte: int, n: int) -> int:
    return int(lib().orc_peel_digit(int(byte), int(n)))


def pack(trits: np.ndarray) -> np.ndarray:
    """N x K int8 trits -> N x (K/128*26) uint8 (raises on invalid input)."""
    trits = _c(trits, np.int8)
    N, K = trits.shape
    wq = np.empty((N, (K // 128) * 26), np.uint8)
    if lib().orc_pack(_ptr(trits), _ptr(wq), N, K) != 0:
        raise ValueError("orc_pack: trit outside {-1,0,1} or K % 128 != 0")
    return wq


def unpack(wq: np.ndarray, K: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    N = wq.shape[0]
    trits = np.empty((N, K), np.int8)
    if lib().orc_unpack(_ptr(wq), _ptr(trits), N, K) != 0:
        raise ValueError("orc_unpack: K % 128 != 0")
    return trits


def pq2_pack(trits: np.ndarray) -> np.ndarray:
    """N x K int8 trits -> N x (K/128*32) uint8 PQ2_0 codes (raises on invalid input)."""
    trits = _c(trits, np.int8)
    N, K = trits.shape
    wq = np.empty((N, (K // 128) * 32), np.uint8)
    if lib().orc_pq2_pack(_ptr(trits), _ptr(wq), N, K) != 0:
        raise ValueError("orc_pq2_pack: trit outside {-1,0,1} or K % 128 != 0")
    return wq


def pq2_unpack(wq: np.ndarray, K: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    N = wq.shape[0]
    trits = np.empty((N, K), np.int8)
    if lib().orc_pq2_unpack(_ptr(wq), _ptr(trits), N, K) != 0:
        raise ValueError("orc_pq2_unpack: K % 128 != 0")
    return trits


def pq2_matmul(wq: np.ndarray, scales: np.ndarray, x: np.ndarray) -> np.ndarray:
    """x (M x K float64) -> y (M x N float64), PQ2_0 weights."""
    wq = _c(wq, np.uint8)
    scales = _c(scales, np.uint16)
    x = _c(x, np.float64)
    M, K = x.shape
    N = wq.shape[0]
    y = np.empty((M, N), np.float64)
    lib().orc_pq2_matmul(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), M, N, K)
    return y


def pq2_matmul_rows(wq, scales, x, rows) -> np.ndarray:
    wq = _c(wq, np.uint8)
    scales = _c(scales, np.uint16)
    x = _c(x, np.float64)
    rows = _c(np.asarray(rows, np.int64), np.int64)
    M, K = x.shape
    y = np.empty((M, rows.size), np.float64)
    lib().orc_pq2_matmul_rows(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), M, wq.shape[0], K,
                              _ptr(rows), rows.size)
    return y


def fwht_def(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    x2 = x.reshape(-1, x.shape[-1])
    signs = _c(signs, np.int8)
    y = np.empty_like(x2)
    lib().orc_fwht_def(_ptr(x2), _ptr(signs), _ptr(y), x2.shape[0], x2.shape[1])
    return y.reshape(x.shape)


def fwht(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    x2 = x.reshape(-1, x.shape[-1])
    signs = _c(signs, np.int8)
    y = np.empty_like(x2)
    lib().orc_fwht_fast(_ptr(x2), _ptr(signs), _ptr(y), x2.shape[0], x2.shape[1])
    return y.reshape(x.shape)


def unrotate_def(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R^T y per 1024-block, by the definition (O(1024^2) per block)."""
    y = _c(y, np.float64)
    y2 = y.reshape(-1, y.shape[-1])
    signs = _c(signs, np.int8)
    x = np.empty_like(y2)
    lib().orc_unrotate_def(_ptr(y2), _ptr(signs), _ptr(x), y2.shape[0], y2.shape[1])
    return x.reshape(y.shape)


def embed(table: np.ndarray, ids: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """out[m] = R^T table[ids[m]] (V x H float64 table); NaN rows for bad ids."""
    table = _c(table, np.float64)
    ids = _c(np.asarray(ids, np.int32), np.int32)
    signs = _c(signs, np.int8)
    V, H = table.shape
    out = np.empty((ids.size, H), np.float64)
    lib().orc_embed(_ptr(table), _ptr(ids), _ptr(signs), _ptr(out), ids.size, V, H)
    return out


def embed_ptq1(wq: np.ndarray, scales: np.ndarray, ids: np.ndarray,
               signs: np.ndarray) -> np.ndarray:
    """The same for a PTQ1_0 table (wq V x H/128*26, scales V x H/128)."""
    wq = _c(wq, np.uint8)
    scales = _c(scales, np.uint16)
    ids = _c(np.asarray(ids, np.int32), np.int32)
    signs = _c(signs, np.int8)
    V, H = scales.shape[0], scales.shape[1] * 128
    out = np.empty((ids.size, H), np.float64)
    if lib().orc_embed_ptq1(_ptr(wq), _ptr(scales), _ptr(ids), _ptr(signs), _ptr(out),
                            ids.size, V, H) != 0:
        raise ValueError("orc_embed_ptq1: H % 1024 != 0 or allocation failure")
    return out


def matmul(wq: np.ndarray, scales: np.ndarray, x: np.ndarray) -> np.ndarray:
    """x (M x K float64) -> y (M x N float64)."""
    wq = _c(wq, np.uint8)
    scales = _c(scales, np.uint16)
    x = _c(x, np.float64)
    M, K = x.shape
    N = wq.shape[0]
    y = np.empty((M, N), np.float64)
    lib().orc_matmul(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), M, N, K)
    return y


def matmul_rows(wq, scales, x, rows) -> np.ndarray:
    """Oracle outputs for the listed rows only: returns M x len(rows)."""
    wq = _c(wq, np.uint8)
    scales = _c(scales, np.uint16)
    x = _c(x, np.float64)
    rows = _c(np.asarray(rows, np.int64), np.int64)
    M, K = x.shape
    y = np.empty((M, rows.size), np.float64)
    lib().orc_matmul_rows(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), M, wq.shape[0], K,
                          _ptr(rows), rows.size)
    return y


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    h = np.empty_like(g)
    lib().orc_swiglu(_ptr(g), _ptr(u), _ptr(h), g.size)
    return h


def ffn(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x) -> np.ndarray:
    """y = W_d R_mid (silu(g) * u), [g; u] = W_gu R_in x; all float64."""
    wgu_q = _c(wgu_q, np.uint8)
    wgu_s = _c(wgu_s, np.uint16)
    wd_q = _c(wd_q, np.uint8)
    wd_s = _c(wd_s, np.uint16)
    signs_in = _c(signs_in, np.int8)
    signs_mid = _c(signs_mid, np.int8)
    x = _c(x, np.float64)
    M, H = x.shape
    I = signs_mid.size
    y = np.empty((M, H), np.float64)
    rc = lib().orc_ffn(_ptr(wgu_q), _ptr(wgu_s), _ptr(wd_q), _ptr(wd_s), _ptr(signs_in),
                       _ptr(signs_mid), _ptr(x), _ptr(y), M, H, I)
    if rc != 0:
        raise ValueError("orc_ffn: H and I must be multiples of 1024")
    return y


def ffn_stack(layers, norm_w, x, eps: float) -> np.ndarray:
    """The pre-norm residual stack: for each layer l,
    x = x + ffn_l(x / sqrt(mean(x^2) + eps) * g_l).  `layers` is a list of
    (wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid); norm_w a list of H-vectors."""
    Lc = len(layers)
    if Lc == 0:
        return np.array(x, dtype=np.float64, copy=True, order="C")
    cols = [[_c(lay[i], dt) for lay in layers]
            for i, dt in enumerate((np.uint8, np.uint16, np.uint8, np.uint16, np.int8, np.int8))]
    gs = [_c(np.asarray(g, np.float64), np.float64) for g in norm_w]
    arrs = [(ctypes.c_void_p * Lc)(*[a.ctypes.data for a in col]) for col in cols]
    garr = (ctypes.c_void_p * Lc)(*[g.ctypes.data for g in gs])
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    M, H = x.shape
    I = cols[5][0].size
    rc = lib().orc_ffn_stack(*[ctypes.cast(a, ctypes.c_void_p) for a in arrs],
                             ctypes.cast(garr, ctypes.c_void_p), Lc, float(eps), _ptr(x), M, H, I)
    if rc != 0:
        raise ValueError("orc_ffn_stack: H and I must be multiples of 1024")
    return x

