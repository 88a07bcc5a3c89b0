"""Python binding of libptq.so, the GB300 (sm_103a) PTQ1_0 ternary matmul
library (C ABI in include/ptq.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library is missing or a call fails,
these functions raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

LIB_PATH = _build.LIB

PTQ_F32 = 0
PTQ_BF16 = 1

STATUS = {
    0: "PTQ_OK", 1: "PTQ_ERR_NULL", 2: "PTQ_ERR_SHAPE", 3: "PTQ_ERR_ALIGN", 4: "PTQ_ERR_VALUE",
    5: "PTQ_ERR_UNSUPPORTED", 6: "PTQ_ERR_WORKSPACE", 7: "PTQ_ERR_CUDA", 8: "PTQ_ERR_TIMEOUT",
    9: "PTQ_ERR_RANGE",
}

# Every symbol include/ptq.h declares.
EXPORTS = ("ptq1_pack", "ptq1_unpack", "ptq_fwht", "ptq_matmul_workspace_bytes", "ptq_matmul",
           "ptq_rotate_matmul_workspace_bytes", "ptq_rotate_matmul",
           "ptq_rotate_matmul_host_workspace_bytes", "ptq_rotate_matmul_host", "ptq_ffn_workspace_bytes",
           "ptq_ffn", "ptq_ffn_noalloc", "ptq_ffn_stack_workspace_bytes", "ptq_ffn_stack",
           "ptq_ffn_stack_ex", "ptq_ffn_stack_route", "ptq2_pack", "ptq2_unpack",
           "ptq_matmul_pq2_workspace_bytes", "ptq_matmul_pq2", "ptq_embed", "ptq_embed_ptq1",
           "ptq_route", "ptq_gemv_plan", "ptq_matmul_bf16_accumulator", "ptq_matmul_f32_peel",
           "ptq_selftest_timeout",
           "ptq_selftest_grid_timeout",
           "ptq_device_check", "ptq_status_str", "ptq_last_error")

# Size of the built-in scratch array behind ptq_ffn_noalloc (include/ptq.h).
FFN_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024


class PTQError(RuntimeError):
    def __init__(self, status: int, call: str, message: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{call}: {self.name}: {message}")


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def load(path: str | None = None):
    """Load libptq.so (building it first if it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        _build.build()
    L = ctypes.CDLL(path)
    L.ptq1_pack.argtypes = [_P, _P, _I64, _I64]
    L.ptq1_unpack.argtypes = [_P, _P, _I64, _I64, _P]
    L.ptq_fwht.argtypes = [_P, _P, _P, _I64, _I64, _I32, _P]
    L.ptq_matmul_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_matmul_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_matmul.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, ctypes.c_size_t, _P]
    L.ptq_rotate_matmul_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_rotate_matmul_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_rotate_matmul_host_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_rotate_matmul_host_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_rotate_matmul_host.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P,
                                         ctypes.c_size_t, _P]
    L.ptq_rotate_matmul_host.restype = _I32
    L.ptq_rotate_matmul.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, ctypes.c_size_t,
                                    _P]
    L.ptq_ffn_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_ffn_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_ffn.argtypes = [_P] * 8 + [_I64, _I64, _I64, _I32, _P, ctypes.c_size_t, _P]
    L.ptq_ffn_noalloc.argtypes = [_P] * 8 + [_I64, _I64, _I64, _I32, _P]
    L.ptq_ffn_stack_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_ffn_stack_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_ffn_stack.argtypes = [_P, _I64, _P, _I64, _I64, _I64, ctypes.c_float, _I32, _P,
                                ctypes.c_size_t, _P]
    L.ptq_ffn_stack_ex.argtypes = [_P, _I64, _P, _I64, _I64, _I64, ctypes.c_float, _I32, _P,
                                   ctypes.c_size_t, ctypes.c_uint, _P]
    L.ptq_ffn_stack_route.argtypes = [_I64, _I64, _I64, _I32, ctypes.POINTER(ctypes.c_char_p)]
    L.ptq2_pack.argtypes = [_P, _P, _I64, _I64]
    L.ptq2_unpack.argtypes = [_P, _P, _I64, _I64, _P]
    L.ptq_matmul_pq2_workspace_bytes.argtypes = [_I64, _I64, _I64, _I32]
    L.ptq_matmul_pq2_workspace_bytes.restype = ctypes.c_size_t
    L.ptq_matmul_pq2.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, ctypes.c_size_t, _P]
    L.ptq_embed.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P]
    L.ptq_embed_ptq1.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P]
    L.ptq_route.argtypes = [_I64, _I32, ctypes.POINTER(ctypes.c_char_p)]
    L.ptq_gemv_plan.argtypes = [_I64, _I64, _I64, _I32, ctypes.POINTER(ctypes.c_int32)]
    L.ptq_matmul_f32_peel.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P]
    L.ptq_matmul_f32_peel.restype = _I32
    L.ptq_matmul_bf16_accumulator.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _P,
                                              ctypes.c_size_t, _P]
    L.ptq_device_check.argtypes = [_P]
    L.ptq_selftest_timeout.argtypes = [_P]
    L.ptq_selftest_grid_timeout.argtypes = [_P]
    L.ptq_status_str.argtypes = [_I32]
    L.ptq_status_str.restype = ctypes.c_char_p
    L.ptq_last_error.argtypes = []
    L.ptq_last_error.restype = ctypes.c_char_p
    for name in ("ptq1_pack", "ptq1_unpack", "ptq_fwht", "ptq_matmul", "ptq_rotate_matmul", "ptq_ffn",
                 "ptq_ffn_noalloc", "ptq_ffn_stack", "ptq_ffn_stack_ex", "ptq_ffn_stack_route", "ptq2_pack",
                 "ptq2_unpack", "ptq_matmul_pq2", "ptq_embed",
                 "ptq_embed_ptq1", "ptq_route", "ptq_gemv_plan", "ptq_device_check",
                 "ptq_selftest_timeout", "ptq_selftest_grid_timeout"):
        getattr(L, name).restype = _I32
    _lib = L
    return L


def _check(status: int, call: str) -> None:
    if status != 0:
        msg = load().ptq_last_error().decode(errors="replace")
        raise PTQError(status, call, msg)


def _stream(stream=None, device=None) -> int:
    """The raw handle of `stream`, else of PyTorch's current stream on
    `device` (an index; the current device when None)."""
    import torch

    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:  # no Stream object per call
        return raw(torch.cuda.current_device() if device is None else device)
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t, dtype=None, name="tensor"):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _act_dtype(t):
    import torch

    if t.dtype == torch.float32:
        return PTQ_F32
    if t.dtype == torch.bfloat16:
        return PTQ_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


# ---- host encoder ------------------------------------------------------------

def pack(trits: np.ndarray) -> np.ndarray:
    """ptq1_pack: N x K int8 trits -> N x (K/128*26) uint8 (host)."""
    trits = np.ascontiguousarray(trits, dtype=np.int8)
    if trits.ndim != 2:
        raise ValueError("trits must be 2-D")
    N, K = trits.shape
    out = np.empty((N, (K // 128) * 26 if K % 128 == 0 else 0), np.uint8)
    _check(load().ptq1_pack(ctypes.c_void_p(trits.ctypes.data), ctypes.c_void_p(out.ctypes.data),
                            N, K), "ptq1_pack")
    return out


# ---- device calls --------------------------------------------------------------

def unpack(wq, K: int, stream=None):
    import torch

    N = wq.shape[0]
    out = torch.empty((N, K), dtype=torch.int8, device=wq.device)
    _check(load().ptq1_unpack(_dev(wq, torch.uint8, "wq"), _dev(out), N, K, _stream(stream)),
           "ptq1_unpack")
    return out


def fwht(x, signs, out=None, stream=None):
    """Signed 1024-wide rotation of the rows of x (in place when out is x)."""
    import torch

    y = torch.empty_like(x) if out is None else out
    M, K = x.shape
    _check(load().ptq_fwht(_dev(x, None, "x"), _dev(y, x.dtype, "out"), _dev(signs, torch.int8, "signs"),
                           M, K, _act_dtype(x), _stream(stream)), "ptq_fwht")
    return y


def matmul_workspace_bytes(M: int, N: int, K: int, dtype: int) -> int:
    return int(load().ptq_matmul_workspace_bytes(M, N, K, dtype))


def matmul(wq, scales, x, out=None, workspace=None, stream=None):
    """y = x W^T, W the PTQ1_0 weight (N x K); x M x K (float32 or bfloat16).
    The scratch the call needs (ptq_matmul_workspace_bytes) is allocated by
    PyTorch here when `workspace` is not given."""
    import torch

    M, K = x.shape
    N = wq.shape[0]
    dt = _act_dtype(x)
    y = torch.empty((M, N), dtype=x.dtype, device=x.device) if out is None else out
    need = matmul_workspace_bytes(M, N, K, dt)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws = _dev(workspace, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ptq_matmul(_dev(wq, torch.uint8, "wq"), _dev(scales, torch.int16, "scales"),
                             _dev(x, None, "x"), _dev(y, x.dtype, "out"), M, N, K, dt, ws,
                             ws_bytes, _stream(stream)), "ptq_matmul")
    return y


def matmul_bf16_accumulator(wq, scales, x, stream=None):
    """Test export: the bf16 prefill GEMM's fp32 accumulator (y = x W^T with
    x bfloat16, y float32), the same kernel as matmul() on bfloat16 input
    without the output's bf16 rounding."""
    import torch

    M, K = x.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    need = matmul_workspace_bytes(M, N, K, PTQ_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device=x.device) if need > 0 else None
    _check(load().ptq_matmul_bf16_accumulator(
        _dev(wq, torch.uint8, "wq"), _dev(scales, torch.int16, "scales"),
        _dev(x, torch.bfloat16, "x"), _dev(y, torch.float32, "out"), M, N, K,
        _dev(ws, None, "workspace") if ws is not None else None, need, _stream(stream)),
        "ptq_matmul_bf16_accumulator")
    return y


def pq2_pack(trits: np.ndarray) -> np.ndarray:
    """ptq2_pack: N x K int8 trits -> N x (K/128*32) uint8 PQ2_0 codes (host)."""
    trits = np.ascontiguousarray(trits, dtype=np.int8)
    if trits.ndim != 2:
        raise ValueError("trits must be 2-D")
    N, K = trits.shape
    out = np.empty((N, K // 4 if K % 128 == 0 else 0), np.uint8)
    _check(load().ptq2_pack(ctypes.c_void_p(trits.ctypes.data), ctypes.c_void_p(out.ctypes.data),
                            N, K), "ptq2_pack")
    return out


def pq2_unpack(wq, K: int, stream=None):
    import torch

    N = wq.shape[0]
    out = torch.empty((N, K), dtype=torch.int8, device=wq.device)
    _check(load().ptq2_unpack(_dev(wq, torch.uint8, "wq"), _dev(out), N, K, _stream(stream)),
           "ptq2_unpack")
    return out


def matmul_pq2_workspace_bytes(M: int, N: int, K: int, dtype: int) -> int:
    return int(load().ptq_matmul_pq2_workspace_bytes(M, N, K, dtype))


def matmul_pq2(wq, scales, x, out=None, workspace=None, stream=None):
    """y = x W^T over PQ2_0 weights (ptq_matmul_pq2); as matmul otherwise."""
    import torch

    M, K = x.shape
    N = wq.shape[0]
    dt = _act_dtype(x)
    y = torch.empty((M, N), dtype=x.dtype, device=x.device) if out is None else out
    need = matmul_pq2_workspace_bytes(M, N, K, dt)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws = _dev(workspace, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ptq_matmul_pq2(_dev(wq, torch.uint8, "wq"), _dev(scales, torch.int16, "scales"),
                                 _dev(x, None, "x"), _dev(y, x.dtype, "out"), M, N, K, dt, ws,
                                 ws_bytes, _stream(stream)), "ptq_matmul_pq2")
    return y


def rotate_matmul_workspace_bytes(M: int, N: int, K: int, dtype: int) -> int:
    return int(load().ptq_rotate_matmul_workspace_bytes(M, N, K, dtype))


def rotate_matmul_host_workspace_bytes(M: int, N: int, K: int, dtype: int) -> int:
    return int(load().ptq_rotate_matmul_host_workspace_bytes(M, N, K, dtype))


def rotate_matmul_host(wq, scales, x_host, signs, y_host, workspace, stream=None):
    """ptq_rotate_matmul_host: x_host (M x K) and y_host (M x N) are CPU
    tensors (page-locked for asynchronous copies) of one dtype, float32 or
    bfloat16; the copies and the product are queued on the stream, and
    y_host is valid once it is synchronised."""
    import torch

    M, K = x_host.shape
    N = wq.shape[0]
    dt = _act_dtype(x_host)
    for t, name in ((x_host, "x_host"), (y_host, "y_host")):
        if t.is_cuda or not t.is_contiguous() or t.dtype != x_host.dtype:
            raise TypeError(f"{name} must be a contiguous CPU tensor of the activations' dtype")
    if tuple(y_host.shape) != (M, N):
        raise ValueError(f"y_host must be {M} x {N}")
    _check(load().ptq_rotate_matmul_host(
        _dev(wq, torch.uint8, "wq"), _dev(scales, torch.int16, "scales"), x_host.data_ptr(),
        _dev(signs, torch.int8, "signs"), y_host.data_ptr(), M, N, K, dt,
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream, wq.device.index)), "ptq_rotate_matmul_host")
    return y_host


def rotate_matmul(wq, scales, x, signs, out=None, workspace=None, stream=None):
    """y = (R x) W^T: the signed rotation of `x` (not modified), then the
    PTQ1_0 matmul; fused into one kernel on the fp32 M = 1 route.  The
    scratch is allocated by PyTorch here when `workspace` is not given."""
    import torch

    M, K = x.shape
    N = wq.shape[0]
    dt = _act_dtype(x)
    y = torch.empty((M, N), dtype=x.dtype, device=x.device) if out is None else out
    if workspace is None:
        workspace = torch.empty(max(1, rotate_matmul_workspace_bytes(M, N, K, dt)),
                                dtype=torch.uint8, device=x.device)
    _check(load().ptq_rotate_matmul(_dev(wq, torch.uint8, "wq"),
                                    _dev(scales, torch.int16, "scales"), _dev(x, None, "x"),
                                    _dev(signs, torch.int8, "signs"), _dev(y, x.dtype, "out"), M, N,
                                    K, dt, _dev(workspace, None, "workspace"),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "ptq_rotate_matmul")
    return y


def ffn_workspace_bytes(M: int, H: int, I: int, dtype: int) -> int:
    return int(load().ptq_ffn_workspace_bytes(M, H, I, dtype))


def ffn(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, out=None, workspace=None, stream=None):
    """The feed-forward block: rotate, gate+up, SwiGLU, rotate, down."""
    import torch

    M, H = x.shape
    I = signs_mid.shape[0]
    dt = _act_dtype(x)
    need = ffn_workspace_bytes(M, H, I, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    y = torch.empty_like(x) if out is None else out
    _check(load().ptq_ffn(_dev(wgu_q, torch.uint8, "wgu_q"), _dev(wgu_s, torch.int16, "wgu_s"),
                          _dev(wd_q, torch.uint8, "wd_q"), _dev(wd_s, torch.int16, "wd_s"),
                          _dev(signs_in, torch.int8, "signs_in"),
                          _dev(signs_mid, torch.int8, "signs_mid"), _dev(x, None, "x"),
                          _dev(y, x.dtype, "out"), M, H, I, dt, _dev(workspace, None, "workspace"),
                          workspace.numel() * workspace.element_size(), _stream(stream)),
           "ptq_ffn")
    return y


class FfnLayer(ctypes.Structure):
    """One layer of ptq_ffn_stack (include/ptq.h): device addresses."""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("wgu_q", "wgu_s", "wd_q", "wd_s", "signs_in", "signs_mid", "norm_w")]


def ffn_stack_workspace_bytes(M: int, H: int, I: int, dtype: int) -> int:
    return int(load().ptq_ffn_stack_workspace_bytes(M, H, I, dtype))


def ffn_stack_route(M: int, H: int, I: int, dtype: int) -> str:
    """The implementation ptq_ffn_stack uses for (M, H, I, dtype) here."""
    name = ctypes.c_char_p()
    _check(load().ptq_ffn_stack_route(M, H, I, dtype, ctypes.byref(name)), "ptq_ffn_stack_route")
    return name.value.decode()


PTQ_STACK_DETERMINISTIC = 1


def ffn_stack(layers, norm_w, x, eps: float, act=None, workspace=None, stream=None,
              deterministic: bool = False):
    """L chained pre-norm feed-forward blocks over the fp32 residual stream x
    (M x H, updated in place and returned): x += ffn_l(rmsnorm(x) * g_l).
    `layers`: per layer (wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid) as for
    ffn(); `norm_w`: per layer an H-vector of fp32 gains.  `act` is the
    blocks' activation dtype, torch.float32 (default) or torch.bfloat16.
    `deterministic` takes the bitwise-reproducible per-layer path."""
    import torch

    if len(layers) != len(norm_w):
        raise ValueError("layers and norm_w differ in length")
    M, H = x.shape
    L = len(layers)
    I = layers[0][5].shape[0] if L else 1024
    dt = _act_dtype(torch.empty(0, dtype=act or torch.float32))
    need = ffn_stack_workspace_bytes(M, H, I, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    arr = (FfnLayer * max(L, 1))()
    names = ("wgu_q", "wgu_s", "wd_q", "wd_s", "signs_in", "signs_mid")
    types = (torch.uint8, torch.int16, torch.uint8, torch.int16, torch.int8, torch.int8)
    for l, (lay, g) in enumerate(zip(layers, norm_w)):
        ptrs = [_dev(t, ty, f"layers[{l}].{n}") for t, ty, n in zip(lay, types, names)]
        ptrs.append(_dev(g, torch.float32, f"norm_w[{l}]"))
        arr[l] = FfnLayer(*ptrs)
    _check(load().ptq_ffn_stack_ex(ctypes.cast(arr, ctypes.c_void_p), L,
                                   _dev(x, torch.float32, "x"), M, H, I, float(eps), dt,
                                   _dev(workspace, None, "workspace"),
                                   workspace.numel() * workspace.element_size(),
                                   PTQ_STACK_DETERMINISTIC if deterministic else 0, _stream(stream)),
           "ptq_ffn_stack")
    return x


def ffn_noalloc(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, out=None, stream=None):
    """The feed-forward block without a workspace: for callers that cannot
    allocate device memory (graph capture, real-time loops, memory owned by
    another allocator).  Its scratch is one built-in device array of
    FFN_NOALLOC_SCRATCH_BYTES shared by all calls, so calls that overlap on
    the GPU race; larger shapes raise PTQ_ERR_WORKSPACE.  Only `out` (if not
    given) is allocated here, by PyTorch, before the call."""
    import torch

    M, H = x.shape
    I = signs_mid.shape[0]
    y = torch.empty_like(x) if out is None else out
    _check(load().ptq_ffn_noalloc(_dev(wgu_q, torch.uint8, "wgu_q"), _dev(wgu_s, torch.int16, "wgu_s"),
                                  _dev(wd_q, torch.uint8, "wd_q"), _dev(wd_s, torch.int16, "wd_s"),
                                  _dev(signs_in, torch.int8, "signs_in"),
                                  _dev(signs_mid, torch.int8, "signs_mid"), _dev(x, None, "x"),
                                  _dev(y, x.dtype, "out"), M, H, I, _act_dtype(x), _stream(stream)),
           "ptq_ffn_noalloc")
    return y


def embed(table, ids, signs, out=None, stream=None):
    """out[m] = R^T table[ids[m]]: the lookup on a rotated embedding table
    (ptq_embed).  table: V x H float32 or bfloat16; ids: M int32 token ids;
    ids outside [0, V) give rows of NaN."""
    import torch

    dt = _act_dtype(table)
    V, H = table.shape
    M = ids.numel()
    y = torch.empty((M, H), dtype=table.dtype, device=table.device) if out is None else out
    _check(load().ptq_embed(_dev(table, None, "table"), _dev(ids, torch.int32, "ids"),
                            _dev(signs, torch.int8, "signs"), _dev(y, table.dtype, "out"), M, V, H,
                            dt, _stream(stream)), "ptq_embed")
    return y


def embed_ptq1(wq, scales, ids, signs, out_dtype=None, out=None, stream=None):
    """ptq_embed_ptq1: the same lookup on a PTQ1_0 table (wq V x H/128*26
    uint8, scales V x H/128 int16 bit patterns); out_dtype float32 (default)
    or bfloat16."""
    import torch

    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    dt = PTQ_F32 if out_dtype == torch.float32 else PTQ_BF16 if out_dtype == torch.bfloat16 else None
    if dt is None:
        raise TypeError(f"out_dtype must be float32 or bfloat16, got {out_dtype}")
    V, H = scales.shape[0], scales.shape[1] * 128
    M = ids.numel()
    y = torch.empty((M, H), dtype=out_dtype, device=wq.device) if out is None else out
    _check(load().ptq_embed_ptq1(_dev(wq, torch.uint8, "wq"), _dev(scales, None, "scales"),
                                 _dev(ids, torch.int32, "ids"), _dev(signs, torch.int8, "signs"),
                                 _dev(y, out_dtype, "out"), M, V, H, dt, _stream(stream)),
           "ptq_embed_ptq1")
    return y


def route(M: int, dtype: int) -> str:
    name = ctypes.c_char_p()
    _check(load().ptq_route(M, dtype, ctypes.byref(name)), "ptq_route")
    return name.value.decode()


def matmul_f32_peel(wq, scales, x, out=None, stream=None):
    """Test export: the fp32 route's SIMT peel GEMV (ptq_matmul_f32_peel),
    y = x W^T with x float32 (already rotated), on any shape."""
    import torch

    M, K = x.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else out
    _check(load().ptq_matmul_f32_peel(
        _dev(wq, torch.uint8, "wq"), _dev(scales, torch.int16, "scales"),
        _dev(x, torch.float32, "x"), _dev(y, torch.float32, "out"), M, N, K, _stream(stream)),
        "ptq_matmul_f32_peel")
    return y


def gemv_plan(M: int, N: int, K: int, pq2: bool = False) -> dict:
    """The launch of the fp32 decode GEMV for (M, N, K) on the current device
    (ptq_gemv_plan): CTAs, cluster size (0: none), K-chunks, kernels."""
    out = (ctypes.c_int32 * 4)()
    _check(load().ptq_gemv_plan(M, N, K, int(pq2), out), "ptq_gemv_plan")
    return {"ctas": out[0], "cluster": out[1], "chunks": out[2], "kernels": out[3]}


def selftest_timeout(stream=None) -> None:
    """Runs the bounded wait that is made to run out (ptq_selftest_timeout);
    the next device_check raises PTQ_ERR_TIMEOUT."""
    _check(load().ptq_selftest_timeout(_stream(stream)), "ptq_selftest_timeout")


def selftest_grid_timeout(stream=None) -> None:
    """Runs the persistent stack's grid barrier with one CTA that never
    arrives (ptq_selftest_grid_timeout); the next device_check raises
    PTQ_ERR_TIMEOUT."""
    _check(load().ptq_selftest_grid_timeout(_stream(stream)), "ptq_selftest_grid_timeout")


def device_check(stream=None) -> None:
    _check(load().ptq_device_check(_stream(stream)), "ptq_device_check")
