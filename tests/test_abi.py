"""The C ABI on the host: the library loads and exports everything the
header declares, the host encoder matches the oracle's encoder byte for byte,
arguments are refused by name before anything is launched, and the routing
table is consistent.  No call here touches a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def P():
    import ternary_weight_ptq1_gb300 as P

    P._build.build()
    P.load()
    return P


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ptq.h")).read()
    return sorted(set(re.findall(r"PTQ_API(?:\s+PTQ_NODISCARD)?\s+[\w\s\*]+?\b(ptq\w+)\s*\(", text)))


def test_header_declares_the_exports(P):
    syms = declared_symbols()
    assert set(syms) == set(P.EXPORTS), syms
    lib = ctypes.CDLL(P.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s


def test_no_oracle_in_the_product():
    pkg = os.path.join(ROOT, "ternary_weight_ptq1_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("the oracle", ""), f
                assert "import synth" not in text, f


def test_pack_matches_oracle_pack(P, orc, syn):
    for seed, N, K, p0 in ((0, 7, 1024, None), (1, 64, 5120, None), (2, 16, 17408, 0.4), (3, 3, 128, None)):
        t, _ = syn.weights(seed, N, K, p0)
        np.testing.assert_array_equal(P.pack(t), orc.pack(t))
    every = np.array(np.meshgrid(*[[-1, 0, 1]] * 5)).reshape(5, -1).T  # 243 tuples
    t = np.zeros((243, 128), np.int8)
    t[:, :5] = every
    t[:, 125:128] = every[:, :3]
    np.testing.assert_array_equal(P.pack(t), orc.pack(t))


def test_pack_refusals(P):
    with pytest.raises(P.PTQError, match="PTQ_ERR_VALUE"):
        t = np.zeros((2, 128), np.int8)
        t[1, 3] = -2
        P.pack(t)
    with pytest.raises(P.PTQError, match="PTQ_ERR_SHAPE"):
        P.pack(np.zeros((2, 100), np.int8))
    L = P.load()
    assert L.ptq1_pack(None, None, 4, 128) == 1  # PTQ_ERR_NULL
    assert L.ptq1_pack(None, None, 0, 128) == 0  # empty is a no-op
    assert L.ptq1_pack(None, None, 2 ** 62, 2 ** 10) == 2  # N*K overflows


def test_refusals_before_launch(P):
    L = P.load()
    p16 = ctypes.c_void_p(16 * 1024)   # never dereferenced: every call below is refused
    odd = ctypes.c_void_p(16 * 1024 + 4)
    # matmul
    mm = lambda *a: L.ptq_matmul(*a[:8], None, 0, None)  # no workspace
    assert mm(p16, p16, p16, p16, 1, 8, 100, P.PTQ_F32) == 2
    assert mm(p16, p16, p16, p16, -1, 8, 128, P.PTQ_F32) == 2
    assert mm(p16, p16, p16, p16, 9, 8, 128, P.PTQ_F32) == 5
    assert b"M=9" in L.ptq_last_error()
    assert mm(p16, p16, p16, p16, 1, 8, 128, 7) == 4
    assert mm(None, p16, p16, p16, 1, 8, 128, P.PTQ_F32) == 1
    assert mm(p16, odd, p16, p16, 1, 8, 128, P.PTQ_F32) == 3
    assert mm(None, None, None, None, 0, 8, 128, P.PTQ_F32) == 0
    assert mm(None, None, None, None, 4, 0, 128, P.PTQ_BF16) == 0
    assert mm(p16, p16, p16, p16, 2 ** 40, 2 ** 40, 128, P.PTQ_BF16) == 2
    # the M = 1 decode needs its scratch: refused by size before any launch
    need = P.matmul_workspace_bytes(1, 17408, 5120, P.PTQ_F32)
    assert need == 9 * 17408 * 4
    args = (p16, p16, p16, p16, 1, 17408, 5120, P.PTQ_F32)
    assert L.ptq_matmul(*args, None, need, None) == 6
    assert L.ptq_matmul(*args, p16, need - 1, None) == 6
    assert L.ptq_matmul(*args, odd, need, None) == 3
    # one scratch row sum per (token, chunk, row): M = 4 needs four times as much
    need4 = P.matmul_workspace_bytes(4, 17408, 5120, P.PTQ_F32)
    assert need4 == 4 * need
    args4 = (p16, p16, p16, p16, 4, 17408, 5120, P.PTQ_F32)
    assert L.ptq_matmul(*args4, p16, need, None) == 6
    assert L.ptq_matmul(*args4, p16, need4 - 1, None) == 6
    assert P.rotate_matmul_workspace_bytes(4, 17408, 5120, P.PTQ_F32) >= need4
    assert P.matmul_workspace_bytes(9, 17408, 5120, P.PTQ_F32) == 0
    assert P.matmul_workspace_bytes(512, 17408, 5120, P.PTQ_BF16) == 0
    assert P.matmul_workspace_bytes(1, 17408, 5120 + 128, P.PTQ_F32) == 0  # K/128 odd
    assert P.matmul_workspace_bytes(1, 17408, 100, P.PTQ_F32) == 0
    # prefill split-K scratch, a function of the shape alone: fewer output
    # tiles than half of 152 SMs split K over up to 6 CTAs (at most one per
    # 1024-wide group), one fp32 M x N partial sum each
    assert P.matmul_workspace_bytes(256, 5120, 17408, P.PTQ_BF16) == 6 * 256 * 5120 * 4
    assert P.matmul_workspace_bytes(64, 1000, 6144, P.PTQ_BF16) == 6 * 64 * 1000 * 4
    assert P.matmul_workspace_bytes(300, 640, 3072, P.PTQ_BF16) == 3 * 300 * 640 * 4
    assert P.matmul_workspace_bytes(128, 17408, 5120, P.PTQ_BF16) == 0  # 136 tiles
    # rotation
    assert L.ptq_fwht(p16, p16, p16, 1, 1000, P.PTQ_F32, None) == 2
    assert L.ptq_fwht(p16, odd, p16, 1, 1024, P.PTQ_F32, None) == 3
    assert L.ptq_fwht(p16, p16, None, 1, 1024, P.PTQ_F32, None) == 1
    assert L.ptq_fwht(None, None, None, 0, 1024, P.PTQ_BF16, None) == 0
    # embedding lookup: shape, NULL, alignment, dtype; M = 0 is a no-op
    em = L.ptq_embed
    assert em(p16, p16, p16, p16, 1, 10, 1000, P.PTQ_F32, None) == 2     # H % 1024
    assert em(p16, p16, p16, p16, 1, 0, 1024, P.PTQ_F32, None) == 2      # V < 1
    assert em(p16, p16, p16, p16, -1, 10, 1024, P.PTQ_F32, None) == 2
    assert em(p16, None, p16, p16, 1, 10, 1024, P.PTQ_F32, None) == 1
    odd2 = ctypes.c_void_p(16 * 1024 + 2)
    assert em(p16, odd2, p16, p16, 1, 10, 1024, P.PTQ_F32, None) == 3    # ids 4-aligned
    assert em(odd, p16, p16, p16, 1, 10, 1024, P.PTQ_BF16, None) == 3
    assert em(p16, p16, p16, p16, 1, 10, 1024, 5, None) == 4
    assert em(None, None, None, None, 0, 10, 1024, P.PTQ_F32, None) == 0
    ep = L.ptq_embed_ptq1
    assert ep(p16, None, p16, p16, p16, 1, 10, 1024, P.PTQ_F32, None) == 1  # scales
    assert ep(p16, odd, p16, p16, p16, 1, 10, 1024, P.PTQ_F32, None) == 3
    assert ep(p16, p16, p16, p16, p16, 1, 10, 2048 + 128, P.PTQ_F32, None) == 2
    assert ep(p16, p16, p16, p16, p16, 1, 2 ** 62, 1024, P.PTQ_F32, None) == 2  # V H overflows
    # feed-forward block
    need = P.ffn_workspace_bytes(1, 1024, 2048, P.PTQ_F32)
    assert need > 0
    args = [p16] * 8 + [1, 1024, 2048, P.PTQ_F32]
    assert L.ptq_ffn(*args, None, need, None) == 6
    assert L.ptq_ffn(*args, p16, need - 1, None) == 6
    assert L.ptq_ffn(*([p16] * 8 + [1, 1000, 2048, P.PTQ_F32]), p16, need, None) == 2
    assert L.ptq_ffn(*([p16] * 8 + [9, 1024, 2048, P.PTQ_F32]), p16, 10 ** 9, None) == 5
    assert P.ffn_workspace_bytes(1, 1000, 2048, P.PTQ_F32) == 0



def test_stack_refusals_before_launch(P):
    L = P.load()
    p16 = ctypes.c_void_p(16 * 1024)   # never dereferenced: every call below is refused
    odd = ctypes.c_void_p(16 * 1024 + 4)
    H, I = 1024, 2048
    need = P.ffn_stack_workspace_bytes(1, H, I, P.PTQ_F32)
    # xn and y regions (256-byte rounded) ahead of the block's own scratch,
    # and for fp32 at M <= 8 a second gate/up buffer of the persistent path
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    assert need == 2 * H * 4 + up(P.ffn_workspace_bytes(1, H, I, P.PTQ_F32)) + 2 * I * 4
    assert P.ffn_stack_workspace_bytes(3, H, I, P.PTQ_BF16) == (
        2 * up(3 * H * 2) + up(P.ffn_workspace_bytes(3, H, I, P.PTQ_BF16)))
    assert P.ffn_stack_workspace_bytes(1, 1000, I, P.PTQ_F32) == 0
    assert P.ffn_stack_workspace_bytes(1, H, I, 9) == 0
    good = P.FfnLayer(*([16 * 1024] * 7))
    bad_w = P.FfnLayer(*([16 * 1024] * 6 + [16 * 1024 + 4]))      # misaligned gains
    no_w = P.FfnLayer(*([16 * 1024] * 6 + [None]))
    no_q = P.FfnLayer(*([None] + [16 * 1024] * 6))

    def st(layers, nL, x=p16, M=1, h=H, eps=1e-6, dt=P.PTQ_F32, ws=p16, wsb=need):
        arr = (P.FfnLayer * max(len(layers), 1))(*layers)
        return L.ptq_ffn_stack(ctypes.cast(arr, ctypes.c_void_p), nL, x, M, h, I, eps, dt, ws, wsb,
                               None)

    assert st([good], 1, dt=7) == 4
    assert st([good], -1) == 2
    assert st([good], 1, h=1000) == 2
    assert st([good], 1, eps=-1.0) == 4
    assert st([good], 1, eps=float("nan")) == 4
    assert st([good], 1, eps=float("inf")) == 4
    assert st([good], 1, x=None) == 1
    assert st([good], 1, x=odd) == 3
    assert st([good], 1, ws=None) == 6
    assert st([good], 1, wsb=need - 1) == 6
    assert st([good], 1, ws=odd) == 3
    assert st([good], 1, M=9, wsb=10 ** 9) == 5         # fp32 serves M <= 8
    arr1 = (P.FfnLayer * 1)(good)
    assert L.ptq_ffn_stack_ex(ctypes.cast(arr1, ctypes.c_void_p), 1, p16, 1, H, I, 1e-6,
                              P.PTQ_F32, p16, need, 2, None) == 4  # unknown flag
    assert L.ptq_ffn_stack(None, 1, p16, 1, H, I, 1e-6, P.PTQ_F32, p16, need, None) == 1
    # every layer is checked before the first launch; the message names it
    assert st([good, no_q], 2) == 1
    assert b"layer 1" in L.ptq_last_error()
    assert st([good, good, no_w], 3) == 1
    assert b"layer 2" in L.ptq_last_error()
    assert st([bad_w], 1) == 3
    # the route query refuses before it looks at the device
    name = ctypes.c_char_p()
    assert L.ptq_ffn_stack_route(1, H, I, P.PTQ_F32, None) == 1
    assert L.ptq_ffn_stack_route(1, H, I, 7, ctypes.byref(name)) == 4
    assert L.ptq_ffn_stack_route(1, 1000, I, P.PTQ_F32, ctypes.byref(name)) == 2
    assert L.ptq_ffn_stack_route(0, H, I, P.PTQ_F32, ctypes.byref(name)) == 2
    assert L.ptq_ffn_stack_route(9, H, I, P.PTQ_F32, ctypes.byref(name)) == 5
    # no layers or no rows: nothing to do
    assert st([], 0, x=None, ws=None, wsb=0) == 0
    assert st([good], 1, M=0, x=None, ws=None, wsb=0) == 0

def test_rotate_matmul_host_refusals(P):
    # host-buffer entry: the workspace holds x and y (256-byte rounded) before
    # ptq_rotate_matmul's own; refusals come before any copy or launch
    L = P.load()
    p16 = ctypes.c_void_p(16 * 1024)
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    inner = P.rotate_matmul_workspace_bytes(1, 17408, 5120, P.PTQ_F32)
    need = P.rotate_matmul_host_workspace_bytes(1, 17408, 5120, P.PTQ_F32)
    assert need == up(5120 * 4) + up(17408 * 4) + inner
    assert P.rotate_matmul_host_workspace_bytes(2, 300, 2048, P.PTQ_BF16) == (
        up(2 * 2048 * 2) + up(2 * 300 * 2) + P.rotate_matmul_workspace_bytes(2, 300, 2048,
                                                                             P.PTQ_BF16))
    assert P.rotate_matmul_host_workspace_bytes(1, 100, 1000, P.PTQ_F32) == 0
    host = lambda x, y, ws, nb: L.ptq_rotate_matmul_host(  # noqa: E731
        p16, p16, x, p16, y, 1, 17408, 5120, P.PTQ_F32, ws, nb, None)
    assert host(None, p16, p16, need) == 1                 # NULL host x
    assert host(p16, None, p16, need) == 1                 # NULL host y
    assert host(p16, p16, None, need) == 6                 # no workspace
    assert host(p16, p16, p16, need - 1) == 6
    assert host(p16, p16, ctypes.c_void_p(16 * 1024 + 16), need) == 3  # not 256-aligned
    assert L.ptq_rotate_matmul_host(p16, p16, p16, p16, p16, 1, 8, 1000, P.PTQ_F32, p16, need,
                                    None) == 2             # K % 1024
    assert L.ptq_rotate_matmul_host(p16, p16, p16, p16, p16, 0, 8, 1024, P.PTQ_F32, None, 0,
                                    None) == 0             # nothing to do


def test_routing_table(P):
    for M in range(1, 9):
        assert P.route(M, P.PTQ_F32) == "gemv_ptq1_f32_lut"
    for M in (1, 8, 64, 128, 512, 2048, 10 ** 6):
        assert P.route(M, P.PTQ_BF16).startswith("gemm_ptq1_bf16")
    with pytest.raises(P.PTQError, match="UNSUPPORTED"):
        P.route(9, P.PTQ_F32)
    with pytest.raises(P.PTQError, match="UNSUPPORTED"):
        P.route(0, P.PTQ_F32)


def test_status_strings(P):
    L = P.load()
    for code, name in P.STATUS.items():
        assert L.ptq_status_str(code).decode() == name


def test_workspace_sizes(P):
    M, H, I = 256, 5120, 17408
    bf = P.ffn_workspace_bytes(M, H, I, P.PTQ_BF16)
    f = P.ffn_workspace_bytes(1, H, I, P.PTQ_F32)
    assert bf >= M * H * 2 + M * 2 * I * 4 + M * I * 4 + M * I * 2
    # decode adds the row sums of the larger projection: 9 chunks of the
    # gate/up rows (K = 5120) against 28 chunks of the down rows (K = 17408)
    gu_part = 9 * 2 * I * 4
    assert gu_part > 28 * H * 4
    assert f >= H * 4 + 2 * I * 4 + I * 4 + gu_part
    assert f <= P.FFN_NOALLOC_SCRATCH_BYTES
    # the allocation-free entry point's stated limits at these shapes: fp32
    # decode up to 2 tokens, bf16 up to 16
    assert P.ffn_workspace_bytes(2, H, I, P.PTQ_F32) <= P.FFN_NOALLOC_SCRATCH_BYTES
    assert P.ffn_workspace_bytes(3, H, I, P.PTQ_F32) > P.FFN_NOALLOC_SCRATCH_BYTES
    assert P.ffn_workspace_bytes(16, H, I, P.PTQ_BF16) <= P.FFN_NOALLOC_SCRATCH_BYTES
    assert P.ffn_workspace_bytes(17, H, I, P.PTQ_BF16) > P.FFN_NOALLOC_SCRATCH_BYTES
    # chunk count: 13 K/256 words per row, at most 32 per chunk
    for K in (256, 512, 1024, 2048, 5120, 17408):
        words = 13 * K // 256
        assert P.matmul_workspace_bytes(1, 100, K, P.PTQ_F32) == (
            0 if words <= 32 else ((words + 31) // 32 * 100 * 4 + 255) // 256 * 256)


def test_pq2_host_side(P, orc, syn):
    # the library's PQ2_0 encoder writes the oracle's bytes; refusals before
    # any launch
    L = P.load()
    t, _ = syn.weights(40, 7, 1024)
    np.testing.assert_array_equal(P.pq2_pack(t), orc.pq2_pack(t))
    with pytest.raises(P.PTQError, match="VALUE"):
        P.pq2_pack(np.full((1, 128), 2, np.int8))
    with pytest.raises(P.PTQError, match="SHAPE"):
        P.pq2_pack(np.zeros((1, 100), np.int8))
    p16 = ctypes.c_void_p(16 * 1024)
    mm = lambda *a: L.ptq_matmul_pq2(*a[:8], None, 0, None)  # noqa: E731
    assert mm(p16, p16, p16, p16, 1, 8, 1152, P.PTQ_F32) == 5     # K % 1024
    assert mm(p16, p16, p16, p16, 9, 8, 1024, P.PTQ_F32) == 5     # fp32 serves M <= 8
    assert mm(p16, p16, p16, p16, 1, 8, 100, P.PTQ_F32) == 2
    assert mm(None, p16, p16, p16, 1, 8, 1024, P.PTQ_BF16) == 1
    need = P.matmul_pq2_workspace_bytes(1, 17408, 5120, P.PTQ_F32)
    assert need == 10 * 17408 * 4                                  # 320 words a row: 10 chunks
    assert P.matmul_pq2_workspace_bytes(8, 17408, 5120, P.PTQ_F32) == 8 * need  # per token
    assert mm(p16, p16, p16, p16, 1, 17408, 5120, P.PTQ_F32) == 6  # no workspace
    assert P.matmul_pq2_workspace_bytes(1, 100, 1152, P.PTQ_F32) == 0

