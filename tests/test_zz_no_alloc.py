"""ptq_ffn_noalloc: the feed-forward block for callers that cannot allocate
device memory (real-time decode loops that may not pay for cudaMalloc,
plug-ins handed a stream but no allocator, hosts whose memory another
allocator owns).  Its scratch is a built-in device array, so its results must
match ptq_ffn (which takes a caller-allocated workspace) within the parity
tolerance, call after call -- the array keeps the previous call's contents --
and both must match the oracle's block.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import parity as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import ternary_weight_ptq1_gb300 as P

    P.load()
    return P


def _layer(P, syn, seed, H, I):
    L = syn.ffn_layer(seed, 0, H, I)
    return [Q.dev(P.pack(L.wgu_trits)), Q.dev(L.wgu_scales), Q.dev(P.pack(L.wd_trits)),
            Q.dev(L.wd_scales), Q.dev(L.signs_in), Q.dev(L.signs_mid)]


@pytest.mark.parametrize("M,dtype,H,I", [(1, "f32", 5120, 17408), (2, "f32", 5120, 17408),
                                         (8, "f32", 1024, 2048), (16, "bf16", 5120, 17408)])
def test_noalloc_matches_ffn_twice(P, orc, syn, M, dtype, H, I):
    import torch

    check = Q.check_f32 if dtype == "f32" else Q.check_bf16
    # the oracle checks every token of small calls and two tokens of large ones
    tokens = np.arange(M) if M * H * I <= 8 * 1024 * 2048 or M == 1 else np.array([0, M - 1])
    for call, seed in enumerate((41, 42)):   # two calls in a row, different data
        L = syn.ffn_layer(seed, 0, H, I)
        w = _layer(P, syn, seed, H, I)
        x = syn.ffn_input(seed, 0, M, H, dtype)
        xd = Q.dev(x) if dtype == "f32" else Q.dev_bf16(x)
        y_ref = P.ffn(*w, xd)
        y = P.ffn_noalloc(*w, xd)
        torch.cuda.synchronize()
        yh = Q.host_f64(y)
        check(yh, Q.host_f64(y_ref), f"noalloc call {call} M={M} {dtype} against ptq_ffn")
        ref = orc.ffn(orc.pack(L.wgu_trits), L.wgu_scales, orc.pack(L.wd_trits), L.wd_scales,
                      L.signs_in, L.signs_mid, Q.x_f64(x)[tokens])
        check(yh[tokens], ref, f"noalloc call {call} M={M} {dtype} against the oracle")


def test_noalloc_refuses_shapes_beyond_its_array(P, syn):
    w = _layer(P, syn, 43, 5120, 17408)
    x = Q.dev(syn.ffn_input(43, 0, 256, 5120, "bf16")).view(__import__("torch").bfloat16)
    need = P.ffn_workspace_bytes(256, 5120, 17408, P.PTQ_BF16)
    assert need > P.FFN_NOALLOC_SCRATCH_BYTES
    with pytest.raises(P.PTQError, match="WORKSPACE"):
        P.ffn_noalloc(*w, x)
