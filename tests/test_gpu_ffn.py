"""GPU parity of ptq_ffn (rotate, gate+up, SwiGLU, rotate, down) against the
oracle's fp64 feed-forward block, on the 64-layer workload's shapes."""
import numpy as np
import pytest

import parity as Q

pytestmark = pytest.mark.gpu

H, I = 5120, 17408


@pytest.fixture(scope="module")
def P():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import ternary_weight_ptq1_gb300 as P

    P.load()
    return P


def device_layer(P, L):
    return (Q.dev(P.pack(L.wgu_trits)), Q.dev(L.wgu_scales), Q.dev(P.pack(L.wd_trits)),
            Q.dev(L.wd_scales), Q.dev(L.signs_in), Q.dev(L.signs_mid))


def oracle_ffn(orc, P, L, x64):
    return orc.ffn(orc.pack(L.wgu_trits), L.wgu_scales, orc.pack(L.wd_trits), L.wd_scales,
                   L.signs_in, L.signs_mid, x64)


@pytest.mark.parametrize("layer", [0, 63])
def test_ffn_decode_layer(P, orc, syn, layer):
    L = syn.ffn_layer(4, layer, H, I)
    x = syn.ffn_input(4, layer, 1, H, "f32")
    y = P.ffn(*device_layer(P, L), Q.dev(x))
    Q.check_f32(Q.host_f64(y), oracle_ffn(orc, P, L, Q.x_f64(x)), f"ffn M=1 layer {layer}")


def test_ffn_prefill_sampled_tokens(P, orc, syn):
    L = syn.ffn_layer(4, 1, H, I)
    x = syn.ffn_input(4, 1, 256, H, "bf16")
    y = Q.host_f64(P.ffn(*device_layer(P, L), Q.dev_bf16(x)))
    tokens = [0, 1, 77, 128, 200, 255]
    ref = oracle_ffn(orc, P, L, Q.x_f64(x)[tokens])
    Q.check_bf16(y[tokens], ref, "ffn M=256 sampled tokens")


@pytest.mark.parametrize("M,dtype", [(1, "f32"), (3, "f32"), (8, "f32"), (5, "bf16"), (70, "bf16")])
def test_ffn_small(P, orc, syn, M, dtype):
    L = syn.ffn_layer(9, M, 1024, 2048)
    x = syn.ffn_input(9, M, M, 1024, dtype)
    xd = Q.dev(x) if dtype == "f32" else Q.dev_bf16(x)
    y = Q.host_f64(P.ffn(*device_layer(P, L), xd))
    ref = oracle_ffn(orc, P, L, Q.x_f64(x))
    (Q.check_f32 if dtype == "f32" else Q.check_bf16)(y, ref, f"ffn small {M} {dtype}")


@pytest.mark.parametrize("M", [70, 300])
def test_ffn_prefill_swiglu_in_the_gemm_epilogue(P, orc, syn, M):
    # I = 9216 gives 144 gate/up tiles: the GEMM runs unsplit, with SwiGLU in
    # its epilogue (a tile pairs 64 gate rows with the matching 64 up rows);
    # M = 70 leaves most of a row tile empty, M = 300 spans two
    L = syn.ffn_layer(10, M, 1024, 9216)
    x = syn.ffn_input(10, M, M, 1024, "bf16")
    y = Q.host_f64(P.ffn(*device_layer(P, L), Q.dev_bf16(x)))
    tokens = [0, 1, M // 2, M - 2, M - 1] + ([255, 256] if M > 256 else [])
    ref = oracle_ffn(orc, P, L, Q.x_f64(x)[tokens])
    Q.check_bf16(y[tokens], ref, f"ffn fused SwiGLU M={M}")


def test_ffn_leaves_x_alone_and_rejects_small_workspace(P, syn):
    import torch

    L = syn.ffn_layer(9, 0, 1024, 2048)
    x = Q.dev(syn.ffn_input(9, 0, 2, 1024, "f32"))
    x0 = x.clone()
    need = P.ffn_workspace_bytes(2, 1024, 2048, P.PTQ_F32)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    P.ffn(*device_layer(P, L), x, workspace=ws)
    assert torch.equal(x, x0)
    with pytest.raises(P.PTQError, match="WORKSPACE"):
        P.ffn(*device_layer(P, L), x, workspace=ws[: need - 256])
