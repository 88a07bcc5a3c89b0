"""The timeout path on a GPU, without a fault: a bounded mbarrier wait that
nothing completes, and a grid barrier one CTA never reaches, run out, raise
the device status word, and ptq_device_check reports PTQ_ERR_TIMEOUT once;
the context stays usable."""
import time

import numpy as np
import pytest

import parity as Q

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_cleared(P, orc, syn):
    import torch

    P.device_check()  # nothing pending
    t0 = time.time()
    P.selftest_timeout()
    with pytest.raises(P.PTQError, match="TIMEOUT"):
        P.device_check()
    assert time.time() - t0 < 30.0  # a bounded wait, not a hang
    P.device_check()  # cleared by the first check
    # the context still computes
    mv = syn.gaussian_matvec(50, 1, 700, 2048)
    y = P.matmul(Q.dev(P.pack(mv.trits)), Q.dev(mv.scales), Q.dev(mv.x))
    torch.cuda.synchronize()
    Q.check_f32(Q.host_f64(y), orc.matmul(orc.pack(mv.trits), mv.scales, Q.x_f64(mv.x)), "after")
    P.device_check()


def test_grid_barrier_that_runs_out_is_reported(P, orc, syn):
    # the persistent stack's grid barrier with one CTA that never arrives:
    # the others give up, raise the status word and return
    import torch

    P.device_check()
    t0 = time.time()
    P.selftest_grid_timeout()
    with pytest.raises(P.PTQError, match="TIMEOUT"):
        P.device_check()
    assert time.time() - t0 < 30.0
    P.device_check()
    # the persistent stack still runs and agrees with the oracle
    H, I = 1024, 2048
    F = syn.ffn_layer(80, 0, H, I)
    lay = (Q.dev(P.pack(F.wgu_trits)), Q.dev(F.wgu_scales), Q.dev(P.pack(F.wd_trits)),
           Q.dev(F.wd_scales), Q.dev(F.signs_in), Q.dev(F.signs_mid))
    g = syn.norm_gain(80, 0, H)
    x = syn.ffn_input(80, 0, 1, H, "f32")
    xd = Q.dev(x.copy())
    assert P.ffn_stack_route(1, H, I, P.PTQ_F32) == "stack_decode_persistent"
    P.ffn_stack([lay], [Q.dev(g)], xd, 1e-6)
    torch.cuda.synchronize()
    P.device_check()
    x64 = x.astype(np.float64)
    ref = orc.ffn_stack([(orc.pack(F.wgu_trits), F.wgu_scales, orc.pack(F.wd_trits), F.wd_scales,
                          F.signs_in, F.signs_mid)], [g.astype(np.float64)], x64, 1e-6)
    Q.check_f32(Q.host_f64(xd) - x64, ref - x64, "stack after the grid timeout")


@pytest.fixture(scope="module")
def P():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import ternary_weight_ptq1_gb300 as P

    P.load()
    return P


def test_fp16_operand_range_is_reported(P, orc, syn):
    # The bf16 route keeps the rotated activation in fp16.  A row of bf16
    # values of 4096 rotates to 4096 * 1024 / 32 = 131072 in one element of
    # each 1024-block (all signs +1): beyond fp16's 65504, so it is stored as
    # infinity, the output is not finite, and ptq_device_check reports
    # PTQ_ERR_RANGE once.  A row of 64s (2048 after the rotation) is in range.
    import torch

    P.device_check()
    M, N, K = 64, 256, 2048
    mv = syn.gaussian_matvec(81, M, N, K)
    wq, sc = Q.dev(P.pack(mv.trits)), Q.dev(mv.scales)
    plus = Q.dev(np.ones(K, np.int8))
    x = torch.full((M, K), 64.0, dtype=torch.bfloat16, device="cuda")
    y = P.rotate_matmul(wq, sc, x, plus)
    torch.cuda.synchronize()
    P.device_check()  # in range: nothing raised
    assert torch.isfinite(y.float()).all()
    x[5] = 4096.0
    y = P.rotate_matmul(wq, sc, x, plus)
    torch.cuda.synchronize()
    with pytest.raises(P.PTQError, match="RANGE"):
        P.device_check()
    P.device_check()  # cleared by the first check
    assert not torch.isfinite(y[5].float()).all()
    assert torch.isfinite(y[4].float()).all()
    # the feed-forward block's first rotation takes the same check
    H, I = 1024, 2048
    F = syn.ffn_layer(82, 0, H, I)
    lay = (Q.dev(P.pack(F.wgu_trits)), Q.dev(F.wgu_scales), Q.dev(P.pack(F.wd_trits)),
           Q.dev(F.wd_scales), Q.dev(np.ones(H, np.int8)), Q.dev(F.signs_mid))
    xb = torch.full((3, H), 4096.0, dtype=torch.bfloat16, device="cuda")
    P.ffn(*lay, xb)
    torch.cuda.synchronize()
    with pytest.raises(P.PTQError, match="RANGE"):
        P.device_check()
    # the context still computes and agrees with the oracle
    xs = syn.ffn_input(82, 0, 2, H, "bf16")
    yb = Q.host_f64(P.ffn(*lay[:4], Q.dev(F.signs_in), lay[5], Q.dev_bf16(xs)))
    torch.cuda.synchronize()
    P.device_check()
    ref = orc.ffn(orc.pack(F.wgu_trits), F.wgu_scales, orc.pack(F.wd_trits), F.wd_scales,
                  F.signs_in, F.signs_mid, Q.x_f64(xs))
    Q.check_bf16(yb, ref, "ffn after the range report")
