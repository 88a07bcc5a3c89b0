"""The timeout path on a GPU, without a fault: a bounded mbarrier wait that
nothing completes runs out, raises the device status word, and
ptq_device_check reports PTQ_ERR_TIMEOUT once; the context stays usable."""
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


@pytest.fixture(scope="module")
def P():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import ternary_weight_ptq1_gb300 as P

    P.load()
    return P
