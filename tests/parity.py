"""Shared helpers of the parity tests: tolerances, device transfer, and the
oracle's view of each workload.  The tolerances are the stated ones:

* fp32 activation paths: |y - y_ref| <= 1e-4 * (|y_ref| + rms(y_ref))
* bf16 activation paths: |y - y_ref| <= 1e-2 * rms(y_ref) + 2^-8 |y_ref|
  (the second term is the storage rounding of a bf16 output: half a unit in
  the last place is at most 2^-8 |y_ref|)
* the rotation: |y - y_ref| <= 1e-5 * (|y_ref| + rms(y_ref)), plus the same
  2^-8 |y_ref| rounding allowance when the output is bf16

rms is taken over the whole output of the call (per layer for ptq_ffn).
"""
import numpy as np
import scipy.special

import oracle
import synth


def rms(a):
    a = np.asarray(a, np.float64)
    return float(np.sqrt(np.mean(a * a)))


def check(y, ref, rel, abs_rms, bf16_round=False, what=""):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    r = rms(ref)
    bound = rel * np.abs(ref) + abs_rms * r
    if bf16_round:
        bound = bound + 2.0 ** -8 * np.abs(ref)
    err = np.abs(y - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
                             f"y={y[i]!r} ref={ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e} rms={r:.3e}")
    return float((err / (np.abs(ref) + r)).max()) if r > 0 else 0.0


def check_f32(y, ref, what=""):
    return check(y, ref, 1e-4, 1e-4, False, what)


def check_bf16(y, ref, what=""):
    return check(y, ref, 0.0, 1e-2, True, what)


def check_fwht(y, ref, bf16_out=False, what=""):
    return check(y, ref, 1e-5, 1e-5, bf16_out, what)


# ---- host <-> device ------------------------------------------------------------

def dev(a):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def dev_bf16(bits):
    import torch

    return dev(bits).view(torch.bfloat16)


def host_f64(t):
    """Device tensor (float32 or bfloat16) -> float64 numpy, decoded exactly."""
    import torch

    if t.dtype == torch.bfloat16:
        return oracle.decode_bf16(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return oracle.decode_f32(t.cpu().numpy())


# ---- oracle views of the workloads ------------------------------------------------

def x_f64(x):
    return oracle.decode_f32(x) if x.dtype == np.float32 else oracle.decode_bf16(x)


def swiglu_like(seed, M, K):
    """Decode-down activations: silu(a) * b with a, b ~ N(0,1), stored fp32."""
    a, b = synth.gated_pair(seed, M, K)
    return (a * scipy.special.expit(a) * b).astype(np.float32)
