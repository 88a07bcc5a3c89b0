"""GPU parity of the codec (bit-exact) and of the signed rotation against the
oracle, through the C ABI."""
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


def test_unpack_every_byte_value(P, orc):
    # all 256 byte values, including the 13 no encoder produces, in every
    # position of a block (the decode is total)
    rng = np.random.default_rng(0)
    wq = rng.integers(0, 256, size=(300, 26 * 8), dtype=np.uint8)
    wq[0, :256 % 208] = np.arange(256 % 208, dtype=np.uint8)
    wq[1, :] = np.arange(48, 256, dtype=np.uint8)
    out = P.unpack(Q.dev(wq), 1024).cpu().numpy()
    np.testing.assert_array_equal(out, orc.unpack(wq, 1024))


@pytest.mark.parametrize("seed,N,K,p0", [(0, 1024, 1024, None), (1, 17408, 5120, None),
                                         (2, 5120, 17408, 0.4), (5, 3, 384, None)])
def test_pack_then_device_unpack_roundtrip(P, orc, syn, seed, N, K, p0):
    t, _ = syn.weights(seed, N, K, p0)
    wq = P.pack(t)
    np.testing.assert_array_equal(wq, orc.pack(t))
    np.testing.assert_array_equal(P.unpack(Q.dev(wq), K).cpu().numpy(), t)


@pytest.mark.parametrize("M,K", [(1, 1024), (1, 5120), (4, 5120), (8, 17408), (3, 2048), (37, 3072)])
def test_fwht_f32(P, orc, syn, M, K):
    x = syn.normal_f32(10 + M, 2, (M, K))
    s = syn.signs(10 + M, 3, K)
    y = P.fwht(Q.dev(x), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.fwht(orc.decode_f32(x), s), what=f"fwht f32 {M}x{K}")


@pytest.mark.parametrize("M,K", [(128, 5120), (2, 1024), (33, 2048)])
def test_fwht_bf16(P, orc, syn, M, K):
    x = syn.normal_bf16(20 + M, 2, (M, K))
    s = syn.signs(20 + M, 3, K)
    y = P.fwht(Q.dev_bf16(x), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.fwht(orc.decode_bf16(x), s), bf16_out=True,
                 what=f"fwht bf16 {M}x{K}")


def test_fwht_in_place_and_unit_vector(P, orc, syn):
    import torch

    s = syn.signs(3, 3, 2048)
    x = np.zeros((2, 2048), np.float32)
    x[0, 0] = 1.0
    x[1, 1024 + 5] = -2.0
    d = Q.dev(x)
    P.fwht(d, Q.dev(s), out=d)
    y = d.cpu().numpy()
    np.testing.assert_array_equal(y[0, :1024], np.full(1024, s[0] / 32.0, np.float32))
    np.testing.assert_array_equal(y[0, 1024:], 0)
    Q.check_fwht(y.astype(np.float64), orc.fwht(x.astype(np.float64), s))
    torch.cuda.synchronize()


def test_fwht_signed_roundtrip_on_device(P, syn):
    # R^T R = I with R^T y = s * (H y / 32): rotate with s, rotate back with
    # all-plus signs, multiply by s
    K = 5120
    x = syn.normal_f32(7, 2, (3, K))
    s = syn.signs(7, 3, K)
    y = P.fwht(Q.dev(x), Q.dev(s))
    back = P.fwht(y, Q.dev(np.ones(K, np.int8))).cpu().numpy() * s
    np.testing.assert_allclose(back, x, atol=2e-6)


def test_fwht_empty_is_noop(P):
    import torch

    x = torch.empty((0, 1024), device="cuda")
    P.fwht(x, torch.ones(1024, dtype=torch.int8, device="cuda"), out=x)
