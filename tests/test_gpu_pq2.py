"""GPU parity of the PQ2_0 path (2-bit codes, one fp16 scale per 128
weights; "Why I Am Building Another Inference Engine", section "Level 2: The
short answer") against the oracle: the device decode bit for bit, the
table-lookup decode GEMV (fp32) and the tensor-core prefill GEMM (bf16), at
the workload sizes and on small and ragged shapes."""
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


def run(P, t, s, x):
    wq = P.pq2_pack(t)
    xd = Q.dev(x) if x.dtype == np.float32 else Q.dev_bf16(x)
    return P.matmul_pq2(Q.dev(wq), Q.dev(s), xd), wq


def test_unpack_bit_exact(P, orc, syn):
    t, _ = syn.weights(41, 300, 2048)
    wq = P.pq2_pack(t)
    got = P.pq2_unpack(Q.dev(wq), 2048).cpu().numpy()
    np.testing.assert_array_equal(got, t)
    # every byte value, code 3 (never written) included: trit = code - 1
    allb = np.arange(256, dtype=np.uint8).reshape(8, 32)
    np.testing.assert_array_equal(P.pq2_unpack(Q.dev(allb), 128).cpu().numpy(),
                                  orc.pq2_unpack(allb, 128))


@pytest.mark.parametrize("M", [1, 4])
def test_decode_gate_up(P, orc, syn, M):
    mv = syn.gaussian_matvec(42, M, 17408, 5120)
    y, wq = run(P, mv.trits, mv.scales, mv.x)
    Q.check_f32(Q.host_f64(y), orc.pq2_matmul(wq, mv.scales, Q.x_f64(mv.x)), f"pq2 gate/up M={M}")


@pytest.mark.parametrize("M", [1, 8])
def test_decode_down(P, orc, syn, M):
    t, s = syn.weights(43, 5120, 17408, p_zero=0.4)
    x = Q.swiglu_like(43, M, 17408)
    y, wq = run(P, t, s, x)
    Q.check_f32(Q.host_f64(y), orc.pq2_matmul(wq, s, Q.x_f64(x)), f"pq2 down M={M}")


@pytest.mark.parametrize("N,K", [(1, 1024), (33, 2048), (700, 3072), (2000, 4096)])
def test_decode_small_shapes(P, orc, syn, N, K):
    mv = syn.gaussian_matvec(44 + K // 1024, 1, N, K)
    y, wq = run(P, mv.trits, mv.scales, mv.x)
    Q.check_f32(Q.host_f64(y), orc.pq2_matmul(wq, mv.scales, Q.x_f64(mv.x)), f"pq2 N={N} K={K}")


def test_decode_every_byte_value(P, orc, syn):
    # every byte at every position of a block, code 3 included
    N, K = 512, 2048
    wq = ((np.arange(N)[:, None] * 5 + np.arange(K // 4)[None, :]) % 256).astype(np.uint8)
    s = syn.scales_f16(45, 1, (N, K // 128))
    x = syn.normal_f32(45, 2, (1, K))
    y = P.matmul_pq2(Q.dev(wq), Q.dev(s), Q.dev(x))
    Q.check_f32(Q.host_f64(y), orc.pq2_matmul(wq, s, Q.x_f64(x)), "pq2 all bytes")


def test_prefill_sampled(P, orc, syn):
    # M = 512 x K = 5120 x N = 17408, bf16; 40 output rows against the oracle
    mv = syn.gaussian_matvec(46, 512, 17408, 5120, dtype="bf16")
    y, wq = run(P, mv.trits, mv.scales, mv.x)
    rows = np.array([0, 1, 127, 128, 129, 5000, 9999, 17407] + list(range(300, 332)))
    ref = orc.pq2_matmul_rows(wq, mv.scales, Q.x_f64(mv.x), rows)
    Q.check_bf16(Q.host_f64(y)[:, rows], ref, "pq2 prefill M=512")


@pytest.mark.parametrize("M,N,K", [(70, 300, 2048), (300, 1000, 1024), (128, 5120, 17408)])
def test_prefill_shapes(P, orc, syn, M, N, K):
    # ragged M and N; the last shape has 40 tiles and runs split along K
    mv = syn.gaussian_matvec(47 + M, M, N, K, dtype="bf16")
    y, wq = run(P, mv.trits, mv.scales, mv.x)
    rows = np.unique(np.linspace(0, N - 1, 37).astype(np.int64))
    ref = orc.pq2_matmul_rows(wq, mv.scales, Q.x_f64(mv.x), rows)
    Q.check_bf16(Q.host_f64(y)[:, rows], ref, f"pq2 prefill {M}x{N}x{K}")


def test_prefill_every_byte_value(P, orc, syn):
    M, N, K = 64, 256, 1024
    wq = ((np.arange(N)[:, None] * 3 + np.arange(K // 4)[None, :]) % 256).astype(np.uint8)
    s = syn.scales_f16(48, 1, (N, K // 128))
    x = syn.normal_bf16(48, 2, (M, K))
    y = P.matmul_pq2(Q.dev(wq), Q.dev(s), Q.dev_bf16(x))
    Q.check_bf16(Q.host_f64(y), orc.pq2_matmul(wq, s, orc.decode_bf16(x)), "pq2 prefill all bytes")


def test_refuses_k_not_multiple_of_1024(P, syn):
    mv = syn.gaussian_matvec(49, 1, 64, 1152)
    with pytest.raises(P.PTQError, match="UNSUPPORTED"):
        run(P, mv.trits, mv.scales, mv.x)
