"""GPU parity of ptq_rotate_matmul, y = (R x) W^T, against the oracle's
rotation followed by its matmul: the fp32 decode route (M <= 8) rotates
inside the table-lookup GEMV (one or two 1024-blocks per chunk, each token in
turn), the bf16 route runs the rotation kernel first."""
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


def rot_ref(orc, t, s, x64, signs):
    return orc.matmul(orc.pack(t), s, orc.fwht(x64, signs))


@pytest.mark.parametrize("N,K", [(1024, 1024), (17408, 5120), (300, 2048), (77, 3072), (5, 1024)])
def test_rotate_gemv_fused(P, orc, syn, N, K):
    # K = 1024: every chunk inside one rotation block; 2048..5120: chunks
    # straddling two blocks
    mv = syn.gaussian_matvec(300 + K // 1024, 1, N, K)
    signs = syn.signs(300 + K // 1024, 9, K)
    y = P.rotate_matmul(Q.dev(P.pack(mv.trits)), Q.dev(mv.scales), Q.dev(mv.x), Q.dev(signs))
    Q.check_f32(Q.host_f64(y), rot_ref(orc, mv.trits, mv.scales, Q.x_f64(mv.x), signs),
                f"rotate+gemv {N}x{K}")


def test_rotate_gemv_down_shape(P, orc, syn):
    t, s = syn.weights(2, 5120, 17408, p_zero=0.4)
    h = Q.swiglu_like(2, 1, 17408)
    signs = syn.signs(2, 9, 17408)
    y = P.rotate_matmul(Q.dev(P.pack(t)), Q.dev(s), Q.dev(h), Q.dev(signs))
    Q.check_f32(Q.host_f64(y), rot_ref(orc, t, s, Q.x_f64(h), signs), "rotate+gemv down")


def test_rotate_gemv_several_tokens_full_size(P, orc, syn):
    # the bench's multi-token decode calls: 4 tokens on the gate/up shape and
    # 8 on the down shape, one launch taking the tokens in turn
    mv = syn.gaussian_matvec(330, 4, 17408, 5120)
    signs = syn.signs(330, 9, 5120)
    y = P.rotate_matmul(Q.dev(P.pack(mv.trits)), Q.dev(mv.scales), Q.dev(mv.x), Q.dev(signs))
    Q.check_f32(Q.host_f64(y), rot_ref(orc, mv.trits, mv.scales, Q.x_f64(mv.x), signs),
                "rotate+gemv M=4 17408x5120")
    t, s = syn.weights(331, 5120, 17408, p_zero=0.4)
    h = Q.swiglu_like(331, 8, 17408)
    signs = syn.signs(331, 9, 17408)
    y = P.rotate_matmul(Q.dev(P.pack(t)), Q.dev(s), Q.dev(h), Q.dev(signs))
    Q.check_f32(Q.host_f64(y), rot_ref(orc, t, s, Q.x_f64(h), signs), "rotate+gemv M=8 down")


def test_rotate_matches_separate_calls(P, syn):
    import torch

    mv = syn.gaussian_matvec(310, 1, 4000, 5120)
    signs = Q.dev(syn.signs(310, 9, 5120))
    wq, s, x = Q.dev(P.pack(mv.trits)), Q.dev(mv.scales), Q.dev(mv.x)
    x0 = x.clone()
    fused = P.rotate_matmul(wq, s, x, signs)
    sep = P.matmul(wq, s, P.fwht(x, signs))
    assert torch.equal(x, x0)  # x is not modified
    # same tables from differently rounded rotations: equal within fp32 noise
    rel = (fused - sep).abs().max() / sep.abs().max()
    assert rel < 1e-5, float(rel)


@pytest.mark.parametrize("M,N,K,dtype", [(1, 17408, 5120, "f32"), (4, 1000, 2048, "f32"),
                                         (3, 700, 3072, "bf16")])
def test_rotate_matmul_host_buffers(P, orc, syn, M, N, K, dtype):
    # ptq_rotate_matmul_host: x from page-locked host memory, y back to it,
    # around the same product; the result has the bits of the device call
    import torch

    mv = syn.gaussian_matvec(330 + M, M, N, K, dtype=dtype)
    signs = Q.dev(syn.signs(330 + M, 9, K))
    wq, s = Q.dev(P.pack(mv.trits)), Q.dev(mv.scales)
    xd = Q.dev(mv.x) if dtype == "f32" else Q.dev_bf16(mv.x)
    ref = P.rotate_matmul(wq, s, xd, signs)
    xh = xd.cpu().pin_memory()
    yh = torch.full((M, N), float("nan"), dtype=xd.dtype).pin_memory()
    ws = torch.empty(P.rotate_matmul_host_workspace_bytes(M, N, K, P._act_dtype(xd)),
                     dtype=torch.uint8, device="cuda")
    # page-locked buffers (mapped: the kernels read x and write y in place),
    # then ordinary pageable ones (the copy path)
    P.rotate_matmul_host(wq, s, xh, signs, yh, ws)
    torch.cuda.synchronize()
    assert torch.equal(yh, ref.cpu())
    xp, yp = xd.cpu(), torch.full((M, N), float("nan"), dtype=xd.dtype)
    P.rotate_matmul_host(wq, s, xp, signs, yp, ws)
    torch.cuda.synchronize()
    assert torch.equal(yp, ref.cpu())
    rows = np.unique(np.linspace(0, N - 1, 64).astype(np.int64))
    want = orc.matmul(orc.pack(mv.trits[rows]), mv.scales[rows],
                      orc.fwht(Q.x_f64(mv.x), syn.signs(330 + M, 9, K)))
    got = yh.float().numpy().astype(np.float64)[:, rows]
    (Q.check_f32 if dtype == "f32" else Q.check_bf16)(got, want, f"host buffers {M}x{N}x{K}")


@pytest.mark.parametrize("M,dtype", [(4, "f32"), (8, "f32"), (64, "bf16"), (3, "bf16")])
def test_rotate_matmul_other_sizes(P, orc, syn, M, dtype):
    N, K = 600, 2048
    mv = syn.gaussian_matvec(320 + M, M, N, K, dtype=dtype)
    signs = syn.signs(320 + M, 9, K)
    xd = Q.dev(mv.x) if dtype == "f32" else Q.dev_bf16(mv.x)
    wq = P.pack(mv.trits)
    y = P.rotate_matmul(Q.dev(wq), Q.dev(mv.scales), xd, Q.dev(signs))
    ref = rot_ref(orc, mv.trits, mv.scales, Q.x_f64(mv.x), signs)
    if dtype == "f32":
        Q.check_f32(Q.host_f64(y), ref, f"rotate+matmul M={M}")
    else:
        # the rotated operand is held in fp16 before the GEMM (2^-11), whose
        # weight tile is then exact
        Q.check_bf16(Q.host_f64(y), ref, f"rotate+gemm M={M}")


def test_rotate_matmul_refusals(P, syn):
    import torch

    mv = syn.gaussian_matvec(330, 1, 64, 1024)
    wq, s, x = Q.dev(P.pack(mv.trits)), Q.dev(mv.scales), Q.dev(mv.x)
    signs = Q.dev(syn.signs(330, 9, 1024))
    need = P.rotate_matmul_workspace_bytes(1, 64, 1024, P.PTQ_F32)
    with pytest.raises(P.PTQError, match="WORKSPACE"):
        P.rotate_matmul(wq, s, x, signs, workspace=torch.empty(need - 16, dtype=torch.uint8,
                                                               device="cuda"))
    mv2 = syn.gaussian_matvec(331, 1, 64, 1280)  # K % 1024 != 0
    with pytest.raises(P.PTQError, match="SHAPE"):
        P.rotate_matmul(Q.dev(P.pack(mv2.trits)), Q.dev(mv2.scales), Q.dev(mv2.x),
                        Q.dev(syn.signs(331, 9, 1280)))
