"""GPU parity of the embedding lookup on a rotated table (ptq_embed and
ptq_embed_ptq1) against the oracle, on the same seeded inputs.

"A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
Bonsai is": the rotation folded into the stored weights is undone on the
embedding table after each lookup.  The output is a rotation of stored
values, so it is held to the rotation's tolerance: 1e-5 (|y_ref| + rms),
plus half a bf16 unit for a bf16 output.
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


def _ids_dev(ids):
    return Q.dev(np.ascontiguousarray(ids, np.int32))


@pytest.mark.parametrize("M,V,H", [(1, 7, 1024), (5, 40, 5120), (300, 64, 2048), (33, 1, 1024)])
def test_dense_f32(P, orc, syn, M, V, H):
    table = syn.normal_f32(30, 0, (V, H))
    ids = syn.token_ids(30, 1, M, V)
    s = syn.signs(30, 2, H)
    y = P.embed(Q.dev(table), _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.embed(orc.decode_f32(table), ids, s), what=f"f32 M={M} H={H}")


@pytest.mark.parametrize("M,V,H", [(1, 9, 5120), (64, 100, 1024)])
def test_dense_bf16(P, orc, syn, M, V, H):
    table = syn.normal_bf16(31, 0, (V, H))
    ids = syn.token_ids(31, 1, M, V)
    s = syn.signs(31, 2, H)
    y = P.embed(Q.dev_bf16(table), _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.embed(orc.decode_bf16(table), ids, s), bf16_out=True,
                 what=f"bf16 M={M} H={H}")


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,V,H", [(1, 11, 5120), (40, 300, 2048)])
def test_ptq1_table(P, orc, syn, out, M, V, H):
    import torch

    t, sc = syn.weights(32, V, H)
    wq = P.pack(t)
    ids = syn.token_ids(32, 5, M, V)
    s = syn.signs(32, 6, H)
    od = torch.float32 if out == "f32" else torch.bfloat16
    y = P.embed_ptq1(Q.dev(wq), Q.dev(sc), _ids_dev(ids), Q.dev(s), out_dtype=od)
    Q.check_fwht(Q.host_f64(y), orc.embed_ptq1(wq, sc, ids, s), bf16_out=out == "bf16",
                 what=f"ptq1 {out} M={M} H={H}")


def test_ptq1_every_byte_value(P, orc, syn):
    # every byte value at every position of a block, the 13 the encoder never
    # writes included: the decode is total over 0..255
    V, H = 256, 1024
    wq = ((np.arange(V)[:, None] * 11 + np.arange(8 * 26)[None, :]) % 256).astype(np.uint8)
    sc = syn.scales_f16(33, 1, (V, H // 128))
    ids = np.arange(V, dtype=np.int32)
    s = syn.signs(33, 2, H)
    y = P.embed_ptq1(Q.dev(wq), Q.dev(sc), _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.embed_ptq1(wq, sc, ids, s), what="all bytes")


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_ptq1_every_byte_value_many_pairs(P, orc, syn, out):
    # the same table looked up 10 times over (2,560 pairs): the warp-per-pair
    # kernel, whose digits come from its code table and whose bf16 output
    # takes its signs after rounding
    import torch

    V, H = 256, 1024
    wq = ((np.arange(V)[:, None] * 7 + np.arange(8 * 26)[None, :] * 3) % 256).astype(np.uint8)
    sc = syn.scales_f16(39, 1, (V, H // 128))
    ids = np.tile(np.arange(V, dtype=np.int32), 10)
    s = syn.signs(39, 2, H)
    od = torch.float32 if out == "f32" else torch.bfloat16
    y = P.embed_ptq1(Q.dev(wq), Q.dev(sc), _ids_dev(ids), Q.dev(s), out_dtype=od)
    Q.check_fwht(Q.host_f64(y), orc.embed_ptq1(wq, sc, ids, s), bf16_out=out == "bf16",
                 what=f"all bytes, many pairs, {out}")


def test_ids_outside_the_table_give_nan_rows(P, orc, syn):
    import torch

    V, H = 16, 2048
    table = syn.normal_f32(34, 0, (V, H))
    s = syn.signs(34, 2, H)
    ids = np.array([0, V - 1, V, -1, 2 ** 31 - 1, 3, -2 ** 31], np.int32)
    y = P.embed(Q.dev(table), _ids_dev(ids), Q.dev(s))
    bad = np.array([False, False, True, True, True, False, True])
    assert torch.isnan(y[torch.from_numpy(bad).cuda()]).all()
    ref = orc.embed(orc.decode_f32(table), ids[~bad], s)
    Q.check_fwht(Q.host_f64(y[torch.from_numpy(~bad).cuda()]), ref, what="valid rows")


def test_lookup_undoes_the_fold(P, syn):
    # A table stored as R e_v (rotated on the GPU by ptq_fwht) returns e_v.
    import torch

    V, H = 12, 3072
    E = syn.normal_f32(35, 0, (V, H))
    s = syn.signs(35, 2, H)
    stored = P.fwht(Q.dev(E), Q.dev(s))
    ids = np.array([5, 0, 11, 5], np.int32)
    y = P.embed(stored, _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), E[ids].astype(np.float64), what="fold undone")
    assert not torch.equal(y, stored[torch.from_numpy(ids).long().cuda()])


def test_empty_and_in_bounds(P, syn):
    import torch

    V, H = 8, 1024
    table = Q.dev(syn.normal_f32(36, 0, (V, H)))
    s = Q.dev(syn.signs(36, 2, H))
    y = P.embed(table, _ids_dev(np.zeros(0, np.int32)), s)
    assert y.shape == (0, H)
    guard = 4096
    buf = torch.full((3 * H + 2 * guard,), float("inf"), device="cuda")
    out = buf[guard:guard + 3 * H].view(3, H)
    P.embed(table, _ids_dev(np.array([1, 7, 0], np.int32)), s, out=out)
    assert torch.isinf(buf[:guard]).all() and torch.isinf(buf[-guard:]).all()
    assert torch.isfinite(out).all()


def test_dispatch_paths(P, orc, syn):
    # a dense table with many (token, block) pairs runs a warp per pair; a
    # PTQ1_0 table past 152 x 64 CTAs x 8 warps makes a warp take several
    import torch

    V, H = 97, 5120
    table = syn.normal_f32(38, 0, (V, H))
    s = syn.signs(38, 2, H)
    ids = syn.token_ids(38, 1, 600, V)            # 3000 pairs
    y = P.embed(Q.dev(table), _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y), orc.embed(orc.decode_f32(table), ids, s), what="warp per pair")
    t, sc = syn.weights(38, V, H)
    wq = P.pack(t)
    ids = syn.token_ids(38, 3, 16000, V)          # 80000 pairs
    # bad ids: in the last pass, and next to good ones mid-way
    bad = [15999, 3000, 3001, 7000]
    ids[bad] = [V, -1, V + 5, -2 ** 31]
    y = P.embed_ptq1(Q.dev(wq), Q.dev(sc), _ids_dev(ids), Q.dev(s))
    rows = np.array([0, 1, 2999, 3002, 6999, 7001, 7777, 15197, 15198, 15998])
    Q.check_fwht(Q.host_f64(y[torch.from_numpy(rows).cuda()]), orc.embed_ptq1(wq, sc, ids[rows], s),
                 what="several pairs per warp")
    isbad = np.zeros(len(ids), bool)
    isbad[bad] = True
    mask = torch.from_numpy(isbad).cuda()
    assert torch.isnan(y[mask]).all() and torch.isfinite(y[~mask]).all()


def test_full_size_sampled(P, orc, syn):
    # the bench's shape: a 131,072 x 5,120 PTQ1_0 table (147 MB) and a bf16
    # one (1.34 GB), 2,048 ids; 24 rows checked against the oracle
    import torch

    V, H, M = 131072, 5120, 2048
    ids = syn.token_ids(37, 1, M, V)
    s = syn.signs(37, 2, H)
    rows = np.array([0, 1, 2, 100, 511, 512, 1023, 1024, 1500, 2046, 2047] +
                    list(range(700, 713)))
    t, sc = syn.weights(37, V, H)
    wq = P.pack(t)
    y = P.embed_ptq1(Q.dev(wq), Q.dev(sc), _ids_dev(ids), Q.dev(s))
    Q.check_fwht(Q.host_f64(y[torch.from_numpy(rows).cuda()]),
                 orc.embed_ptq1(wq, sc, ids[rows], s), what="ptq1 full size")
    del y
    table = syn.normal_bf16(37, 8, (V, H))
    y = P.embed(Q.dev_bf16(table), _ids_dev(ids), Q.dev(s))
    sub = orc.decode_bf16(table[ids[rows]])
    Q.check_fwht(Q.host_f64(y[torch.from_numpy(rows).cuda()]),
                 orc.embed(sub, np.arange(len(rows), dtype=np.int32), s), bf16_out=True,
                 what="bf16 full size")
