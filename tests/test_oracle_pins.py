"""Pins of the CPU oracle against what the pages and mathematics fix.

Every test here checks the oracle against something other than itself: the
hand-worked codec examples and geometry printed on the pages (tests/golden),
an independent characterisation of the base-3 decode, the textbook Sylvester
Hadamard matrix (scipy.linalg.hadamard), closed forms, invariants
(orthogonality, Parseval, the weight fold) and brute force on tiny inputs.

Source pages: "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally",
sections "What Bonsai is", "What Ferrox does with it" and "Speed, and where
it goes".
"""
import itertools

import numpy as np
import pytest
import scipy.linalg
import scipy.special

from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


# ---- codec ---------------------------------------------------------------

def test_codec_golden_examples(orc):
    rows = read_golden("ptq1_codec_examples.txt")
    for kind, *rest in rows:
        byte = int(rest[-1])
        trits = [int(v) for v in rest[:-1]]
        t = np.zeros((1, 128), np.int8)
        if kind == "full":
            t[0, 0:5] = trits            # byte 0 holds weights 0..4
            wq = orc.pack(t)
            assert wq[0, 0] == byte, (trits, wq[0, 0], byte)
        else:
            t[0, 125:128] = trits        # byte 25 holds weights 125..127
            wq = orc.pack(t)
            assert wq[0, 25] == byte, (trits, wq[0, 25], byte)
        back = orc.unpack(wq, 128)
        np.testing.assert_array_equal(back, t)


def test_codec_roundtrip_all_243_tuples(orc):
    tuples = list(itertools.product((-1, 0, 1), repeat=5))
    assert len(tuples) == 243
    # one row per tuple: byte 0 carries the tuple, the rest of the block is 0
    t = np.zeros((243, 128), np.int8)
    t[:, :5] = np.array(tuples, np.int8)
    wq = orc.pack(t)
    np.testing.assert_array_equal(orc.unpack(wq, 128), t)
    assert len(set(wq[:, 0].tolist())) == 243


def test_decode_of_every_byte_is_base3_of_floor(orc):
    # Independent characterisation: the five peeled digits of any byte are the
    # base-3 digits (most significant first) of floor(243 * byte / 256).
    for byte in range(256):
        digits = [orc.peel_digit(byte, n) for n in range(5)]
        assert all(d in (0, 1, 2) for d in digits)
        v = (243 * byte) // 256
        expect = [(v // 3 ** (4 - n)) % 3 for n in range(5)]
        assert digits == expect, byte


def test_peel_is_exact_in_fp32(orc):
    # The pages state the peel is exact in fp32: every product 3^k * byte / 256
    # has at most 16 significant bits.  Evaluate it in float32 and compare.
    for byte in range(256):
        u = np.float32(byte) / np.float32(256)
        for n in range(5):
            a = np.floor(np.float32(3 ** (n + 1)) * u)
            b = np.floor(np.float32(3 ** n) * u)
            assert int(a - np.float32(3) * b) == orc.peel_digit(byte, n)


def test_pack_refuses_invalid(orc):
    t = np.zeros((2, 128), np.int8)
    t[1, 7] = 2
    with pytest.raises(ValueError):
        orc.pack(t)
    with pytest.raises(ValueError):
        orc.pack(np.zeros((1, 100), np.int8))


def test_geometry_matches_pages(orc):
    g = {k: v for k, v in read_golden("ptq1_geometry.txt")}
    block = int(g["weights_per_block"])
    K = 4 * block
    wq = orc.pack(np.zeros((3, K), np.int8))
    bytes_per_block = wq.shape[1] // (K // block)
    assert bytes_per_block * int(g["trits_per_byte"]) >= block
    bits = (bytes_per_block * 8 + int(g["scale_bits"])) / block
    assert bits == float(g["bits_per_weight"])
    # 27e9 weights at 1.75 bits: 5.9e9 bytes = 5.5 GiB, the size on disk
    gib = float(g["model_params"]) * bits / 8 / 2 ** 30
    assert abs(gib - float(g["model_gb_on_disk"])) < 0.05


# ---- PQ2_0 ------------------------------------------------------------------

def test_pq2_geometry_matches_pages(orc):
    g = {k: v for k, v in read_golden("pq2_geometry.txt")}
    block = int(g["weights_per_block"])
    K = 4 * block
    wq = orc.pq2_pack(np.zeros((3, K), np.int8))
    bytes_per_block = wq.shape[1] // (K // block)
    assert bytes_per_block * 8 == block * int(g["bits_per_code"])
    bits = (bytes_per_block * 8 + int(g["scale_bits"])) / block
    assert bits == float(g["bits_per_weight"])
    # 27e9 weights at 2.125 bits: 7.17e9 bytes, "7.2 GB"; 16 bits: 54 GB
    assert abs(float(g["model_params"]) * bits / 8 / 1e9 - float(g["model_gb"])) < 0.05
    assert float(g["model_params"]) * 16 / 8 / 1e9 == float(g["model_gb_16bit"])


def test_pq2_fields_are_independent(orc):
    # changing one weight changes one 2-bit field of one byte, and a byte's
    # four fields are its four weights in order
    rng = np.random.default_rng(30)
    t = rng.integers(-1, 2, size=(2, 256)).astype(np.int8)
    w0 = orc.pq2_pack(t)
    for k in (0, 1, 3, 4, 127, 128, 255):
        t2 = t.copy()
        t2[1, k] = (t2[1, k] + 2) % 3 - 1
        diff = np.argwhere(orc.pq2_pack(t2) != w0)
        assert diff.tolist() == [[1, k // 4]]
        bits = int(orc.pq2_pack(t2)[1, k // 4]) ^ int(w0[1, k // 4])
        assert bits & ~(3 << (2 * (k % 4))) == 0
    np.testing.assert_array_equal(orc.pq2_unpack(w0, 256), t)


def test_pq2_decode_of_every_byte(orc):
    # 256 bytes x 4 fields: exactly 81 = 3^4 bytes decode to four trits, the
    # rest hold at least one code 3, which decodes to +2
    codes = np.arange(256, dtype=np.uint8).reshape(8, 32)  # 8 one-block rows
    allb = orc.pq2_unpack(codes, 128).reshape(256, 4)      # byte b -> its 4 weights
    assert set(np.unique(allb).tolist()) == {-1, 0, 1, 2}
    assert int((allb <= 1).all(axis=1).sum()) == 81
    # byte 0b11100100 holds codes 0, 1, 2, 3 from the low bits up
    np.testing.assert_array_equal(allb[0b11100100], [-1, 0, 1, 2])


def test_pq2_matmul_brute_force(orc):
    # against a dense product built from the trits and scales directly
    rng = np.random.default_rng(31)
    N, K, M = 6, 512, 3
    t = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    sbits = (np.abs(rng.standard_normal((N, K // 128))) * 0.02).astype(np.float16).view(np.uint16)
    x = rng.standard_normal((M, K))
    W = t * np.repeat(_f16(sbits), 128, axis=1)
    y = orc.pq2_matmul(orc.pq2_pack(t), sbits, x)
    np.testing.assert_allclose(y, x @ W.T, rtol=1e-12, atol=1e-12)
    rows = [5, 0, 3]
    np.testing.assert_allclose(orc.pq2_matmul_rows(orc.pq2_pack(t), sbits, x, rows), (x @ W.T)[:, rows],
                               rtol=1e-12, atol=1e-12)


def test_pq2_pack_refuses_invalid(orc):
    with pytest.raises(ValueError):
        orc.pq2_pack(np.full((1, 128), 2, np.int8))
    with pytest.raises(ValueError):
        orc.pq2_pack(np.zeros((1, 100), np.int8))


# ---- storage decodes -------------------------------------------------------

def test_half_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    assert orc.half_to_double(0x0001) == 2.0 ** -24


def test_bf16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.decode_bf16(bits)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])


# ---- rotation --------------------------------------------------------------

def test_fwht_unsigned_is_sylvester_hadamard(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 1024))
    ones = np.ones(1024, np.int8)
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    np.testing.assert_allclose(orc.fwht_def(x, ones), x @ H.T / 32, rtol=0, atol=1e-12)


def test_fwht_signed_flips_then_rotates(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 2048))
    s = np.where(rng.random(2048) < 0.5, -1, 1).astype(np.int8)
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    y = orc.fwht_def(x, s)
    for b in range(2):
        sl = slice(1024 * b, 1024 * (b + 1))
        expect = (x[:, sl] * s[sl]) @ H.T / 32
        np.testing.assert_allclose(y[:, sl], expect, rtol=0, atol=1e-12)


def test_fwht_butterfly_equals_definition(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 3072))
    s = np.where(rng.random(3072) < 0.5, -1, 1).astype(np.int8)
    np.testing.assert_allclose(orc.fwht(x, s), orc.fwht_def(x, s), rtol=0, atol=1e-12)


def test_fwht_unsigned_is_involution(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 1024))
    ones = np.ones(1024, np.int8)
    np.testing.assert_allclose(orc.fwht(orc.fwht(x, ones), ones), x, atol=1e-12)


def test_fwht_signed_roundtrip_and_parseval(orc):
    # R = H D_s / 32 is orthogonal: R^T (R x) = D_s H (R x) / 32 = x.
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 2048))
    s = np.where(rng.random(2048) < 0.5, -1, 1).astype(np.int8)
    y = orc.fwht(x, s)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    back = orc.fwht(y, np.ones(2048, np.int8)) * s
    np.testing.assert_allclose(back, x, atol=1e-12)


def test_fwht_unit_vector(orc):
    s = np.where(np.arange(1024) % 3 == 0, -1, 1).astype(np.int8)
    e0 = np.zeros((1, 1024))
    e0[0, 0] = 1.0
    np.testing.assert_array_equal(orc.fwht_def(e0, s), np.full((1, 1024), s[0] / 32.0))


def test_weight_fold_identity(orc):
    # The fold of "What Bonsai is": a weight multiplied by the rotation,
    # applied to a rotated activation, gives the plain product:
    # (W R^T)(R x) = W x, with row n of W R^T equal to R w_n.
    rng = np.random.default_rng(6)
    for K in (1024, 2048):
        W = rng.standard_normal((3, K))
        x = rng.standard_normal((1, K))
        s = np.where(rng.random(K) < 0.5, -1, 1).astype(np.int8)
        folded = orc.fwht(W, s)
        xr = orc.fwht(x, s)
        np.testing.assert_allclose(folded @ xr[0], W @ x[0], rtol=1e-12, atol=1e-12)


# ---- inverse rotation and the embedding lookup -------------------------------

def _signs(rng, n):
    return np.where(rng.random(n) < 0.5, -1, 1).astype(np.int8)


def test_unrotate_is_transpose_of_sylvester_rotation(orc):
    # R = H D_s / 32 with the textbook Sylvester H (scipy), so R^T = D_s H / 32:
    # the butterfly first, then the signs -- not the forward transform again.
    rng = np.random.default_rng(21)
    y = rng.standard_normal((2, 2048))
    s = _signs(rng, 2048)
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    x = orc.unrotate_def(y, s)
    for b in range(2):
        sl = slice(1024 * b, 1024 * (b + 1))
        np.testing.assert_allclose(x[:, sl], (y[:, sl] @ H / 32) * s[sl], rtol=0, atol=1e-12)
    assert np.abs(x - orc.fwht(y, s)).max() > 0.1  # signed R is not symmetric


def test_unrotate_inverts_the_rotation(orc):
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 3072))
    s = _signs(rng, 3072)
    np.testing.assert_allclose(orc.unrotate_def(orc.fwht_def(x, s), s), x, rtol=0, atol=1e-12)
    np.testing.assert_allclose(orc.fwht_def(orc.unrotate_def(x, s), s), x, rtol=0, atol=1e-12)


def test_unrotate_closed_forms(orc):
    # R^T (32 e_j) = s * H[:, j], i.e. x_i = s_i (-1)^popcount(i & j); for
    # j = 0 that is the sign vector itself.  With all signs +1 the all-ones
    # block goes to 32 e_0.
    s = np.where(np.arange(1024) % 5 == 1, -1, 1).astype(np.int8)
    i = np.arange(1024)
    for j in (0, 1, 7, 640, 1023):
        y = np.zeros((1, 1024))
        y[0, j] = 32.0
        parity = np.array([bin(v & j).count("1") & 1 for v in i])
        np.testing.assert_array_equal(orc.unrotate_def(y, s)[0], s * np.where(parity, -1.0, 1.0))
    ones = np.ones(1024, np.int8)
    e0 = np.zeros(1024)
    e0[0] = 32.0
    np.testing.assert_array_equal(orc.unrotate_def(np.ones((1, 1024)), ones)[0], e0)


def test_embed_undoes_the_fold(orc):
    # "What Bonsai is": the rotation is folded into the stored table and
    # undone after each lookup.  A table stored as R e_v returns e_v.
    rng = np.random.default_rng(23)
    V, H = 9, 2048
    E = rng.standard_normal((V, H))
    s = _signs(rng, H)
    stored = orc.fwht_def(E, s)
    ids = np.array([3, 0, 8, 3, 9, -1, 2 ** 31 - 1], np.int32)
    out = orc.embed(stored, ids, s)
    np.testing.assert_allclose(out[:4], E[[3, 0, 8, 3]], rtol=0, atol=1e-12)
    assert np.isnan(out[4:]).all()  # ids outside [0, V)


def test_embed_ptq1_row_is_trits_times_block_scales(orc):
    # the table row decoded straight from the trits and scales the encoder
    # was given (numpy here, not the oracle's peel), then un-rotated
    rng = np.random.default_rng(24)
    V, H = 5, 1024
    t = rng.integers(-1, 2, size=(V, H)).astype(np.int8)
    sbits = (np.abs(rng.standard_normal((V, H // 128))) * 0.02).astype(np.float16).view(np.uint16)
    dense = t * np.repeat(_f16(sbits), 128, axis=1)
    s = _signs(rng, H)
    ids = np.array([4, 1, 1, 5], np.int32)
    out = orc.embed_ptq1(orc.pack(t), sbits, ids, s)
    H1 = scipy.linalg.hadamard(1024).astype(np.float64)
    np.testing.assert_allclose(out[:3], (dense[[4, 1, 1]] @ H1 / 32) * s, rtol=0, atol=1e-12)
    assert np.isnan(out[3]).all()


# ---- ternary matmul --------------------------------------------------------

def test_ternary_dot_brute_force(orc):
    rng = np.random.default_rng(7)
    N, K, M = 5, 384, 2
    t = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    sbits = (np.abs(rng.standard_normal((N, K // 128))) * 0.02).astype(np.float16).view(np.uint16)
    x = rng.standard_normal((M, K))
    y = orc.matmul(orc.pack(t), sbits, x)
    s = _f16(sbits)
    for m in range(M):
        for n in range(N):
            total = 0.0
            for b in range(K // 128):
                plus = minus = 0.0
                for i in range(128 * b, 128 * (b + 1)):
                    if t[n, i] == 1:
                        plus += x[m, i]
                    elif t[n, i] == -1:
                        minus += x[m, i]
                total += s[n, b] * (plus - minus)
            assert abs(y[m, n] - total) <= 1e-12 * (1 + abs(total))


def test_matmul_one_hot_is_exact(orc):
    rng = np.random.default_rng(8)
    N, K = 6, 512
    t = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    sbits = (np.abs(rng.standard_normal((N, K // 128))) + 0.5).astype(np.float16).view(np.uint16)
    wq = orc.pack(t)
    s = _f16(sbits)
    for k in (0, 4, 5, 127, 128, 300, 511):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        y = orc.matmul(wq, sbits, x)
        np.testing.assert_array_equal(y[0], s[:, k // 128] * t[:, k])


def test_matmul_special_scales(orc):
    K = 256
    ones = np.ones((2, K), np.int8)
    x = np.arange(K, dtype=np.float64)[None, :]
    one = np.full((2, 2), 0x3C00, np.uint16)                   # 1.0
    y = orc.matmul(orc.pack(ones), one, x)
    assert y[0, 0] == x.sum() and y[0, 1] == x.sum()
    zero = np.zeros((2, 2), np.uint16)
    assert not orc.matmul(orc.pack(ones), zero, x).any()
    sub = np.full((2, 2), 0x0001, np.uint16)                   # 2^-24
    e = np.zeros((1, K))
    e[0, 200] = 1.0
    assert orc.matmul(orc.pack(ones), sub, e)[0, 0] == 2.0 ** -24
    assert not orc.matmul(orc.pack(np.zeros((2, K), np.int8)), one, x).any()


def test_matmul_rows_equals_full(orc, syn):
    mv = syn.gaussian_matvec(11, 3, 40, 1024)
    wq = orc.pack(mv.trits)
    x = orc.decode_f32(mv.x)
    full = orc.matmul(wq, mv.scales, x)
    rows = [0, 7, 39, 13]
    np.testing.assert_array_equal(orc.matmul_rows(wq, mv.scales, x, rows), full[:, rows])


# ---- SwiGLU and the feed-forward block ------------------------------------

def test_swiglu_closed_forms(orc):
    g = np.array([0.0, 40.0, -40.0, 1.5, -1.5, 3.0])
    one = np.ones_like(g)
    h = orc.swiglu(g, one)
    assert h[0] == 0.0
    assert abs(h[1] - 40.0) < 1e-12 and abs(h[2]) < 1e-12
    assert abs((h[3] - h[4]) - 1.5) < 1e-15          # silu(a) - silu(-a) = a
    u = np.array([2.0, 1.0, 1.0, -3.0, 0.5, 0.25])
    np.testing.assert_allclose(orc.swiglu(g, u), g * scipy.special.expit(g) * u, rtol=1e-14)


def test_ffn_against_dense_numpy(orc, syn):
    # Independent route: dense real-valued weights from the trits and the
    # numpy fp16 decode, the rotation as the scipy Sylvester matrix.
    H_, I_, M = 1024, 2048, 2
    t_gu, s_gu = syn.weights(21, 2 * I_, H_)
    t_d, s_d = syn.weights(22, H_, I_)
    s_in = syn.signs(23, 3, H_)
    s_mid = syn.signs(23, 4, I_)
    x = syn.normal_f64(23, 2, (M, H_))
    y = orc.ffn(orc.pack(t_gu), s_gu, orc.pack(t_d), s_d, s_in, s_mid, x)

    Had = scipy.linalg.hadamard(1024).astype(np.float64) / 32

    def rot(v, s):
        out = np.empty_like(v)
        for b in range(v.shape[1] // 1024):
            sl = slice(1024 * b, 1024 * (b + 1))
            out[:, sl] = (v[:, sl] * s[sl]) @ Had.T
        return out

    def dense(t, sbits):
        return t.astype(np.float64) * np.repeat(_f16(sbits), 128, axis=1)

    gu = rot(x, s_in) @ dense(t_gu, s_gu).T
    h = gu[:, :I_] * scipy.special.expit(gu[:, :I_]) * gu[:, I_:]
    ref = rot(h, s_mid) @ dense(t_d, s_d).T
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())


# ---- the chained feed-forward stack ------------------------------------------

def _stack_layer(syn, seed, l, H, I):
    L = syn.ffn_layer(seed, l, H, I)
    return (np.ascontiguousarray(__import__("oracle").pack(L.wgu_trits)), L.wgu_scales,
            np.ascontiguousarray(__import__("oracle").pack(L.wd_trits)), L.wd_scales,
            L.signs_in, L.signs_mid)


def test_stack_identities(orc, syn):
    H, I = 1024, 1024
    x = syn.normal_f64(60, 2, (2, H))
    lay = _stack_layer(syn, 60, 0, H, I)
    g = np.ones(H)
    np.testing.assert_array_equal(orc.ffn_stack([], [], x, 1e-6), x)  # no layers
    zero = (orc.pack(np.zeros((2 * I, H), np.int8)), lay[1], orc.pack(np.zeros((H, I), np.int8)),
            lay[3], lay[4], lay[5])
    np.testing.assert_array_equal(orc.ffn_stack([zero], [g], x, 1e-6), x)  # residual only


def test_stack_composes_and_is_scale_free(orc, syn):
    H, I = 1024, 2048
    x = syn.normal_f64(61, 2, (3, H))
    l0, l1 = _stack_layer(syn, 61, 0, H, I), _stack_layer(syn, 61, 1, H, I)
    g0 = 1.0 + 0.1 * syn.normal_f64(61, 7, (H,))
    g1 = 1.0 + 0.1 * syn.normal_f64(61, 8, (H,))
    two = orc.ffn_stack([l0, l1], [g0, g1], x, 1e-5)
    one_one = orc.ffn_stack([l1], [g1], orc.ffn_stack([l0], [g0], x, 1e-5), 1e-5)
    np.testing.assert_allclose(two, one_one, rtol=0, atol=1e-12)
    # eps = 0: the norm removes any positive scale of x, so the block adds the
    # same increment to c x as to x
    c = 3.7
    inc = orc.ffn_stack([l0], [g0], x, 0.0) - x
    inc_c = orc.ffn_stack([l0], [g0], c * x, 0.0) - c * x
    np.testing.assert_allclose(inc_c, inc, rtol=1e-12, atol=1e-12)


def test_stack_rows_are_independent(orc, syn):
    # every token row goes through the stack on its own (the norm is per row):
    # a 3-row call equals three 1-row calls, for rows of different scales
    H, I = 1024, 1024
    x = syn.normal_f64(64, 2, (3, H)) * np.array([[1.0], [5.0], [0.2]])
    lay = _stack_layer(syn, 64, 0, H, I)
    g = 1.0 + 0.1 * syn.normal_f64(64, 7, (H,))
    all3 = orc.ffn_stack([lay], [g], x, 1e-5)
    for m in range(3):
        np.testing.assert_allclose(all3[m:m + 1], orc.ffn_stack([lay], [g], x[m:m + 1], 1e-5),
                                   rtol=0, atol=1e-12)


def test_stack_rmsnorm_worked_values(orc, syn):
    # rows of 3s and 4s have mean square 12.5: with eps = 0 and unit gains
    # the block's input is x / sqrt(12.5), i.e. 0.8485... and 1.1313...
    H, I = 1024, 1024
    x = np.tile([3.0, 4.0], (1, H // 2))
    lay = _stack_layer(syn, 62, 0, H, I)
    xn = np.tile([3.0 / np.sqrt(12.5), 4.0 / np.sqrt(12.5)], (1, H // 2))
    expect = x + orc.ffn(*lay, xn)
    np.testing.assert_allclose(orc.ffn_stack([lay], [np.ones(H)], x, 0.0), expect, rtol=1e-12,
                               atol=1e-12)


def test_stack_gain_and_eps_worked_values(orc, syn):
    # rows of 3s and 4s (mean square 12.5).  Gains alternating 2 and 1/2 with
    # eps = 0 give the block 6/sqrt(12.5) and 2/sqrt(12.5); eps = 3.5 with unit
    # gains makes the divisor sqrt(16) = 4 exactly, so the block sees 0.75 and
    # 1.0 (a divisor sqrt(12.5) + 3.5 would not)
    H, I = 1024, 1024
    x = np.tile([3.0, 4.0], (1, H // 2))
    lay = _stack_layer(syn, 63, 0, H, I)
    g = np.tile([2.0, 0.5], H // 2)
    xn = np.tile([6.0 / np.sqrt(12.5), 2.0 / np.sqrt(12.5)], (1, H // 2))
    np.testing.assert_allclose(orc.ffn_stack([lay], [g], x, 0.0), x + orc.ffn(*lay, xn),
                               rtol=1e-12, atol=1e-12)
    xn = np.tile([0.75, 1.0], (1, H // 2))
    np.testing.assert_allclose(orc.ffn_stack([lay], [np.ones(H)], x, 3.5), x + orc.ffn(*lay, xn),
                               rtol=1e-12, atol=1e-12)
