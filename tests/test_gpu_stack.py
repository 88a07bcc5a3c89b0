"""GPU parity of ptq_ffn_stack (L chained pre-norm feed-forward blocks over
an fp32 residual stream) against the oracle's fp64 stack.

Tolerance.  The stack's error is the sum of its blocks' errors plus what the
later blocks do with the earlier ones.  Block l adds y_l to x; its own error
is within the single-block tolerance of y_l (fp32 path: 1e-4 (|y_l| +
rms(y_l)); bf16 path: 1e-2 rms(y_l) + 2^-8 |y_l|).  An error d in x reaches
the next block's output scaled by at most 2 rho, with
rho = max_l rms(y_l) / rms(x_l): the norm divides d by rms(x), and SwiGLU's
product of two linear maps at most doubles a relative change.  So after L
blocks
    |x - x_ref| <= (1 + 2 rho)^(L-1) * sum_l [tol(y_l) + k 2^-24 |x_(l+1)|],
with every y_l and x_l taken from the oracle, layer by layer.  The last
term is the fp32 storage of the residual stream itself: each addition into
x rounds once, by at most 2^-24 |x|, and a layer makes k of them -- one per
K-chunk of the down projection (ceil(13 I / 256 / 32) chunks of at most 32
words) when the chunk sums are added into x one at a time, which bounds the
single addition of the per-layer path too."""
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


def make_layers(P, orc, syn, seed, Lc, H, I):
    """Device tuples, oracle tuples and fp32 gains of Lc seeded layers."""
    dev, host, gains = [], [], []
    for l in range(Lc):
        F = syn.ffn_layer(seed, l, H, I)
        gq, dq = P.pack(F.wgu_trits), P.pack(F.wd_trits)
        dev.append((Q.dev(gq), Q.dev(F.wgu_scales), Q.dev(dq), Q.dev(F.wd_scales),
                    Q.dev(F.signs_in), Q.dev(F.signs_mid)))
        host.append((orc.pack(F.wgu_trits), F.wgu_scales, orc.pack(F.wd_trits), F.wd_scales,
                     F.signs_in, F.signs_mid))
        del F
        gains.append(syn.norm_gain(seed, l, H))
    return dev, host, gains


def down_chunks(I):
    """K-chunks of a row of the down projection: 13 I / 256 words, <= 32 each."""
    return -(-(13 * I // 256) // 32)


def oracle_with_bound(orc, host, gains, x64, eps, bf16):
    """The oracle's stack output and the elementwise bound of the docstring."""
    x = x64.copy()
    tol = np.zeros_like(x)
    rho = 0.0
    k = down_chunks(host[0][5].shape[0]) if host else 1
    for lay, g in zip(host, gains):
        nx = orc.ffn_stack([lay], [g.astype(np.float64)], x, eps)
        y = nx - x
        r = Q.rms(y)
        tol += (1e-2 * r + 2.0 ** -8 * np.abs(y)) if bf16 else 1e-4 * (np.abs(y) + r)
        tol += k * 2.0 ** -24 * np.abs(nx)
        rho = max(rho, r / Q.rms(x))
        x = nx
    return x, tol * (1.0 + 2.0 * rho) ** (len(host) - 1)


def check_stack(y, ref, bound, what):
    y = np.asarray(y, np.float64)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    err = np.abs(y - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
                             f"y={y[i]!r} ref={ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")


def run_stack(P, dev, gains, x, eps, act):
    import torch

    xd = Q.dev(np.ascontiguousarray(x, np.float32))
    P.ffn_stack(dev, [Q.dev(g) for g in gains], xd, eps, act=act)
    torch.cuda.synchronize()
    return xd.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,act", [(1, "f32"), (3, "f32"), (8, "f32"), (5, "bf16"), (70, "bf16")])
def test_stack_small(P, orc, syn, M, act):
    import torch

    H, I, Lc, eps = 1024, 2048, 3, 1e-6
    dev, host, gains = make_layers(P, orc, syn, 30 + M, Lc, H, I)
    x = syn.ffn_input(30 + M, 0, M, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.float32 if act == "f32" else torch.bfloat16)
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, act == "bf16")
    check_stack(got, ref, bound, f"stack L={Lc} M={M} {act}")


@pytest.mark.parametrize("H", [1024, 5120, 12288, 17408])
@pytest.mark.parametrize("M,act", [(1, "f32"), (2, "f32"), (3, "bf16")])
def test_stack_row_lengths(P, orc, syn, H, M, act):
    # fp32 runs the persistent kernel, whose gate/up rows are cut into 4 to
    # 28 K-chunks and whose down rows into 2; bf16 runs per layer, where the
    # add-and-norm kernel holds 1, 2 or 4 vectors of a row per thread (H =
    # 1024, 5120, 12288) and loops over longer rows (H = 17408)
    import torch

    I, Lc, eps = 1024, 2, 1e-6
    dev, host, gains = make_layers(P, orc, syn, 50 + H // 1024, Lc, H, I)
    x = syn.ffn_input(50, 0, M, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.float32 if act == "f32" else torch.bfloat16)
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, act == "bf16")
    check_stack(got, ref, bound, f"stack H={H} M={M} {act}")


def test_stack_routes(P):
    # 1 to 8 fp32 tokens run the persistent kernel; bf16 runs per layer
    for M in (1, 2, 8):
        assert P.ffn_stack_route(M, 5120, 17408, P.PTQ_F32) == "stack_decode_persistent"
    assert P.ffn_stack_route(1, 1024, 2048, P.PTQ_F32) == "stack_decode_persistent"
    assert P.ffn_stack_route(1, 5120, 17408, P.PTQ_BF16) == "stack_per_layer"
    assert P.ffn_stack_route(256, 5120, 17408, P.PTQ_BF16) == "stack_per_layer"


@pytest.mark.parametrize("M", [1, 3, 8])
def test_stack_deterministic_path(P, orc, syn, M):
    # the per-layer path on request: within the bound, and bitwise the same
    # on a second run
    import torch

    H, I, Lc, eps = 1024, 2048, 3, 1e-6
    dev, host, gains = make_layers(P, orc, syn, 90 + M, Lc, H, I)
    x = syn.ffn_input(90 + M, 0, M, H, "f32")
    gd = [Q.dev(g) for g in gains]
    runs = []
    for _ in range(2):
        xd = Q.dev(x.copy())
        P.ffn_stack(dev, gd, xd, eps, deterministic=True)
        torch.cuda.synchronize()
        runs.append(xd)
    assert torch.equal(runs[0], runs[1])
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, False)
    check_stack(Q.host_f64(runs[0]), ref, bound, f"deterministic stack M={M}")


def quarter_scales(bits):
    """fp16 scale patterns divided by 4 (exact for normal values)."""
    return (bits.view(np.float16) / np.float16(4)).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("Lc", [24, 25, 26])
def test_stack_decode_spans_launches(P, orc, syn, Lc):
    # 24 layers fill one persistent launch exactly; 25 and 26 run as two
    # launches (24 + 1, 24 + 2), the second starting on the buffers the first
    # zeroed.  Quarter scales keep each block's increment small against the
    # stream, so the bound stays tight enough that a dropped or repeated layer
    # fails it.
    import torch

    H, I, eps = 1024, 2048, 1e-6
    dev, host, gains = [], [], []
    for l in range(Lc):
        F = syn.ffn_layer(70, l, H, I)
        sg, sd = quarter_scales(F.wgu_scales), quarter_scales(F.wd_scales)
        dev.append((Q.dev(P.pack(F.wgu_trits)), Q.dev(sg), Q.dev(P.pack(F.wd_trits)), Q.dev(sd),
                    Q.dev(F.signs_in), Q.dev(F.signs_mid)))
        host.append((orc.pack(F.wgu_trits), sg, orc.pack(F.wd_trits), sd, F.signs_in, F.signs_mid))
        gains.append(syn.norm_gain(70, l, H))
    x = syn.ffn_input(70, 0, 1, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.float32)
    P.device_check()
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, False)
    check_stack(got, ref, bound, f"stack decode L={Lc}")
    # the bound is far below one layer's increment
    one = orc.ffn_stack(host[-1:], [gains[-1].astype(np.float64)], ref, eps) - ref
    assert bound.max() < 0.2 * np.abs(one).max()


def test_stack_persistent_in_a_graph(P, orc, syn):
    # the bench replays the persistent launches from a CUDA graph: capture two
    # calls of three layers (one cooperative launch each, with the memsets
    # before it), replay them, and compare with the oracle's six layers
    import torch

    H, I, Lc, eps = 1024, 2048, 3, 1e-6
    dev, host, gains = make_layers(P, orc, syn, 44, Lc, H, I)
    x = syn.ffn_input(44, 0, 1, H, "f32")
    xd = Q.dev(x.copy())
    gd = [Q.dev(g) for g in gains]
    ws = torch.empty(P.ffn_stack_workspace_bytes(1, H, I, P.PTQ_F32), dtype=torch.uint8,
                     device="cuda")
    P.ffn_stack(dev, gd, xd, eps, workspace=ws)  # warm-up outside the capture
    torch.cuda.synchronize()
    xd.copy_(Q.dev(x.copy()))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            P.ffn_stack(dev, gd, xd, eps, workspace=ws)
            P.ffn_stack(dev, gd, xd, eps, workspace=ws)
    torch.cuda.synchronize()
    xd.copy_(Q.dev(x.copy()))  # the capture did not run the kernels
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    P.device_check()
    got = Q.host_f64(xd)
    ref, bound = oracle_with_bound(orc, host + host, gains + gains, x.astype(np.float64), eps,
                                   False)
    check_stack(got, ref, bound, "persistent stack replayed from a graph")


@pytest.mark.parametrize("M,act", [(1, "f32"), (4, "f32"), (3, "bf16")])
def test_stack_writes_stay_in_bounds(P, orc, syn, M, act):
    # the residual and the workspace sit between guard bands of a known byte
    # pattern; after the call (persistent for fp32, per layer for bf16) the
    # guards are untouched and the result still agrees with the oracle
    import torch

    H, I, Lc, eps, guard = 1024, 2048, 2, 1e-6, 4096
    dev, host, gains = make_layers(P, orc, syn, 46, Lc, H, I)
    x = syn.ffn_input(46, 0, M, H, "f32")
    xbuf = torch.full((M * H + 2 * guard,), float("nan"), device="cuda")
    xd = xbuf[guard:guard + M * H].view(M, H)
    xd.copy_(Q.dev(x.copy()))
    pdt = P.PTQ_F32 if act == "f32" else P.PTQ_BF16
    need = P.ffn_stack_workspace_bytes(M, H, I, pdt)
    wbuf = torch.full((need + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = wbuf[guard:guard + need]
    P.ffn_stack(dev, [Q.dev(g) for g in gains], xd, eps,
                act=torch.float32 if act == "f32" else torch.bfloat16, workspace=ws)
    torch.cuda.synchronize()
    P.device_check()
    assert torch.isnan(xbuf[:guard]).all() and torch.isnan(xbuf[-guard:]).all()
    assert (wbuf[:guard] == 0xA5).all() and (wbuf[-guard:] == 0xA5).all()
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, act == "bf16")
    check_stack(Q.host_f64(xd), ref, bound, f"stack between guard bands M={M}")


def test_stack_one_layer_is_residual_plus_block(P, orc, syn):
    # with one layer the stack is x + ffn(rmsnorm(x) g): compare the increment
    # with the single-block tolerance directly
    import torch

    H, I, eps = 1024, 2048, 1e-5
    dev, host, gains = make_layers(P, orc, syn, 40, 1, H, I)
    x = syn.ffn_input(40, 0, 2, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.float32)
    x64 = x.astype(np.float64)
    ref = orc.ffn_stack(host, [g.astype(np.float64) for g in gains], x64, eps)
    Q.check_f32(got - x64, ref - x64, "stack L=1 increment")


def test_stack_eps_dominates_a_tiny_row(P, orc, syn):
    # a row of mean square 1e-8 with eps = 1e-2: the norm is x / sqrt(eps)
    # to within 1e-6, so eps must reach the kernel as given
    import torch

    H, I, eps = 1024, 2048, 1e-2
    dev, host, gains = make_layers(P, orc, syn, 41, 2, H, I)
    x = (1e-4 * syn.ffn_input(41, 0, 1, H, "f32")).astype(np.float32)
    got = run_stack(P, dev, gains, x, eps, torch.float32)
    ref, bound = oracle_with_bound(orc, host, gains, x.astype(np.float64), eps, False)
    check_stack(got, ref, bound, "stack eps-dominated row")


def test_stack_refused_layer_leaves_x_alone(P, syn):
    import torch

    H, I = 1024, 2048
    F = syn.ffn_layer(42, 0, H, I)
    lay = (Q.dev(P.pack(F.wgu_trits)), Q.dev(F.wgu_scales), Q.dev(P.pack(F.wd_trits)),
           Q.dev(F.wd_scales), Q.dev(F.signs_in), Q.dev(F.signs_mid))
    g = Q.dev(syn.norm_gain(42, 0, H))
    x = Q.dev(syn.ffn_input(42, 0, 2, H, "f32"))
    x0 = x.clone()
    short = (lay[0], lay[1], lay[2], lay[3][:-8], lay[4], lay[5])  # fine for the ABI ...
    bad = (lay[0], lay[1], lay[2], lay[3], lay[4], lay[5][1:])     # ... misaligned signs are not
    with pytest.raises(P.PTQError, match="ALIGN"):
        P.ffn_stack([lay, short, bad], [g, g, g], x, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(x, x0)


def assert_bound_discriminates(orc, host, gains, x64, eps, ref, bound, drop):
    """The bound must be able to fail: far below one layer's increment, and
    exceeded somewhere by the oracle's own stack with layer `drop` left out
    (the mistake a chained kernel that skipped or repeated a layer would
    make)."""
    g64 = [g.astype(np.float64) for g in gains]
    one = orc.ffn_stack(host[-1:], g64[-1:], ref, eps) - ref
    assert bound.max() < 0.2 * np.abs(one).max(), (bound.max(), np.abs(one).max())
    dropped = orc.ffn_stack(host[:drop] + host[drop + 1:], g64[:drop] + g64[drop + 1:], x64, eps)
    assert (np.abs(dropped - ref) > bound).any(), "a dropped layer would pass this bound"


def quarter_scale_layers(P, orc, syn, seed, Lc, H, I):
    """As make_layers, with every block scale divided by 4: each block's
    increment stays small against the residual stream, so the chained bound
    (1 + 2 rho)^(L-1) stays tight enough to catch a dropped or repeated layer."""
    dev, host, gains = [], [], []
    for l in range(Lc):
        F = syn.ffn_layer(seed, l, H, I)
        sg, sd = quarter_scales(F.wgu_scales), quarter_scales(F.wd_scales)
        gq, dq = P.pack(F.wgu_trits), P.pack(F.wd_trits)
        dev.append((Q.dev(gq), Q.dev(sg), Q.dev(dq), Q.dev(sd), Q.dev(F.signs_in),
                    Q.dev(F.signs_mid)))
        host.append((orc.pack(F.wgu_trits), sg, orc.pack(F.wd_trits), sd, F.signs_in,
                     F.signs_mid))
        del F
        gains.append(syn.norm_gain(seed, l, H))
    return dev, host, gains


def test_stack_decode_full_size_ring(P, orc, syn):
    # the bench's decode shape: H = 5120, I = 17408, M = 1, fp32, over the 8
    # distinct layers the 64-layer step cycles through.  At the workload's
    # own scales one layer multiplies rms(x) by about 1.8, and the chained
    # bound grows to 25 times the last layer's increment -- a dropped layer
    # would pass; with quarter scales the bound is 1e-3 of an increment and a
    # dropped layer exceeds it about 1500-fold.
    import torch

    H, I, Lc, eps = 5120, 17408, 8, 1e-6
    dev, host, gains = quarter_scale_layers(P, orc, syn, 4, Lc, H, I)
    x = syn.ffn_input(4, 0, 1, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.float32)
    P.device_check()
    x64 = x.astype(np.float64)
    ref, bound = oracle_with_bound(orc, host, gains, x64, eps, False)
    check_stack(got, ref, bound, "stack decode H=5120 I=17408 L=8")
    assert_bound_discriminates(orc, host, gains, x64, eps, ref, bound, drop=3)


def test_stack_prefill_full_size_sampled_tokens(P, orc, syn):
    # the bench's prefill shape (M = 256, bf16 activations) over two layers;
    # rows are independent in the stack, so the oracle runs sampled tokens.
    # Two layers keep the bound at 0.05 of the last increment, and the stack
    # without its first layer exceeds it about 40-fold.
    import torch

    H, I, Lc, eps, M = 5120, 17408, 2, 1e-6, 256
    dev, host, gains = make_layers(P, orc, syn, 4, Lc, H, I)
    x = syn.ffn_input(4, 1, M, H, "f32")
    got = run_stack(P, dev, gains, x, eps, torch.bfloat16)
    tokens = [0, 1, 128, 255]
    x64 = x[tokens].astype(np.float64)
    ref, bound = oracle_with_bound(orc, host, gains, x64, eps, True)
    check_stack(got[tokens], ref, bound, "stack prefill M=256 sampled tokens")
    assert_bound_discriminates(orc, host, gains, x64, eps, ref, bound, drop=0)
