"""Benchmark of the PTQ1_0 hot path on one GB300 (or N independent replicas).

Headline workload (decode gate/up): M=1, K=5120, N=17408 PTQ1_0 weights
(19,496,960 bytes).  One step = rotate the activation (5 signed 1024-blocks)
+ decode GEMV.  Metric: weight bytes per second.  Line items beside it: the
decode at 4 tokens (the same shape) and at 8 tokens (K=17408, N=5120); the
prefill GEMM (M=512, K=5120, N=17408, bf16) in TFLOP/s, with M=128 and
M=2048.

Inputs are resident in HBM before the timed region.  Every step uses the next
of R distinct weight sets (R * 19.5 MB > the 129 MB L2), so no step finds its
weights in L2.  Steps are captured in CUDA graphs and timed with CUDA events
on the launching stream; the dominant kernel is also timed on its own.

--impl reference times the CPU oracle (fp64 C, all host cores) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

N_ROWS, K_COLS = 17408, 5120
WEIGHT_BYTES = N_ROWS * (K_COLS // 128) * 28          # 19,496,960
PREFILL_M = 512
METRIC = "PTQ1_0 GEMV weight GB/s (% HBM peak) at M=1; prefill GEMM TFLOP/s"
L2_BYTES = 129 * 2 ** 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---- our arm -------------------------------------------------------------------

def make_ring(P, torch, syn, R, M, N, K, dtype):
    """R distinct weight sets (packed once on the host, copied to HBM)."""
    import ternary_weight_ptq1_gb300  # noqa: F401

    ring = []
    for r in range(R):
        t, s = syn.weights(1000 + r, N, K)
        wq = torch.from_numpy(P.pack(t)).cuda()
        sc = torch.from_numpy(s.view(np.int16)).cuda()
        if dtype == "f32":
            x = torch.from_numpy(syn.normal_f32(1000 + r, 2, (M, K))).cuda()
        else:
            x = torch.from_numpy(syn.normal_bf16(1000 + r, 2, (M, K)).view(np.int16)).cuda().view(
                torch.bfloat16)
        ring.append((wq, sc, x))
    return ring


def capture(torch, fn, n_steps, start):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_steps):
            fn(start + i)
    return g


def timed_steps(torch, fn, K, W, chunk=500):
    """W warm-up steps, then exactly K steps in CUDA graphs of <= chunk steps.
    Returns (elapsed ms, graphs)."""
    for i in range(W):
        fn(i)
    torch.cuda.synchronize()
    full, rem = divmod(K, chunk)
    g_full = capture(torch, fn, min(chunk, K), 0) if full else None
    g_rem = capture(torch, fn, rem, full * chunk) if rem else None
    # one untimed replay so the graphs are uploaded
    if g_full:
        g_full.replay()
    if g_rem:
        g_rem.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(full):
        g_full.replay()
    if g_rem:
        g_rem.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


_dist = None


def barrier():
    if _dist is not None:
        _dist.barrier()


def max_over_ranks(v: float) -> float:
    if _dist is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64)
    _dist.all_reduce(t, op=_dist.ReduceOp.MAX)
    return float(t.item())


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel, from the ncu capture of the matching `bench.py --profile`
# case; None when the kernel has changed since those counters were taken.
# Prefill: the capture is this exact launch (M=512, N=17408, K=5120).
TRAFFIC_PREFILL = 24_838_144 + 2_816
# Decode: the capture of the bench's own call (`--profile gemv1`).
TRAFFIC_DECODE = 19_558_400 + 0


def ffn_lines(P, torch, syn, pk, world, args):
    """The feed-forward block (rotate, fused gate+up, SwiGLU, rotate, down),
    H=5120, I=17408, 64 layers per step: decode (M=1, fp32) and prefill
    (M=256, bf16); then the same 64 blocks chained as a pre-norm residual
    stack (RMSNorm and residual add between blocks).  The 64 layers cycle
    through 8 distinct seeded layers (470 MB of weights, more than the L2), so
    every layer streams its weights from HBM as 64 distinct layers would."""
    H, I, LAYERS, RING = 5120, 17408, 64, 8
    layers = []
    for l in range(RING):
        L = syn.ffn_layer(4, l, H, I)
        layers.append(tuple(torch.from_numpy(a).cuda() for a in (
            P.pack(L.wgu_trits), L.wgu_scales.view(np.int16), P.pack(L.wd_trits),
            L.wd_scales.view(np.int16), L.signs_in, L.signs_mid)))
    wbytes = LAYERS * 3 * H * I * 7 // 32                 # 3,743,416,320 B per token-step
    out = {}
    for name, M, dt, pdt in (("decode", 1, torch.float32, P.PTQ_F32),
                             ("prefill", 256, torch.bfloat16, P.PTQ_BF16)):
        xa = syn.ffn_input(4, 0, M, H, "f32" if M == 1 else "bf16")
        x = torch.from_numpy(xa if M == 1 else xa.view(np.int16)).cuda()
        if dt == torch.bfloat16:
            x = x.view(torch.bfloat16)
        y = torch.empty((M, H), device="cuda", dtype=dt)
        ws = torch.empty(P.ffn_workspace_bytes(M, H, I, pdt), dtype=torch.uint8, device="cuda")

        def step(i, x=x, y=y, ws=ws):  # one token-step: all 64 layers
            for l in range(LAYERS):
                P.ffn(*layers[l % RING], x, out=y, workspace=ws)

        K = max(3, min(args.steps, 40 if M == 1 else 8))
        ms = timed_steps(torch, step, K, 3, chunk=2) / K
        line = {"workload": f"feed-forward block x {LAYERS} layers, M={M}", "M": M, "H": H, "I": I,
                "dtype": "f32" if M == 1 else "bf16 in/out, fp16 rotated operands",
                "ms_per_step": round(ms, 4), "weight_bytes_per_step": wbytes,
                "weight_GB/s": round(world * wbytes / (ms * 1e-3) / 1e9, 1)}
        if M == 1:
            line["tokens_per_s"] = round(world * 1e3 / ms, 1)
        else:
            tf = 2.0 * M * LAYERS * 3 * H * I / (ms * 1e-3) / 1e12
            line["TFLOP/s"] = round(world * tf, 1)
            line["frac_of_bf16_peak"] = round(tf / pk["bf16"], 4)
        out[name] = line
    # the chained stack: the same 64 blocks, each preceded by the residual add
    # and RMSNorm kernel, over an fp32 residual stream updated in place
    gains = [torch.from_numpy(syn.norm_gain(4, l, H)).cuda() for l in range(RING)]
    # M = 4 decode tokens: the persistent kernel, and beside it the
    # bitwise-reproducible per-layer path the caller can ask for instead
    for name, M, act, det in (("stack_decode", 1, torch.float32, False),
                              ("stack_decode_m4", 4, torch.float32, False),
                              ("stack_decode_m4_per_layer", 4, torch.float32, True),
                              ("stack_prefill", 256, torch.bfloat16, False)):
        xs = torch.from_numpy(syn.ffn_input(4, 0, M, H, "f32")).cuda()
        pdt = P.PTQ_F32 if act == torch.float32 else P.PTQ_BF16
        ws = torch.empty(P.ffn_stack_workspace_bytes(M, H, I, pdt), dtype=torch.uint8, device="cuda")
        lays = [layers[l % RING] for l in range(LAYERS)]
        gs = [gains[l % RING] for l in range(LAYERS)]

        def step(i, xs=xs, ws=ws, act=act, lays=lays, gs=gs, det=det):
            P.ffn_stack(lays, gs, xs, 1e-6, act=act, workspace=ws, deterministic=det)

        K = max(3, min(args.steps, 40 if M <= 4 else 8))
        ms = timed_steps(torch, step, K, 3, chunk=2) / K
        line = {"workload": f"pre-norm residual stack of {LAYERS} feed-forward blocks, M={M}",
                "M": M, "H": H, "I": I, "dtype": "f32 residual stream, "
                + ("f32 activations" if act == torch.float32 else "bf16 activations"),
                "path": P.ffn_stack_route(M, H, I, pdt) if not det else "stack_per_layer",
                "ms_per_step": round(ms, 4),
                "weight_GB/s": round(world * wbytes / (ms * 1e-3) / 1e9, 1)}
        if M in (1, 256):
            base = out["decode" if M == 1 else "prefill"]["ms_per_step"]
            line["norm_and_residual_ms"] = round(ms - base, 4)
        if act == torch.float32:
            line["tokens_per_s"] = round(world * M * 1e3 / ms, 1)
        else:
            line["TFLOP/s"] = round(world * 2.0 * M * LAYERS * 3 * H * I / (ms * 1e-3) / 1e12, 1)
        out[name] = line
    return out


def fwht_lines(P, torch, syn, pk, world, args):
    """The stand-alone signed rotation (ptq_fwht) where it is bandwidth-bound:
    the prefill activations (M=2048 x K=5120, bf16 in and out) and the
    feed-forward prefill's intermediate (M=256 x I=17408, fp32 in and out;
    inside ptq_ffn the same kernel writes fp16).  Each step rotates the next
    of 8 distinct inputs into its own output (336 MB and 285 MB in all, more
    than the L2).  Algorithmic bytes: the input and the output once each,
    plus the K sign bytes."""
    out = {}
    R = 8
    for name, M, K, dt in (("prefill_x_bf16", 2048, 5120, torch.bfloat16),
                           ("ffn_prefill_h_f32", 256, 17408, torch.float32)):
        sg = torch.from_numpy(syn.signs(11, 3, K)).cuda()
        if dt == torch.bfloat16:
            xs = [torch.from_numpy(syn.normal_bf16(1100 + r, 2, (M, K)).view(np.int16)).cuda()
                  .view(torch.bfloat16) for r in range(R)]
        else:
            xs = [torch.from_numpy(syn.normal_f32(1100 + r, 2, (M, K))).cuda() for r in range(R)]
        ys = [torch.empty_like(xs[0]) for _ in range(R)]
        esz = 2 if dt == torch.bfloat16 else 4
        nbytes = 2 * M * K * esz + K
        Kf = max(3, min(args.steps, 400))
        us = timed_steps(torch, lambda i: P.fwht(xs[i % R], sg, out=ys[i % R]), Kf, 3,
                         chunk=100) / Kf * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"workload": f"signed FWHT-1024, M={M}, K={K}, "
                                 f"{'bf16' if esz == 2 else 'f32'} in and out",
                     "us_per_call": round(us, 3), "bytes_per_call": nbytes,
                     "GB/s": round(world * gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
                     "kernel": "fwht1024_kernel"}
        del xs, ys
    return out


def embed_lines(P, torch, syn, pk, world, args):
    """The token-embedding lookup on a rotated table (gather + inverse signed
    rotation), V=131,072 x H=5,120: one token (decode) and 2,048 (prefill),
    from a PTQ1_0 table (147 MB) and a bf16 one (1.34 GB); ids change every
    step (a ring of 16 seeded id sets)."""
    V, H, RING = 131072, 5120, 16
    s = torch.from_numpy(syn.signs(9, 2, H)).cuda()
    t, sc = syn.weights(9, V, H)
    tabs = {"ptq1": (torch.from_numpy(P.pack(t)).cuda(), torch.from_numpy(sc.view(np.int16)).cuda())}
    del t
    tabs["bf16"] = torch.from_numpy(syn.normal_bf16(9, 8, (V, H)).view(np.int16)).cuda().view(
        torch.bfloat16)
    out = {}
    for name, M in (("decode", 1), ("prefill", 2048)):
        ids = [torch.from_numpy(syn.token_ids(9, 100 + r, M, V)).cuda() for r in range(RING)]
        for kind in ("ptq1", "bf16"):
            y = torch.empty((M, H), device="cuda",
                            dtype=torch.float32 if kind == "ptq1" else torch.bfloat16)
            if kind == "ptq1":
                wq, scd = tabs["ptq1"]
                fn = lambda i, y=y: P.embed_ptq1(wq, scd, ids[i % RING], s, out=y)  # noqa: E731
                nbytes = M * (H // 128 * 28 + H * 4) + M * 4 + H
            else:
                tb = tabs["bf16"]
                fn = lambda i, y=y: P.embed(tb, ids[i % RING], s, out=y)  # noqa: E731
                nbytes = M * H * 2 * 2 + M * 4 + H
            K = max(3, min(args.steps, 2000 if M == 1 else 200))
            us = timed_steps(torch, fn, K, 3) / K * 1e3
            gbs = nbytes / (us * 1e-6) / 1e9
            out[f"{name}_{kind}"] = {
                "workload": f"embedding lookup + inverse rotation, {kind} table {V} x {H}, M={M}",
                "us_per_call": round(us, 3), "bytes_per_call": nbytes,
                "GB/s": round(world * gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
                "out_dtype": "f32" if kind == "ptq1" else "bf16"}
    return out


def plan_text(plan, gemv):
    """The decode launch ptq_gemv_plan reports, in words."""
    if plan["cluster"]:
        return (f"{gemv}: {plan['ctas']} CTAs in clusters of {plan['cluster']} (one per K-chunk), "
                "row sums added in distributed shared memory; no second kernel")
    return f"{gemv} ({plan['ctas']} CTAs) + gemv_lut_reduce_kernel"


def pq2_lines(P, torch, syn, pk, world, args):
    """The same hot path over PQ2_0 weights (2 bits a weight + a 16-bit scale
    per 128: 34 bytes a block): the decode GEMV at the gate/up shape (M=1,
    K=5120, N=17408; x already rotated; a ring of 16 weight sets, 357 MB > L2)
    and the prefill GEMM at M=512."""
    N, K = N_ROWS, K_COLS
    wbytes = N * K // 128 * 34
    R = 16
    ring = []
    for r in range(R):
        t, s = syn.weights(2000 + r, N, K)
        ring.append((torch.from_numpy(P.pq2_pack(t)).cuda(), torch.from_numpy(s.view(np.int16)).cuda()))
    x = torch.from_numpy(syn.normal_f32(2000, 2, (1, K))).cuda()
    ys = [torch.empty((1, N), device="cuda") for _ in range(R)]
    ws = torch.empty(P.matmul_pq2_workspace_bytes(1, N, K, P.PTQ_F32), dtype=torch.uint8,
                     device="cuda")
    K1 = max(3, min(args.steps, 2000))
    us = timed_steps(torch, lambda i: P.matmul_pq2(ring[i % R][0], ring[i % R][1], x, out=ys[i % R],
                                                    workspace=ws), K1, 3) / K1 * 1e3
    gbs = (wbytes + 4 * K + 4 * N) / (us * 1e-6) / 1e9
    plan = P.gemv_plan(1, N, K, pq2=True)
    dec = {"workload": "PQ2_0 decode GEMV, M=1, K=5120, N=17408 (x rotated)", "us_per_call": round(us, 3),
           "weight_bytes": wbytes, "GB/s": round(world * gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
           "kernels": plan_text(plan, "gemv_lut_tma_kernel<PQ2_0>")}
    M = PREFILL_M
    xb = torch.from_numpy(syn.normal_bf16(2000, 2, (M, K)).view(np.int16)).cuda().view(torch.bfloat16)
    yb = [torch.empty((M, N), device="cuda", dtype=torch.bfloat16) for _ in range(8)]
    K2 = max(3, min(args.steps, 200))
    ms = timed_steps(torch, lambda i: P.matmul_pq2(ring[i % 8][0], ring[i % 8][1], xb, out=yb[i % 8]),
                     K2, 3, chunk=50) / K2
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    pre = {"workload": "PQ2_0 prefill GEMM, M=512, K=5120, N=17408, bf16", "us_per_call": round(ms * 1e3, 2),
           "TFLOP/s": round(world * tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
    return {"decode": dec, "prefill": pre}


def run_ours(args, world, rank):
    import torch

    import synth as syn
    import ternary_weight_ptq1_gb300 as P

    P.load()
    pk = peaks()
    dev_index = torch.cuda.current_device()
    R = max(8, int(np.ceil(4 * L2_BYTES / WEIGHT_BYTES)))       # 28 sets, 546 MB
    ring = make_ring(P, torch, syn, R, 1, N_ROWS, K_COLS, "f32")
    signs = torch.from_numpy(syn.signs(1, 3, K_COLS)).cuda()
    xr = [torch.empty((1, K_COLS), device="cuda") for _ in range(R)]
    ys = [torch.empty((1, N_ROWS), device="cuda") for _ in range(R)]
    # one scratch for every call: they are ordered on one stream
    ws = torch.empty(max(1, P.rotate_matmul_workspace_bytes(1, N_ROWS, K_COLS, P.PTQ_F32)),
                     dtype=torch.uint8, device="cuda")

    def step(i):  # rotation fused into the table-lookup GEMV
        wq, sc, x = ring[i % R]
        P.rotate_matmul(wq, sc, x, signs, out=ys[i % R], workspace=ws)

    def gemv_only(i):
        wq, sc, _ = ring[i % R]
        P.matmul(wq, sc, xr[i % R], out=ys[i % R], workspace=ws)

    def fwht_only(i):
        P.fwht(ring[i % R][2], signs, out=xr[i % R])

    def peel_only(i):  # the pages' decode design: the trits peeled on the float pipe
        wq, sc, _ = ring[i % R]
        P.matmul_f32_peel(wq, sc, xr[i % R], out=ys[i % R])

    K, W = args.steps, args.warmup
    with ClockSampler(dev_index) as clk:
        ms = max_over_ranks(timed_steps(torch, step, K, W))
        ms_gemv = timed_steps(torch, gemv_only, K, W)
        ms_fwht = timed_steps(torch, fwht_only, K, W)
        ms_peel = timed_steps(torch, peel_only, K, W)
    P.device_check()
    ms_per_step = ms / K
    value = world * WEIGHT_BYTES / (ms_per_step * 1e-3) / 1e9       # GB/s, all ranks
    gemv_bytes = WEIGHT_BYTES + K_COLS * 4 + N_ROWS * 4
    plan1 = P.gemv_plan(1, N_ROWS, K_COLS)
    gemv_us = ms_gemv / K * 1e3
    step_us = ms_per_step * 1e3
    achieved = gemv_bytes / (step_us * 1e-6) / 1e9

    # e2e through the public API on host buffers: ptq_rotate_matmul_host moves
    # the pinned host x in and y out around the fused rotation + GEMV
    xh = torch.from_numpy(syn.normal_f32(77, 2, (1, K_COLS))).pin_memory()
    yhs = [torch.empty((1, N_ROWS)).pin_memory() for _ in range(4)]
    wsh = torch.empty(P.rotate_matmul_host_workspace_bytes(1, N_ROWS, K_COLS, P.PTQ_F32),
                      dtype=torch.uint8, device="cuda")
    E = max(50, min(K, 2000))
    for i in range(5):
        P.rotate_matmul_host(ring[0][0], ring[0][1], xh, signs, yhs[0], wsh)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for i in range(E):
        wq, sc, _ = ring[i % R]
        P.rotate_matmul_host(wq, sc, xh, signs, yhs[i % 4], wsh)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1)) / E
    e2e = world * WEIGHT_BYTES / (ms_e2e * 1e-3) / 1e9

    # the other decode sizes of the workload, rotation fused, in CUDA graphs:
    # 4 tokens on the gate/up shape (this ring's weights) and 8 tokens on the
    # down shape (K = 17408, N = 5120, a ring of its own, 156 MB)
    dec = {}
    if not args.skip_decode_m:
        for Mo, No, Ko in ((4, N_ROWS, K_COLS), (8, K_COLS, N_ROWS)):
            dring = ring if No == N_ROWS else make_ring(P, torch, syn, 8, 1, No, Ko, "f32")
            Rd = len(dring)
            dxs = [torch.from_numpy(syn.normal_f32(2000 + r, 5, (Mo, Ko))).cuda() for r in range(8)]
            dys = [torch.empty((Mo, No), device="cuda") for _ in range(8)]
            dsg = torch.from_numpy(syn.signs(1, 3, Ko)).cuda()
            dws = torch.empty(max(1, P.rotate_matmul_workspace_bytes(Mo, No, Ko, P.PTQ_F32)),
                              dtype=torch.uint8, device="cuda")

            def dstep(i, dring=dring, Rd=Rd, dxs=dxs, dys=dys, dsg=dsg, dws=dws):
                wq, sc, _ = dring[i % Rd]
                P.rotate_matmul(wq, sc, dxs[i % 8], dsg, out=dys[i % 8], workspace=dws)

            dK = max(3, min(K, 200))
            dms = timed_steps(torch, dstep, dK, 3, chunk=100) / dK
            wb = No * Ko * 7 / 32
            dec[f"M{Mo}"] = {"workload": f"decode rotate+GEMV, M={Mo}, K={Ko}, N={No}, fp32",
                             "us_per_call": round(dms * 1e3, 2),
                             "weight_GB/s_per_pass": round(world * wb / (dms * 1e-3) / 1e9, 1),
                             "tokens_per_s_equiv": round(world * Mo * wb / (dms * 1e-3) / 5.906e9, 1),
                             "kernels": "one gemv_lut_tma_kernel over the M tokens + one reduction"}
            if dring is not ring:
                del dring
            del dxs, dys, dws
        P.device_check()

    # prefill GEMM line item (M=512, bf16)
    pre = None
    if not args.skip_prefill:
        pre_R = 8
        pring = make_ring(P, torch, syn, pre_R, PREFILL_M, N_ROWS, K_COLS, "bf16")
        pys = [torch.empty((PREFILL_M, N_ROWS), device="cuda", dtype=torch.bfloat16)
               for _ in range(pre_R)]

        def pstep(i):
            wq, sc, x = pring[i % pre_R]
            P.matmul(wq, sc, x, out=pys[i % pre_R])

        pK = max(3, min(K, 200))
        pms = timed_steps(torch, pstep, pK, max(3, min(W, 10)), chunk=50) / pK
        flops = 2.0 * PREFILL_M * N_ROWS * K_COLS
        tf = flops / (pms * 1e-3) / 1e12
        pre = {"value": round(world * tf, 2), "unit": "TFLOP/s", "ms_per_step": round(pms, 4),
               "config": {"workload": "prefill GEMM", "M": PREFILL_M, "K": K_COLS, "N": N_ROWS,
                          "dtype": "bf16 in, fp32 accumulate, bf16 out",
                          "l2": f"ring of {pre_R} weight/activation sets"},
               "kernel": P.route(PREFILL_M, P.PTQ_BF16),
               "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16"],
                            "unit": "TFLOP/s", "frac": round(tf / pk["bf16"], 4),
                            "traffic": TRAFFIC_PREFILL, "peak_source": pk["source"] + " burst bf16"}}
        # the other two prefill sizes of the workload, on the same weight ring
        # with activations of their own
        pre["other_M"] = {}
        for Mo in (128, 2048):
            oxs = [torch.from_numpy(syn.normal_bf16(1000 + r, 4, (Mo, K_COLS)).view(np.int16)).cuda()
                   .view(torch.bfloat16) for r in range(pre_R)]
            oys = [torch.empty((Mo, N_ROWS), device="cuda", dtype=torch.bfloat16)
                   for _ in range(pre_R)]

            def ostep(i, oxs=oxs, oys=oys):
                wq, sc, _ = pring[i % pre_R]
                P.matmul(wq, sc, oxs[i % pre_R], out=oys[i % pre_R])

            oK = max(3, min(K, 100))
            oms = timed_steps(torch, ostep, oK, 3, chunk=50) / oK
            otf = 2.0 * Mo * N_ROWS * K_COLS / (oms * 1e-3) / 1e12
            pre["other_M"][str(Mo)] = {"us_per_call": round(oms * 1e3, 2),
                                       "TFLOP/s": round(world * otf, 1),
                                       "frac_of_bf16_peak": round(otf / pk["bf16"], 4)}
            del oxs, oys

    fwht = None if args.skip_fwht else fwht_lines(P, torch, syn, pk, world, args)
    ffn = None if args.skip_ffn else ffn_lines(P, torch, syn, pk, world, args)
    emb = None if args.skip_embed else embed_lines(P, torch, syn, pk, world, args)
    pq2 = None if args.skip_pq2 else pq2_lines(P, torch, syn, pk, world, args)

    cpu = cpu_baseline(args) if rank == 0 and not args.skip_cpu else None
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "decode gate/up: rotate (5 signed 1024-blocks) + PTQ1_0 GEMV, "
                               "one ptq_rotate_matmul call",
                   "M": 1, "K": K_COLS, "N": N_ROWS, "weight_bytes_per_step": WEIGHT_BYTES,
                   "l2": f"inputs larger than L2: ring of {R} distinct weight sets "
                         f"({R * WEIGHT_BYTES / 1e6:.0f} MB)",
                   "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
                   "timing": "CUDA graphs of <=500 steps, CUDA events on the launching stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4),
                     "traffic": TRAFFIC_DECODE,
                     "kernel": P.route(1, P.PTQ_F32), "kernel_us": round(step_us, 3),
                     "timed": "one ptq_rotate_matmul call: the table-lookup GEMV with the "
                              "rotation fused in (" + plan_text(plan1, "gemv_lut_tma_kernel") + ")",
                     "bytes_per_launch": gemv_bytes, "peak_source": pk["source"] + " copy bandwidth"},
        "stage_us": {"step_rotate_gemv_fused": round(step_us, 3),
                     "unfused_fwht": round(ms_fwht / K * 1e3, 3),
                     "unfused_gemv_on_rotated_x": round(gemv_us, 3)},
        "decode_peel": {"workload": "the same GEMV (rotated x, the same ring) by the SIMT kernel "
                                    "that peels the trits on the float pipe with 16-byte loads",
                        "us_per_call": round(ms_peel / K * 1e3, 3),
                        "GB/s": round(world * gemv_bytes / (ms_peel / K * 1e-3) / 1e9, 1),
                        "frac_of_hbm": round(gemv_bytes / (ms_peel / K * 1e-3) / 1e9 / pk["hbm"], 4),
                        "kernel": "gemv_ptq1_f32_kernel (ptq_matmul_f32_peel)"},
        "tokens_per_s_equiv": round(value * 1e9 / 5.906e9, 1),
        "e2e": {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": K_COLS * 4,
                "d2h_bytes_per_step": N_ROWS * 4, "ms_per_step": round(ms_e2e, 5),
                "path": "ptq_rotate_matmul_host (C ABI on host buffers) through the Python binding, "
                        "eager; the page-locked x and y are mapped into the device's address "
                        "space, so the fused rotation + GEMV reads x and writes y over the "
                        "host link (no copy engine)"},
        "gpu_launches": plan1["kernels"] * K,   # per call, as ptq_gemv_plan reports
        "clocks": clocks,
        "decode_other_M": dec or None,
        "prefill": pre,
        "fwht": fwht,
        "ffn": ffn,
        "embed": emb,
        "pq2": pq2,
        "cpu_baseline": cpu,
        "host": host_receipt() if rank == 0 else None,
    }
    if rank == 0:
        print(json.dumps(line))


# ---- the oracle arm -------------------------------------------------------------

def _oracle_step(orc, syn, reps):
    """Rotation + GEMV of the headline workload on the oracle, `reps` times on
    distinct seeds.  Returns (seconds, weight bytes processed)."""
    t0 = 0.0
    done = 0
    for r in range(reps):
        t, s = syn.weights(2000 + r, N_ROWS, K_COLS)
        wq = orc.pack(t)
        x = orc.decode_f32(syn.normal_f32(2000 + r, 2, (1, K_COLS)))
        sg = syn.signs(2000 + r, 3, K_COLS)
        a = time.perf_counter()
        xr = orc.fwht(x, sg)
        orc.matmul(wq, s, xr)
        t0 += time.perf_counter() - a
        done += WEIGHT_BYTES
    return t0, done


def cpu_baseline(args):
    import oracle as orc
    import synth as syn

    reps = max(1, args.cpu_reps)
    secs, nbytes = _oracle_step(orc, syn, reps)
    cores = orc.get_threads()
    out = {"value": round(nbytes / secs / 1e9, 3), "unit": "GB/s", "cores": cores,
           "kind": "oracle",
           "sample": f"{reps} full decode gate/up steps (rotation + 17408x5120 GEMV, fp64 C, "
                     f"OpenMP over output rows), {secs:.2f} s"}
    # the same oracle on one core, on a sample of about the same CPU time
    reps1 = max(1, reps // max(1, cores))
    orc.set_threads(1)
    try:
        secs1, nbytes1 = _oracle_step(orc, syn, reps1)
    finally:
        orc.set_threads(cores)
    out["single_thread"] = {"value": round(nbytes1 / secs1 / 1e9, 4), "unit": "GB/s",
                            "sample": f"{reps1} steps on one core, {secs1:.2f} s"}
    return out


def host_receipt():
    """Load, CPU, the GPU (name, driver, SMs) and the other processes on it,
    for the JSON line."""
    rec = {"loadavg": [round(v, 2) for v in os.getloadavg()],
           "cpus": len(os.sched_getaffinity(0))}
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    rec["cpu"] = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        r = subprocess.run(["nvidia-smi", "--query-compute-apps=pid,used_memory",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True,
                           timeout=20)
        rec["gpu_processes"] = [ln.strip() for ln in r.stdout.splitlines() if ln.strip()]
        r = subprocess.run(["nvidia-smi", "--query-gpu=name,driver_version", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
        rec["gpu"] = r.stdout.strip().splitlines()[0] if r.stdout.strip() else None
    except Exception:
        rec["gpu_processes"] = None
    try:
        import torch

        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        rec["sms"] = props.multi_processor_count
        rec["torch"] = torch.__version__
    except Exception:
        pass
    return rec


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle as orc
    import synth as syn

    K, W = args.steps, args.warmup
    per = 1  # one full rotation + GEMV per step
    # warm-up steps are bounded too
    _oracle_step(orc, syn, min(W, 3))
    steps = min(K, args.reference_max_steps)
    secs, nbytes = _oracle_step(orc, syn, steps * per)
    ms_per_step = secs * 1e3 / steps
    value = nbytes / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": min(W, 3), "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode gate/up: rotate (5 signed 1024-blocks) + PTQ1_0 GEMV, "
                               "one ptq_rotate_matmul call",
                   "M": 1, "K": K_COLS, "N": N_ROWS, "weight_bytes_per_step": WEIGHT_BYTES},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": orc.get_threads(),
                         "kind": "oracle",
                         "sample": f"{steps} full steps (of {K} requested), {secs:.2f} s"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def run_profile_case(which: str):
    """A few launches of one kernel on a small case sized for an ncu capture:
    gemv -- decode GEMV, M=1, K=5120, N=8*17408 (156 MB of weights > L2);
    gemv1 -- the bench's decode call itself, M=1, K=5120, N=17408 (ncu
    flushes the caches before each pass, so its DRAM counters are cold, as
    in the bench's ring of weight sets);
    gemm -- prefill GEMM, M=512, K=5120, N=17408, bf16 (gemm128: M=128);
    stack -- the persistent decode stack, 4 layers of H=5120, I=17408, one
    token (stack4: four tokens);
    fwht -- the stand-alone rotation, M=16384 x K=5120, bf16 in and out.
    Prints the event time of the last call (not a bench number)."""
    import torch

    import synth as syn
    import ternary_weight_ptq1_gb300 as P

    if which == "fwht":
        # the stand-alone rotation of bf16 prefill activations, M=16384 x
        # K=5120 (168 MB in and 168 MB out, more than the L2)
        M, K = 16384, K_COLS
        x = torch.from_numpy(syn.normal_bf16(11, 2, (M, K)).view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty_like(x)
        sg = torch.from_numpy(syn.signs(11, 3, K)).cuda()
        call = lambda: P.fwht(x, sg, out=y)  # noqa: E731
        N = 0
    elif which in ("stack", "stack4"):
        # the persistent decode stack over 4 layers (234 MB of weights > L2),
        # H=5120, I=17408: one cooperative launch
        H, I, T = 5120, 17408, 1 if which == "stack" else 4
        lays, gains = [], []
        for l in range(4):
            F = syn.ffn_layer(4, l, H, I)
            lays.append(tuple(torch.from_numpy(a).cuda() for a in (
                P.pack(F.wgu_trits), F.wgu_scales.view(np.int16), P.pack(F.wd_trits),
                F.wd_scales.view(np.int16), F.signs_in, F.signs_mid)))
            gains.append(torch.from_numpy(syn.norm_gain(4, l, H)).cuda())
        x = torch.from_numpy(syn.ffn_input(4, 0, T, H, "f32")).cuda()
        ws = torch.empty(P.ffn_stack_workspace_bytes(T, H, I, P.PTQ_F32), dtype=torch.uint8,
                         device="cuda")
        call = lambda: P.ffn_stack(lays, gains, x, 1e-6, workspace=ws)  # noqa: E731
        M, N = T, 3 * H * I // K_COLS
    elif which == "gemv":
        M, N, dt = 1, 8 * N_ROWS, "f32"
    elif which == "gemv1":
        M, N, dt = 1, N_ROWS, "f32"
    elif which == "gemm128":
        M, N, dt = 128, N_ROWS, "bf16"
    else:
        M, N, dt = PREFILL_M, N_ROWS, "bf16"
    if which in ("stack", "stack4", "fwht"):
        pass
    elif dt == "f32":  # the bench's decode call: rotation fused into the GEMV
        mv = syn.gaussian_matvec(7, M, N, K_COLS, dtype=dt)
        wq = torch.from_numpy(P.pack(mv.trits)).cuda()
        sc = torch.from_numpy(mv.scales.view(np.int16)).cuda()
        x = torch.from_numpy(mv.x).cuda()
        y = torch.empty((M, N), device="cuda")
        signs = torch.from_numpy(syn.signs(7, 3, K_COLS)).cuda()
        call = lambda: P.rotate_matmul(wq, sc, x, signs, out=y)
    else:
        mv = syn.gaussian_matvec(7, M, N, K_COLS, dtype=dt)
        wq = torch.from_numpy(P.pack(mv.trits)).cuda()
        sc = torch.from_numpy(mv.scales.view(np.int16)).cuda()
        x = torch.from_numpy(mv.x.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        call = lambda: P.matmul(wq, sc, x, out=y)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    call()
    e1.record()
    torch.cuda.synchronize()
    P.device_check()
    print(json.dumps({"profile_case": which, "M": M, "N": N, "K": K_COLS,
                      "last_launch_us": round(e0.elapsed_time(e1) * 1e3, 2)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-reps", type=int, default=1000)       # about 10 s of oracle work
    ap.add_argument("--reference-max-steps", type=int, default=1000)
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-decode-m", action="store_true")
    ap.add_argument("--skip-ffn", action="store_true")
    ap.add_argument("--skip-fwht", action="store_true")
    ap.add_argument("--skip-embed", action="store_true")
    ap.add_argument("--skip-pq2", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--profile", choices=["gemv", "gemv1", "gemm", "gemm128", "stack", "stack4",
                                          "fwht"],
                    help="run a small case of one kernel for an ncu capture, then exit")
    args = ap.parse_args()
    if args.profile:
        import torch

        torch.cuda.set_device(0)
        run_profile_case(args.profile)
        return
    if args.warmup < 3:
        args.warmup = 3

    global _dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
        _dist = dist
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        import torch

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        run_ours(args, world, rank)
    if _dist is not None:
        _dist.barrier()
        _dist.destroy_process_group()


if __name__ == "__main__":
    main()
