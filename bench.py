#!/usr/bin/env python3
"""Benchmark of the rotated-INT8 hot path on GB300 (one JSON line on stdout).

One step = one pass over every row of the hot path, each on its own seeded
synthetic workload (shapes and distributions of the method's configurations):
  prefill linear   x bf16 [1024,4096] (1% outlier channels x30), W8 [14336,4096], bias,
                   R = H64 (x) H64 / 64 -> y bf16          (headline: TOPS)
  linear_acc       same, int32 accumulator, then the standalone dequant epilogue
  decode GEMV      x [1,4096], W8 [4096,4096], no bias      (GB/s of the weight stream)
  SwiGLU FFN       x [1024,4096], W_gate/W_up [16384,4096], W_down [4096,16384],
                   R_d = H64 (x) H64, R_h = H128 (x) H128
  backward dx      dy [4096,16384], W8 [16384,4096]: dequant_weight, linear_dx (bf16),
                   linear_dx_int8
  rotated bf16     the page's fair comparator on the prefill shape: rotate-only kernel on x,
                   then a bf16 linear against the pre-rotated bf16 weight (+ bias); the
                   line reports the int8 layer's speedup over it
  quantize_act     x [4096,16384] rotated + quantized as H128 (x) H128 (the three-pass
                   kernel) and as H64 (x) H256 (the generic-descriptor kernel)
Inputs are resident in HBM; L2 is flushed (a 512 MB write, then a read of the
same buffer so that its dirty lines are written back too) before every timed
operation, outside its CUDA-event window.  `value` is the prefill linear's
throughput 2*M*N*K / t.  The int8 contraction runs exactly on the f16 tensor
pipe (sm_103a has no int8 MMA kind; its legacy mma.sync int8 path peaks at
158 TOPS, measured), so its roofline peak is the measured dense f16/bf16 figure.

--impl reference times the CPU oracle (the only other implementation that
exists) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "int8 linear TOPS & % INT8 peak (M≥1024); decode GEMV GB/s & % HBM peak"
PREFILL = dict(M=1024, K=4096, N=14336, rot=(64, 64, 1))
DECODE = dict(M=1, K=4096, N=4096, rot=(64, 64, 1))
FFN = dict(M=1024, d=4096, H=16384, rot_d=(64, 64, 1), rot_h=(128, 128, 1))
BWD = dict(M=4096, N=16384, K=4096, rot=(64, 64, 1))
QACT = dict(M=4096, K=16384)  # activation rotate+quantize rows: square (128 x 128) vs non-square (64 x 256)
DECODE_BYTES = 4096 * 4096 + 4096 * 4 + 4096 * 2 + 4096 * 2  # W8 + s + x + y
DEQW_BYTES = 16384 * 4096 * 3 + 16384 * 4  # int8 read + bf16 write + scales
WORKLOAD = ("prefill INT8 linear x[1024,4096] @ W8[14336,4096]^T + bias, R=H64(x)H64/64; "
            "step also runs decode GEMV [1x4096x4096], SwiGLU FFN [1024,4096,16384], "
            "backward dx [4096,16384,4096], rotated-bf16 comparator [1024,4096,14336], activation "
            "rotate+quantize [4096,16384] as H128(x)H128 and H64(x)H256")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from profiles/traffic.txt, or None when the kernel's sources
    changed since that ncu capture (the record keys the bytes on a hash of the source files)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            fields = line.split()
            if len(fields) < 4 or fields[0].startswith("#") or fields[0] != kernel:
                continue
            h = hashlib.sha256()
            for src in fields[1].split(","):
                with open(os.path.join(ROOT, src), "rb") as g:
                    h.update(g.read())
            return int(fields[3]) if h.hexdigest()[:16] == fields[2] else None
    return None


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(local_ms: float, local_units: float, world: int, group=None):
    """Max elapsed over ranks and the sum of units over ranks (replicas: weak scaling)."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (arrival time, csv line)
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The host-time window of the timed region (samples arriving in it are the ones reported)."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines, scope = [ln for _, ln in self.lines], "all samples (none arrived during the timed steps)"
        if self.window is not None:
            inside = [ln for t, ln in self.lines if self.window[0] <= t <= self.window[1] + 0.06]
            if inside:
                lines, scope = inside, "samples arriving during the timed steps"
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": scope}


# ---------------------------------------------------------------------------------------------
def run_ours(args):
    import torch

    from ffn_rotate_quantize_gb300 import inputs as I
    from ffn_rotate_quantize_gb300 import ops as G

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    G.init()
    peaks = load_peaks()
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---------------- inputs (untimed), only for the selected rows ----------------
    only = set(args.only.split(",")) if args.only else None
    want = lambda *names: only is None or any(n in only for n in names)
    M3, N3, K3 = PREFILL["M"], PREFILL["N"], PREFILL["K"]
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ops = []
    if want("linear", "linear_acc", "dequant", "linear_bf16_rotated") or not args.only:
        c3 = I.linear_case(M3, K3, N3, n_outliers=I.outlier_count(K3), outlier_scale=30.0, bias_std=0.01, seed=0)
        x3, b3 = bf(c3["x"]), bf(c3["bias"])
        w3 = bf(c3["w"])
        w83, s3 = G.prepare_weight(w3, PREFILL["rot"])
        # the rotate-only BF16 path stores the weight pre-rotated in bf16 (one-time, untimed)
        wr3 = G.rotate_bf16(w3, PREFILL["rot"]) if want("linear_bf16_rotated") else None
        del c3, w3
        ws_lin = torch.empty(G.workspace_size(G.OP_LINEAR, M3, N3, K3), dtype=torch.uint8, device=dev)
        y3 = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)
        acc3 = torch.empty((M3, N3), dtype=torch.int32, device=dev)
        xs3 = torch.empty((M3,), dtype=torch.float32, device=dev)
        y3b = torch.empty_like(y3)
        if want("linear"):
            ops.append(("linear", lambda i: G.linear(x3, w83, s3, b3, PREFILL["rot"], ws_lin, out=y3)))
        if want("linear_acc", "dequant"):
            ops.append(("linear_acc", lambda i: G.lib().gbq_linear_acc(
                G._ptr(x3), G._ptr(w83), G._ptr(acc3), N3, G._ptr(xs3), M3, N3, K3, G._rot(PREFILL["rot"]),
                G._ptr(ws_lin), ws_lin.numel(), G._stream())))
        if want("dequant"):
            ops.append(("dequant", lambda i: G.dequant(acc3, xs3, s3, b3, out=y3b)))
        if want("linear_bf16_rotated"):
            # the page's fair comparator: rotate-only kernel on x, then a bf16 linear against bf16(W R)
            xr3 = torch.empty_like(x3)
            ops.append(("linear_bf16_rotated", lambda i: (G.rotate_bf16(x3, PREFILL["rot"], out=xr3),
                                                          G.linear_bf16(xr3, wr3, b3, out=y3b))))
    if want("decode_gemv", "small_batch"):
        c2 = I.linear_case(DECODE["M"], DECODE["K"], DECODE["N"], n_outliers=I.outlier_count(DECODE["K"]),
                           outlier_scale=30.0, bias_std=None, seed=0)
        x2 = bf(c2["x"])
        w82, s2 = G.prepare_weight(bf(c2["w"]), DECODE["rot"])
        # 16 copies of the decode weight (268 MB > L2) so every decode call streams from HBM
        w82c = [w82.clone() for _ in range(16)]
        ws_dec = torch.empty(max(G.workspace_size(G.OP_LINEAR, 1, DECODE["N"], DECODE["K"]), 256),
                             dtype=torch.uint8, device=dev)
        y2 = torch.empty((1, DECODE["N"]), dtype=torch.bfloat16, device=dev)
        if want("decode_gemv"):
            ops.append(("decode_gemv", lambda i: G.linear(x2, w82c[i % len(w82c)], s2, None, DECODE["rot"],
                                                          ws_dec, out=y2)))
        # A chain of dependent decode layers (N = K): call i reads call i-1's output as its x.
        chain = [x2] + [torch.empty((1, DECODE["N"]), dtype=torch.bfloat16, device=dev) for _ in range(32)]
        decode_chain = lambda i: G.linear(chain[i % 32], w82c[i % len(w82c)], s2, None, DECODE["rot"], ws_dec,
                                          out=chain[i % 32 + 1])
    if want("ffn_fused"):
        c4 = I.ffn_case(FFN["M"], FFN["d"], FFN["H"], seed=0)
        x4 = bf(c4["x"])
        wg8, sg = G.prepare_weight(bf(c4["wg"]), FFN["rot_d"])
        wu8, su = G.prepare_weight(bf(c4["wu"]), FFN["rot_d"])
        wd8, sd = G.prepare_weight(bf(c4["wd"]), FFN["rot_h"])
        del c4
        ws_ffn = torch.empty(G.workspace_size(G.OP_FFN, FFN["M"], 0, FFN["d"], FFN["H"]), dtype=torch.uint8,
                             device=dev)
        y4 = torch.empty((FFN["M"], FFN["d"]), dtype=torch.bfloat16, device=dev)
        ops.append(("ffn_fused", lambda i: G.ffn_fused(x4, wg8, sg, wu8, su, wd8, sd, FFN["rot_d"], FFN["rot_h"],
                                                       ws_ffn, out=y4)))
    if want("dequant_weight", "linear_dx", "linear_dx_int8"):
        c5 = I.backward_case(BWD["M"], BWD["N"], BWD["K"], seed=0)
        dy5 = bf(c5["dy"])
        w85, s5 = G.prepare_weight(bf(c5["w"]), BWD["rot"])
        del c5
        what = torch.empty((BWD["N"], BWD["K"]), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((BWD["M"], BWD["K"]), dtype=torch.bfloat16, device=dev)
        dx8 = torch.empty_like(dx)
        ws_dx8 = torch.empty(G.workspace_size(G.OP_LINEAR_DX_INT8, BWD["M"], BWD["N"], BWD["K"]),
                             dtype=torch.uint8, device=dev)
        if want("dequant_weight", "linear_dx"):
            ops.append(("dequant_weight", lambda i: G.lib().gbq_dequant_weight(
                G._ptr(w85), G._ptr(s5), G._ptr(what), BWD["N"], BWD["K"], G._rot(BWD["rot"]), G._stream())))
        if want("linear_dx"):
            ops.append(("linear_dx", lambda i: G.linear_dx(dy5, what, out=dx)))
        if want("linear_dx_int8"):
            ops.append(("linear_dx_int8", lambda i: G.linear_dx_int8(dy5, w85, s5, BWD["rot"], ws_dx8, out=dx8)))
    if want("quantize_act_128x128", "quantize_act_64x256"):
        # The activation rotate+quantize of a 16384-wide row as a square descriptor (the three-pass kernel)
        # and as a non-square one of the same width (the generic-descriptor kernel).
        xq = bf(I.bf16_bits(np.random.default_rng(5).standard_normal((QACT["M"], QACT["K"]), dtype=np.float32)))
        qq = torch.empty((QACT["M"], QACT["K"]), dtype=torch.int8, device=dev)
        sq = torch.empty((QACT["M"],), dtype=torch.float32, device=dev)
        for name, r in (("quantize_act_128x128", (128, 128, 1)), ("quantize_act_64x256", (64, 256, 1))):
            if want(name):
                ops.append((name, lambda i, r=r: G.lib().gbq_quantize_act(
                    G._ptr(xq), G._ptr(qq), G._ptr(sq), QACT["M"], QACT["K"], G._rot(r), G._stream())))
    opfn = dict(ops)
    work = {  # algorithmic units per call
        "linear": (2.0 * M3 * N3 * K3, "TOPS"),
        "linear_acc": (2.0 * M3 * N3 * K3, "TOPS"),
        "dequant": (M3 * N3 * (4 + 2) + M3 * 4 + N3 * 6, "GB/s"),
        "decode_gemv": (float(DECODE_BYTES), "GB/s"),
        "ffn_fused": (2.0 * FFN["M"] * FFN["d"] * FFN["H"] * 3, "TOPS"),
        "dequant_weight": (float(DEQW_BYTES), "GB/s"),
        "linear_dx": (2.0 * BWD["M"] * BWD["N"] * BWD["K"], "TFLOP/s"),
        "linear_dx_int8": (2.0 * BWD["M"] * BWD["N"] * BWD["K"], "TOPS"),
        "linear_bf16_rotated": (2.0 * M3 * N3 * K3, "TFLOP/s"),
        "quantize_act_128x128": (float(QACT["M"] * QACT["K"] * 3 + QACT["M"] * 4), "GB/s"),
        "quantize_act_64x256": (float(QACT["M"] * QACT["K"] * 3 + QACT["M"] * 4), "GB/s"),
    }
    evs = {name: [] for name, _ in ops}

    def step(i, timed):
        for name, fn in ops:
            flush_l2(flush)
            if timed:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            rc = fn(i)
            if isinstance(rc, int) and rc != 0:
                G.check(rc)
            if timed:
                e1.record(stream)
                evs[name].append((e0, e1))

    for i in range(args.warmup):
        step(i, False)
    torch.cuda.synchronize()
    assert G.device_status() == 0, "a kernel reported a device-side wait timeout"
    # Launch census on one more (untimed) step: the library's own event hooks count every kernel it
    # launches, per kernel class.  The timed steps run the same calls without the hooks (events
    # between the quantizer and the GEMM would keep the GEMM from starting while the quantizer ends).
    G.prof_enable(True)
    step(args.warmup, False)
    torch.cuda.synchronize()
    prof = {k: G.prof_read(k) for k in (G.K_ROTATE, G.K_I8GEMM, G.K_BF16GEMM, G.K_GEMV, G.K_ELEMWISE)}
    G.prof_enable(False)
    launches_per_step = sum(n for n, _ in prof.values())

    # ---------------- timed region ----------------
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    h0 = time.monotonic()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(h0, time.monotonic())
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = t_start.elapsed_time(t_end) / args.steps
    launches = launches_per_step * args.steps
    assert G.device_status() == 0, "a kernel reported a device-side wait timeout"

    rows = {}
    for name, _ in ops:
        ms = float(np.median([e0.elapsed_time(e1) for e0, e1 in evs[name]]))
        units, unit = work[name]
        scale = 1e-12 if unit in ("TOPS", "TFLOP/s") else 1e-9
        val = units / (ms * 1e-3) * scale
        peak = peaks["hbm"] if unit == "GB/s" else peaks["bf16"]
        rows[name] = {"ms": round(ms, 4), "value": round(val, 2), "unit": unit, "frac_of_peak": round(val / peak, 4)}

    value, roof, dec, e2e = None, None, None, None
    if "linear" in opfn:
        total_ms, total_units = aggregate(rows["linear"]["ms"], work["linear"][0], world)
        value = total_units / (total_ms * 1e-3) * 1e-12
        # Dominant kernels, timed alone with library-owned CUDA events on their launch stream.
        # Four copies of the weight (235 MB, above the 129 MB L2) so that back-to-back launches stream
        # their weight from HBM, as the prefill layer does.
        w83c = [w83] + [w83.clone() for _ in range(3)]
        gemm_ms = kernel_ms(G, torch, flush, G.K_I8GEMM,
                            lambda i: G.linear(x3, w83c[i % 4], s3, b3, PREFILL["rot"], ws_lin, out=y3), reps=12)
        del w83c
        achieved = work["linear"][0] / (gemm_ms * 1e-3) * 1e-12
        roof = {"bound": "tensor", "kernel": "i8gemm_kernel (prefill 1024x14336x4096)",
                "achieved": round(achieved, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16"], 4), "traffic": profiled_traffic("i8gemm_kernel"),
                "ms": round(gemm_ms, 4),
                "peak_note": f"dense f16/bf16 tensor peak ({peaks['src']}, burst): the int8 contraction runs "
                             "exactly on the f16 pipe, the fastest int8 route of sm_103a (no tcgen05 int8 kind; "
                             "mma.sync s8 measured at 158 TOPS)"}
        e2e = measure_e2e(G, torch, dev, x3, w83, s3, b3, ws_lin, args)
    if "decode_gemv" in opfn:
        # gbq_linear at M = 1 is one GEMV launch: time a chain of 32 dependent decode layers (call i reads
        # call i-1's output; 16 weight copies, 268 MB) captured in a CUDA graph, one event pair per replay
        # (median of five), after checking the launch census of a call.
        G.prof_enable(True)
        opfn["decode_gemv"](0)
        torch.cuda.synchronize()
        n_gv, _ = G.prof_read(G.K_GEMV)
        n_other = sum(G.prof_read(k)[0] for k in (G.K_ROTATE, G.K_I8GEMM, G.K_BF16GEMM, G.K_ELEMWISE))
        G.prof_enable(False)
        assert n_gv == 1 and n_other == 0, "the decode call is not a single GEMV launch"
        gv_ms = batch_ms(torch, flush, decode_chain, reps=32)
        ach = DECODE_BYTES / (gv_ms * 1e-3) * 1e-9
        graph_ms = graph_batch_ms(torch, flush, decode_chain, reps=32)
        ach_g = DECODE_BYTES / (graph_ms * 1e-3) * 1e-9
        # Decode is served from CUDA graphs: the primary figure is the replay of the captured chain (host
        # launch overhead out of the timed region; device-side gaps and the per-layer dependency stay in).
        # The eager chain is reported beside it: from Python it is bound by the host's launch rate.
        dec = {"bound": "hbm", "kernel": "gemv_direct_kernel (decode 1x4096x4096)",
               "achieved": round(ach_g, 1), "peak": peaks["hbm"], "unit": "GB/s",
               "frac": round(ach_g / peaks["hbm"], 4), "ms": round(graph_ms, 4),
               "traffic": profiled_traffic("gemv_direct_kernel"),
               "mode": "CUDA-graph replay of 32 dependent decode layers (call i's x is call i-1's y; 16 weight "
                       "copies, 268 MB), one event pair per replay, median of 5 replays after L2 flushes",
               "eager": {"ms": round(gv_ms, 4), "achieved": round(ach, 1), "frac": round(ach / peaks["hbm"], 4),
                         "note": "the same chain launched from Python, one event pair (host launch rate bound)"}}

    small = None
    if want("small_batch"):
        # Few-token calls served by weight-streaming GEMVs (graph-replayed chains of dependent layers whose
        # weights together exceed L2): the SwiGLU FFN at one token (d = 4096, H = 16384; four layers with
        # their own weights, 804 MB) and the 4096 x 4096 linear at eight tokens (the 16 decode weight copies).
        gen = torch.Generator(device=dev).manual_seed(7)
        dF, HF = FFN["d"], FFN["H"]
        layers = []
        for _ in range(4):
            lw = []
            for (n_, k_, r_) in ((HF, dF, FFN["rot_d"]), (HF, dF, FFN["rot_d"]), (dF, HF, FFN["rot_h"])):
                wb = (torch.randn((n_, k_), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
                lw.extend(G.prepare_weight(wb, r_))
                del wb
            layers.append(lw)
        ws_f1 = torch.empty(G.workspace_size(G.OP_FFN, 1, 0, dF, HF), dtype=torch.uint8, device=dev)
        xf = [(torch.randn((1, dF), generator=gen, device=dev)).to(torch.bfloat16) for _ in range(9)]
        ffn1 = lambda i: G.ffn_fused(xf[i], *layers[i % 4], FFN["rot_d"], FFN["rot_h"], ws_f1, out=xf[i + 1])
        ffn_ms = graph_batch_ms(torch, flush, ffn1, reps=8)
        ffn_bytes = 3 * HF * dF + 2 * 4 * HF + 4 * dF + 2 * dF * 2
        ws_m8 = torch.empty(G.workspace_size(G.OP_LINEAR, 8, DECODE["N"], DECODE["K"]), dtype=torch.uint8,
                            device=dev)
        x8 = [(torch.randn((8, DECODE["K"]), generator=gen, device=dev)).to(torch.bfloat16) for _ in range(33)]
        lin8 = lambda i: G.linear(x8[i], w82c[i % len(w82c)], s2, None, DECODE["rot"], ws_m8, out=x8[i + 1])
        lin8_ms = graph_batch_ms(torch, flush, lin8, reps=32)
        lin8_bytes = DECODE["N"] * DECODE["K"] + 4 * DECODE["N"] + 2 * 8 * (DECODE["K"] + DECODE["N"])
        small = {
            "ffn_decode_1x4096x16384": {
                "ms": round(ffn_ms, 4), "achieved": round(ffn_bytes / (ffn_ms * 1e-3) * 1e-9, 1), "unit": "GB/s",
                "frac": round(ffn_bytes / (ffn_ms * 1e-3) * 1e-9 / peaks["hbm"], 4),
                "route": "x codes -> one gate|up GEMV over [W_gate; W_up] -> SiLU-GLU + H128(x)H128 codes -> down GEMV"},
            "linear_8x4096x4096": {
                "ms": round(lin8_ms, 4), "achieved": round(lin8_bytes / (lin8_ms * 1e-3) * 1e-9, 1),
                "unit": "GB/s", "frac": round(lin8_bytes / (lin8_ms * 1e-3) * 1e-9 / peaks["hbm"], 4),
                "route": "rotation kernel -> codes GEMV"},
            "mode": "CUDA-graph replay of dependent layers (call i's x is call i-1's y), one event pair per "
                    "replay, median of 5 replays after L2 flushes"}
        del layers

    out = {
        "metric": METRIC, "value": None if value is None else round(value, 2), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M3, "N": N3, "K": K3, "rotation": "H64(x)H64/64",
                   "l2": "step: flushed before every timed op (512 MB write, then a read of it that evicts the "
                         "dirty lines); roofline kernels: back-to-back "
                         "launches cycling inputs larger than L2 (4 prefill / 16 decode weight copies)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "decode_roofline": dec, "small_batch": small, "rows": rows, "gpu_launches": launches,
        "int8_speedup_vs_rotated_bf16": (round(rows["linear_bf16_rotated"]["ms"] / rows["linear"]["ms"], 3)
                                         if "linear_bf16_rotated" in rows and "linear" in rows else None),
        "kernel_ms_census_step": {k: round(v[1], 3) for k, v in zip(("rotate", "i8gemm", "bf16gemm", "gemv",
                                                                     "elemwise"), prof.values())},
        "e2e": e2e, "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline and not args.only:
        out["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def flush_l2(flush):
    """Write a buffer larger than L2 (512 MB), then read it back: the read evicts the write's dirty lines
    (written back outside any timed window), so the next op starts from a clean L2 holding none of its
    inputs and pays for no one else's write-back."""
    import torch
    flush.zero_()
    flush.view(torch.float32).sum()  # a float sum reads the buffer in place (no widened copy)


def batch_ms(torch, flush, fn, reps=32):
    """Average duration of fn(i) launched reps times back to back on the current stream, one CUDA
    event pair around the batch (for single-kernel ops, whose per-launch events would add gaps).
    fn(i) must cycle through inputs whose total exceeds the L2 cache."""
    fn(0)
    torch.cuda.synchronize()
    flush_l2(flush)
    st = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(reps):
        fn(i)
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def graph_batch_ms(torch, flush, fn, reps=32, samples=5):
    """batch_ms with the reps calls captured once in a CUDA graph (after an eager warm-up call) and the
    replay timed: host launch overhead leaves the timed region, device-side launch gaps stay.  The median
    of `samples` replays, each after an L2 flush."""
    fn(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fn(i)
    g.replay()  # first replay uploads the graph
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    times = []
    for _ in range(samples):
        flush_l2(flush)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    del g
    return float(np.median(times))


def kernel_ms(G, torch, flush, kind, fn, reps=10):
    """Average device duration of one library kernel class launched by fn(i), i = 0..reps-1.

    The calls run back to back on one stream (after one L2 flush), each bracketed by the
    library's own CUDA events on its launch stream, so every start event is reached with the
    kernel already queued: the pair measures the kernel, not launch gaps.  fn(i) must cycle
    through inputs whose total exceeds the L2 cache, so no call finds its operands there."""
    fn(0)  # warm-up (first-launch set-up outside the measurement)
    torch.cuda.synchronize()
    flush_l2(flush)
    G.prof_enable(True)
    for i in range(reps):
        fn(i)
    torch.cuda.synchronize()
    n, t = G.prof_read(kind)
    G.prof_enable(False)
    return t / n if n else float("nan")


def measure_e2e(G, torch, dev, x3, w83, s3, b3, ws_lin, args):
    """Prefill linear through the public API with pinned host input/output copies inside the timed region.

    The rows are independent, so the step runs as a user overlapping transfers would: four chunks of 256
    token rows (one GEMM token tile each) on three streams -- host->device copies on one, the linear layer
    on a second (chunk c waits for its copy), device->host copies on a third (chunk c waits for its linear)
    -- so every transfer after the first chunk's overlaps compute and the other direction. The result
    equals a single call's bit for bit (checked once). The copy-only floor moves the same bytes with the
    two directions concurrent and no compute."""
    M, N = PREFILL["M"], PREFILL["N"]
    chunks = 4
    xh = x3.cpu().pin_memory()
    yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x3)
    yd = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    main = torch.cuda.current_stream()
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    rows = M // chunks
    ref = G.linear(x3, w83, s3, b3, PREFILL["rot"], ws_lin).cpu()
    ev = lambda: torch.cuda.Event()

    def step():
        e_in = [ev() for _ in range(chunks)]
        e_comp = [ev() for _ in range(chunks)]
        for c in range(chunks):
            r0, r1 = c * rows, (c + 1) * rows
            with torch.cuda.stream(s_in):
                xd[r0:r1].copy_(xh[r0:r1], non_blocking=True)
                e_in[c].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(e_in[c])
                G.linear(xd[r0:r1], w83, s3, b3, PREFILL["rot"], ws_lin, out=yd[r0:r1])
                e_comp[c].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_comp[c])
                yh[r0:r1].copy_(yd[r0:r1], non_blocking=True)

    def copies_only():
        with torch.cuda.stream(s_in):
            xd.copy_(xh, non_blocking=True)
        with torch.cuda.stream(s_out):
            yh.copy_(yd, non_blocking=True)

    def timed(fn):
        times = []
        for i in range(args.warmup + args.steps):
            flush_l2(flush)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(main)
            for s in (s_in, s_comp, s_out):
                s.wait_event(e0)
            fn()
            for s in (s_in, s_comp, s_out):
                e = ev()
                e.record(s)
                main.wait_event(e)
            e1.record(main)
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(e0.elapsed_time(e1))
        return float(np.median(times))

    eager_ms = timed(step)
    assert torch.equal(yh.view(torch.int16), ref.view(torch.int16)), "chunked e2e result differs"
    # The same step captured once in a CUDA graph (every call in it is capturable) and replayed: the host's
    # enqueue rate of the ~20 copies, launches and cross-stream events per step leaves the measurement; the
    # transfers stay inside the timed region.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(main)
    with torch.cuda.graph(graph, stream=cap):
        fork = ev()
        fork.record(cap)
        for s in (s_in, s_comp, s_out):
            s.wait_event(fork)
        step()
        for s in (s_in, s_comp, s_out):
            e = ev()
            e.record(s)
            cap.wait_event(e)
    main.wait_stream(cap)
    yh.zero_()
    ms = timed(graph.replay)
    assert torch.equal(yh.view(torch.int16), ref.view(torch.int16)), "graph-replayed e2e result differs"
    copy_ms = timed(copies_only)
    units = 2.0 * M * N * PREFILL["K"]
    return {"value": round(units / (ms * 1e-3) * 1e-12, 2), "unit": "TOPS", "ms": round(ms, 4),
            "h2d_bytes_per_step": int(xh.numel() * 2), "d2h_bytes_per_step": int(yh.numel() * 2),
            "copy_only_ms": round(copy_ms, 4), "vs_copy_only": round(ms / copy_ms, 3),
            "eager_ms": round(eager_ms, 4),
            "pipeline": f"{chunks} chunks of {rows} token rows on 3 streams (copy in | linear | copy out), "
                        "captured once in a CUDA graph and replayed each step (eager_ms: launched from Python)"}


# ---------------------------------------------------------------------------------------------
def cpu_baseline(args, target_s: float = 12.0):
    """The CPU oracle, as it stands, on a bounded row sample of the prefill linear."""
    import oracle as O
    from ffn_rotate_quantize_gb300 import inputs as I
    c = I.linear_case(PREFILL["M"], PREFILL["K"], PREFILL["N"], n_outliers=I.outlier_count(PREFILL["K"]),
                      outlier_scale=30.0, bias_std=0.01, seed=0)
    rot = PREFILL["rot"]
    w8, ws = O.prepare_weight(c["w"], rot)  # one-time weight preparation, untimed
    rows = 4
    t0 = time.perf_counter()
    O.linear(c["x"][:rows], w8, ws, c["bias"], rot)
    t_small = time.perf_counter() - t0
    rows = int(min(PREFILL["M"], max(rows, rows * target_s / max(t_small, 1e-3))))
    t0 = time.perf_counter()
    O.linear(c["x"][:rows], w8, ws, c["bias"], rot)
    t = time.perf_counter() - t0
    ops = 2.0 * rows * PREFILL["N"] * PREFILL["K"]
    return {"value": round(ops / t * 1e-12, 6), "unit": "TOPS", "cores": O.num_threads(), "kind": "oracle",
            "sample": f"prefill linear on {rows} of {PREFILL['M']} rows (full N={PREFILL['N']}, K={PREFILL['K']}); "
                      f"{t:.1f} s", "seconds": round(t, 2)}


def run_reference(args):
    """The CPU oracle timed as the reference arm (rank 0 only)."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle as O
    from ffn_rotate_quantize_gb300 import inputs as I
    c = I.linear_case(PREFILL["M"], PREFILL["K"], PREFILL["N"], n_outliers=I.outlier_count(PREFILL["K"]),
                      outlier_scale=30.0, bias_std=0.01, seed=0)
    rot = PREFILL["rot"]
    w8, ws = O.prepare_weight(c["w"], rot)
    rows = 8
    times = []
    for i in range(args.warmup + args.steps):
        r0 = (i * rows) % PREFILL["M"]
        t0 = time.perf_counter()
        O.linear(c["x"][r0:r0 + rows], w8, ws, c["bias"], rot)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = float(np.median(times))
    ops = 2.0 * rows * PREFILL["N"] * PREFILL["K"]
    val = ops / t * 1e-12
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TOPS", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
           "config": {"workload": WORKLOAD, "M": PREFILL["M"], "N": PREFILL["N"], "K": PREFILL["K"],
                      "sample_rows_per_step": rows},
           "cpu_baseline": {"value": round(val, 6), "unit": "TOPS", "cores": O.num_threads(), "kind": "oracle",
                            "sample": f"prefill linear, {rows} rows per step (full N, K)"},
           "e2e": {"value": round(val, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)  # ~0.1 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", help="comma-separated rows to run (profiling); default: all")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
