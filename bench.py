#!/usr/bin/env python
"""Benchmark of the GB300 MXFP8 block-scaled linear layer.

One step = one ``mxfp8_linear`` call (BF16 activation quantization with the
8x4 scale layout + block-scaled GEMM + padded-N slice + bias) on the
decode-shaped fused-QKV workload: M=16 tokens, N=5120, K=2048, BF16 bias.
The headline metric is weight GB/s: bytes of MXFP8 weight (E4M3 data + E8M0
scales) streamed per second.  Inputs are already in HBM when the timed region
starts; the weights (and activations) rotate over enough copies that every
call reads them from HBM (copies x bytes >= 4x L2), and the K steps run as
replays of CUDA graphs of back-to-back calls.

Before the contract line, one compact JSON line per workload of the layer
(key "bench_config": tiny, decode M=1/16, mid, mid N=130, prefill 8192^3 with
8x4 and 128x4 activation scales, grouped MoE gate_up, MoE expert MLP,
autotuned decode/mid): time per call, TFLOP/s, GB/s, roofline fraction, and
the CPU oracle's time on the same workload.  The contract line (last) holds:
  e2e           the same metric through the host-buffer call (mxfp8_linear_host
                via its Python binding): each step copies x in from pinned host
                memory, runs the layer and copies y back to pinned host memory;
                steps alternate over four streams (four requests in flight);
  roofline      the dominant kernel of the timed step (the GEMM, which at
                decode fuses the activation quantization) against HBM bandwidth;
  large_m       the large-M half of the metric: the 8x4 prefill layer and its
                GEMM alone in TFLOP/s and as a fraction of the FP8 tensor peak;
  cpu_baseline  the CPU oracle (plain C, one core) on the full decode call,
                with the host's core count and CPU model;
  clocks        SM clocks and throttle reasons sampled during the timed region;
  weight_prep   the load-time weight preparation of the headline's weight, a
                one-off outside the metric: time and HBM rate.
Floats on the printed lines carry 4 significant digits.

``--impl reference`` times the CPU oracle on the same workload instead
(bounded per step) and prints the same kind of line with "impl": "reference".
Multi-GPU: replicas only (each rank runs its own copy of the workload; no
collective on the data path); value = all ranks' bytes / max time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor-rate ratio (4.5 / 2.25 PF)
L2_BYTES = 126 * 1024 * 1024
GPU_DELAY_CYCLES = 2_000_000  # ~1 ms at 2 GHz, queued ahead of each timed region
E2E_STREAMS = 4   # e2e: independent requests in flight, one stream each
E2E_STEPS = 2000  # e2e: steps timed (a few ms), reported in its "steps" field


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table")
    ap.add_argument("--cpu-seconds", type=float, default=5.0, help="oracle CPU-baseline budget")
    ap.add_argument("--workload", default="decode16",
                    choices=["decode16", "decode1", "tiny", "mid", "mid130", "prefill", "grouped", "moe",
                             "prefill128x4"],
                    help="decode16 = the contract line; any other runs only that workload "
                         "for --steps calls (profiling aid) and prints its table entry")
    return ap.parse_args()


# ------------------------------------------------------------------ peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = float(d.get("hbm_gbs") or d.get("hbm_GBs") or FALLBACK_HBM_GBS)
            bf16 = float(d.get("bf16_tflops") or FALLBACK_BF16_TFLOPS)
            bf16s = float(d.get("bf16_tflops_sustained") or bf16)
            return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16s,
                    "source": "measured"}
        except Exception:  # noqa: BLE001
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_median": statistics.median(power), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ timing utils
def graph_of(fn, n, pre=None, post=None):
    """Capture n back-to-back invocations of fn(i) into one CUDA graph.
    pre: an event recorded (event record node) once an untimed invocation
    captured ahead of the n has completed, on a side branch: the first of the
    n keeps its programmatic dependency on that invocation, as every call has
    on the one before it.  post: an event recorded after the n (and the side
    branch) complete."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(min(n, 2)):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        if pre is not None:
            fn(n)  # untimed: the call before the first timed one
            side.wait_stream(cs)
            with torch.cuda.stream(side):
                pre.record()
        for i in range(n):
            fn(i)
        if pre is not None:
            cs.wait_stream(side)
        if post is not None:
            post.record()
    return g


def graph_events():
    """Two timing events that record inside a captured graph (event record
    nodes), or None where this PyTorch has no such option."""
    import torch
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


TIMING = {"in_graph": "CUDA events inside the captured graphs: start when an untimed call ahead of the "
                      "timed ones completes, stop when the last timed call completes (steady-state periods)",
          "delay": "CUDA events on the launching stream after a queued GPU delay"}


def time_steps(fn, steps, warmup, chunk=1000, barrier=None):
    """Run exactly `warmup` untimed then `steps` timed invocations of fn(i)
    as CUDA-graph replays; return elapsed ms of the timed region (CUDA events,
    synchronised on both sides).  Where PyTorch can record events inside a
    captured graph, the first timed graph opens with one untimed call and the
    start event records when it completes; the timed calls follow it as they
    follow each other (the first may begin its prologue, e.g. its weight
    loads, under that call, as every call does under its predecessor), and
    the stop event records when the last timed call completes: the region is
    `steps` steady-state periods, with no cold first call and no graph launch
    latency in it.  Otherwise both events are recorded on the launching
    stream around the replays."""
    import torch
    chunk = max(1, min(chunk, steps))
    sizes = [chunk] * (steps // chunk) + ([steps % chunk] if steps % chunk else [])
    ev = graph_events()
    if ev is not None:
        e0, e1 = ev
        if len(sizes) == 1:
            graphs = [graph_of(fn, sizes[0], pre=e0, post=e1)]
        else:
            first = graph_of(fn, sizes[0], pre=e0)
            mid = graph_of(fn, chunk) if len(sizes) > 2 else None
            last = graph_of(fn, sizes[-1], post=e1)
            graphs = [first] + [mid] * (len(sizes) - 2) + [last]
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        g_main = graph_of(fn, chunk)
        g_rem = graph_of(fn, sizes[-1]) if sizes[-1] != chunk else None
        graphs = [g_main] * (steps // chunk) + ([g_rem] if g_rem is not None else [])
    wchunk = min(chunk, max(1, warmup))
    g_warm = graph_of(fn, wchunk)
    for _ in range(max(1, warmup // wchunk)):
        g_warm.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # A bounded GPU delay (a fixed number of clock cycles, ~1 ms) ahead of the
    # timed replays: the host submits them while the GPU is still busy with
    # it, so no host submission latency falls between or before them.
    torch.cuda._sleep(GPU_DELAY_CYCLES)
    if ev is None:
        e0.record(stream)
    for g in graphs:
        g.replay()
    if ev is None:
        e1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)


def timing_method():
    return TIMING["in_graph" if graph_events() is not None else "delay"]


def copies_for(nbytes, minimum=2, cap=96):
    return int(min(cap, max(minimum, -(-4 * L2_BYTES // max(nbytes, 1)))))


# --------------------------------------------------------------- workloads
def dense_bytes(m, n, k, bias):
    """Algorithmic bytes of one call: x BF16 + W E4M3 + W scales + bias + y."""
    return 2 * m * k + n * k + n * (k // 32) + (2 * n if bias else 0) + 2 * m * n


def weight_bytes(n, k, experts=1):
    return experts * (n * k + n * (k // 32))


def roofline_entry(flops, nbytes, ms, peaks):
    t = ms * 1e-3
    fp8_tflops = peaks["bf16_tflops"] * FP8_PER_BF16
    t_roof = max(flops / (fp8_tflops * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    bound = "tensor" if flops / (fp8_tflops * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"
    return {"bound": bound, "t_roof_us": t_roof * 1e6, "frac_of_roofline": t_roof / t}


class DenseSetup:
    """Prepared weights + activations for a dense workload on the GPU, in R
    copies so consecutive calls read different memory."""

    def __init__(self, mx, d, copies):
        import torch
        self.d = d
        w = torch.from_numpy(d.w).cuda()
        pw0 = mx.prepare_weight(w)
        del w
        self.pws = [pw0] + [mx.PreparedWeight(pw0.q.clone(), pw0.sf.clone(), pw0.n)
                            for _ in range(copies - 1)]
        x0 = torch.from_numpy(d.x).cuda().to(torch.bfloat16)
        self.xs = [x0] + [x0.clone() for _ in range(copies - 1)]
        self.bias = None if d.bias is None else torch.from_numpy(d.bias).cuda().to(torch.bfloat16)
        self.ws = torch.empty(mx.linear_workspace_bytes(d.m, d.k), dtype=torch.uint8, device="cuda")
        self.y = torch.empty((d.m, d.n), dtype=torch.bfloat16, device="cuda")
        self.mx = mx
        self.R = copies
        q, sf = mx.quantize_act(x0)
        self.qs = [(q, sf)] + [(q.clone(), sf.clone()) for _ in range(copies - 1)]

    def linear(self, i):
        r = i % self.R
        lib = self.mx.library()
        import ctypes
        st = lib.mxfp8_linear(ctypes.c_void_p(self.xs[r].data_ptr()), self.d.m,
                              ctypes.byref(self.pws[r].c),
                              None if self.bias is None else ctypes.c_void_p(self.bias.data_ptr()),
                              ctypes.c_void_p(self.y.data_ptr()), ctypes.c_void_p(self.ws.data_ptr()),
                              self.ws.numel(), self._stream())
        assert st == 0, st

    def gemm(self, i):
        r = i % self.R
        lib = self.mx.library()
        import ctypes
        q, sf = self.qs[r]
        st = lib.mxfp8_gemm(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sf.data_ptr()), self.d.m,
                            ctypes.byref(self.pws[r].c),
                            None if self.bias is None else ctypes.c_void_p(self.bias.data_ptr()),
                            ctypes.c_void_p(self.y.data_ptr()), self._stream())
        assert st == 0, st

    def quant(self, i):
        r = i % self.R
        q, sf = self.qs[r]
        lib = self.mx.library()
        import ctypes
        st = lib.mxfp8_quantize_act(ctypes.c_void_p(self.xs[r].data_ptr()), self.d.m, self.d.k,
                                    ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
                                    self._stream())
        assert st == 0, st

    @staticmethod
    def _stream():
        import ctypes
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def measure_prepare(mx, d, peaks, reps=12):
    """Load-time weight preparation (quantize + pad N + lay out), a one-off
    per weight and not part of the per-call metric: CUDA-event time of
    mxfp8_prepare_weight on the FP32 weight, re-preparing in place over
    enough source copies that every repetition reads HBM (more than 4x L2),
    and its rate over the algorithmic bytes (4NK read; N_pad*K data and
    N_pad*K/32 scales written)."""
    import torch
    w0 = torch.from_numpy(d.w).cuda()
    src_bytes = 4 * d.n * d.k
    copies = min(64, max(2, -(-4 * L2_BYTES // src_bytes) + 1))
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    pw = mx.prepare_weight(w0)
    for i in range(3):
        mx.prepare_weight(ws[i % copies], out=pw)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        mx.prepare_weight(ws[(i + 3) % copies], out=pw)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    n_pad = (d.n + 127) // 128 * 128
    nbytes = src_bytes + n_pad * d.k + n_pad * (d.k // 32)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"us": ms * 1e3, "alg_bytes": nbytes, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "reps": reps, "source": "float32 [%d, %d]" % (d.n, d.k)}


def measure_config(mx, name, d, peaks, calls=2000, tune=False):
    """Time one dense workload.  tune: run the autotuner on the first copy
    first (the stored tactic then serves every call of this class), report
    the chosen tactic, and clear the table afterwards."""
    import torch
    wb = weight_bytes(d.n, d.k)
    nbytes = dense_bytes(d.m, d.n, d.k, d.bias is not None)
    gemm_bytes = (d.m * d.k + mx.act_scale_bytes(d.m, d.k) + wb + (2 * d.n if d.bias is not None else 0)
                  + 2 * d.m * d.n)
    setup = DenseSetup(mx, d, copies_for(nbytes))
    tactic = None
    if tune:
        mx.tactic_clear()
        tactic = mx.autotune_linear(setup.xs[0], setup.pws[0], setup.bias, iters=200)
    warm = max(3, calls // 10)
    ms = time_steps(setup.linear, calls, warmup=warm) / calls
    ms_g = time_steps(setup.gemm, calls, warmup=warm) / calls
    ms_q = time_steps(setup.quant, calls, warmup=warm) / calls
    flops = 2.0 * d.m * d.n * d.k
    out = {"m": d.m, "n": d.n, "k": d.k, "bias": d.bias is not None, "copies": setup.R,
           "us_per_call": ms * 1e3, "gemm_us": ms_g * 1e3, "quant_us": ms_q * 1e3,
           "tflops": flops / (ms * 1e-3) / 1e12, "gemm_tflops": flops / (ms_g * 1e-3) / 1e12,
           "weight_gbs": wb / (ms * 1e-3) / 1e9, "alg_gbs": nbytes / (ms * 1e-3) / 1e9,
           "flops": flops, "alg_bytes": nbytes, "gemm_alg_bytes": gemm_bytes}
    if tune:
        out["tactic"] = {"tokens_per_tile": tactic[0], "split_k": tactic[1], "fuse_quant": tactic[2],
                         "pipes": tactic[3], "note": "autotuned linear; the gemm_us column keeps the heuristic"}
        mx.tactic_clear()
    out.update(roofline_entry(flops, nbytes, ms, peaks))
    out["gemm_only"] = roofline_entry(flops, gemm_bytes, ms_g, peaks)
    del setup
    torch.cuda.empty_cache()
    return out


def measure_128x4(mx, d, peaks, calls=40):
    """The high-M variant with 128x4 activation scales (persistent 256-token
    tiles), timed like measure_config: the whole layer and the GEMM alone."""
    import ctypes
    import torch
    nbytes = dense_bytes(d.m, d.n, d.k, d.bias is not None)
    setup = DenseSetup(mx, d, copies_for(nbytes))
    lib = mx.library()
    ws = torch.empty(lib.mxfp8_linear_128x4_workspace_bytes(d.m, d.k), dtype=torch.uint8, device="cuda")
    q128 = [mx.quantize_act_128x4(x) for x in setup.xs]
    bias = None if setup.bias is None else ctypes.c_void_p(setup.bias.data_ptr())

    def lin(i):
        r = i % setup.R
        st = lib.mxfp8_linear_128x4(ctypes.c_void_p(setup.xs[r].data_ptr()), d.m, ctypes.byref(setup.pws[r].c), bias,
                                    ctypes.c_void_p(setup.y.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                    setup._stream())
        assert st == 0, st

    def gem(i):
        r = i % setup.R
        q, sf = q128[r]
        st = lib.mxfp8_gemm_128x4(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(sf.data_ptr()), d.m,
                                  ctypes.byref(setup.pws[r].c), bias, ctypes.c_void_p(setup.y.data_ptr()),
                                  setup._stream())
        assert st == 0, st

    warm = max(3, calls // 10)
    ms = time_steps(lin, calls, warmup=warm) / calls
    ms_g = time_steps(gem, calls, warmup=warm) / calls
    flops = 2.0 * d.m * d.n * d.k
    out = {"m": d.m, "n": d.n, "k": d.k, "us_per_call": ms * 1e3, "gemm_us": ms_g * 1e3,
           "tflops": flops / (ms * 1e-3) / 1e12, "gemm_tflops": flops / (ms_g * 1e-3) / 1e12,
           "note": "128x4 activation scales, persistent 256-token tiles (vs the 8x4 path's 192-token dual tiles)"}
    out.update(roofline_entry(flops, nbytes, ms, peaks))
    del setup, q128, ws
    torch.cuda.empty_cache()
    return out


def measure_grouped(mx, peaks, calls=200, g=None):
    import torch
    import workloads
    if g is None:
        g = workloads.grouped()
    w = torch.from_numpy(g.w).cuda()
    pw = mx.prepare_weight(w)
    del w
    x = torch.from_numpy(g.x_sorted).cuda().to(torch.bfloat16)
    off = torch.from_numpy(g.offsets).cuda()
    ws = torch.empty(mx.linear_workspace_bytes(g.rows, g.k), dtype=torch.uint8, device="cuda")
    y = torch.empty((g.rows, g.n), dtype=torch.bfloat16, device="cuda")
    lib = mx.library()
    import ctypes

    def call(i):
        st = lib.mxfp8_grouped_linear(ctypes.c_void_p(x.data_ptr()), g.rows,
                                      ctypes.c_void_p(off.data_ptr()), ctypes.byref(pw.c), None,
                                      ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                      ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, st

    ms = time_steps(call, calls, warmup=10) / calls
    flops = 2.0 * g.rows * g.n * g.k
    wb = weight_bytes(g.n, g.k, g.experts)
    nbytes = wb + 2 * g.rows * g.k + 2 * g.rows * g.n + 4 * (g.experts + 1)
    out = {"rows": g.rows, "experts": g.experts, "n": g.n, "k": g.k, "us_per_call": ms * 1e3,
           "tflops": flops / (ms * 1e-3) / 1e12, "weight_gbs": wb / (ms * 1e-3) / 1e9,
           "alg_gbs": nbytes / (ms * 1e-3) / 1e9, "flops": flops, "alg_bytes": nbytes,
           "note": "weights (415 MB) exceed L2; single copy"}
    out.update(roofline_entry(flops, nbytes, ms, peaks))
    del pw, x, ws, y
    torch.cuda.empty_cache()
    return out


def measure_moe(mx, peaks, calls=200):
    """The whole MoE expert MLP (routing, gather + quantize, gated GEMM1 with
    SwiGLU, quantize h, GEMM2, top-k finalize) of the 256-token, 128-expert,
    top-8 layer with H=2048, I=768.  HBM-bound: both weight sets stream once
    per call (604 MB > L2)."""
    import torch
    import workloads
    g = workloads.moe()
    w13 = mx.prepare_gate_up_weight(torch.from_numpy(g.w13).cuda())
    w2 = mx.prepare_weight(torch.from_numpy(g.w2).cuda())
    x = torch.from_numpy(g.x).cuda().to(torch.bfloat16)
    lg = torch.from_numpy(g.logits).cuda()
    ws = torch.empty(mx.moe_workspace_bytes(g.tokens, g.experts, g.topk, g.hidden, g.inter),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((g.tokens, g.hidden), dtype=torch.bfloat16, device="cuda")
    lib = mx.library()
    import ctypes

    def call(i):
        st = lib.mxfp8_moe_expert_mlp(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(lg.data_ptr()), g.tokens,
                                      g.topk, 0, ctypes.byref(w13.c), ctypes.byref(w2.c),
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                      ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, st

    ms = time_steps(call, calls, warmup=10) / calls
    rows = g.tokens * g.topk
    flops = 2.0 * rows * (2 * g.inter) * g.hidden + 2.0 * rows * g.hidden * g.inter
    wb = weight_bytes(2 * g.inter, g.hidden, g.experts) + weight_bytes(g.hidden, g.inter, g.experts)
    # algorithmic bytes: weights + x + logits + out (the intermediates stay in L2)
    nbytes = wb + 2 * g.tokens * g.hidden + 4 * g.tokens * g.experts + 2 * g.tokens * g.hidden
    res = {"tokens": g.tokens, "experts": g.experts, "topk": g.topk, "hidden": g.hidden, "inter": g.inter,
           "us_per_call": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12, "weight_gbs": wb / (ms * 1e-3) / 1e9,
           "alg_gbs": nbytes / (ms * 1e-3) / 1e9, "flops": flops, "alg_bytes": nbytes,
           "note": "route + gate_up/SwiGLU + down + finalize; weights (604 MB) exceed L2; single copy"}
    res.update(roofline_entry(flops, nbytes, ms, peaks))
    del w13, w2, x, lg, ws, out
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU baseline
def host_description():
    """Host core count and CPU model (lscpu, else /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:  # noqa: BLE001
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.machine()}


def _timed(fn, min_s):
    """Mean seconds per call of fn(), repeated until min_s has elapsed (at
    least once)."""
    n = 0
    t0 = time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= min_s:
            return el / n, n


def oracle_dense(d, min_s, rows=None):
    """The CPU oracle (plain C, one core) on one dense call: quantize x, the
    block-scaled product in double, bias.  The weight is quantized first and
    outside the timed region (it is load-time work).  rows: time only these
    output rows and scale the time to all M rows (labelled)."""
    import oracle
    wq, wsf = oracle.quantize_rows(d.w)
    if rows is None:
        sec, n = _timed(lambda: oracle.linear(d.x, wq, wsf, d.bias), min_s)
        scale, sample = 1.0, "full call (all %d rows), %d repetitions" % (d.m, n)
    else:
        sec, n = _timed(lambda: oracle.linear(d.x, wq, wsf, d.bias, rows=rows), min_s)
        scale = d.m / len(rows)
        sample = ("%d sampled rows of %d (all N columns), time scaled by %d to the full call"
                  % (len(rows), d.m, int(scale)))
    sec *= scale
    flops = 2.0 * d.m * d.n * d.k
    return {"us_per_call": sec * 1e6, "tflops": flops / sec / 1e12,
            "weight_gbs": weight_bytes(d.n, d.k) / sec / 1e9, "cores": 1, "kind": "oracle",
            "sample": sample}


def oracle_grouped(g, n_experts):
    """The CPU oracle on the grouped gate_up call, timed on the rows of the
    first n_experts experts (their weights quantized outside the timed region)
    and scaled to all rows by the row count."""
    import oracle
    import oracle.moe as moe
    e = n_experts
    r1 = int(g.offsets[e])
    gq, gsf = moe.prepare_experts(g.w[:e])
    off = np.ascontiguousarray(g.offsets[:e + 1])
    sec, n = _timed(lambda: oracle.grouped_linear(g.x_sorted[:r1], off, gq, gsf), 0.5)
    scale = g.rows / max(r1, 1)
    sec *= scale
    flops = 2.0 * g.rows * g.n * g.k
    return {"us_per_call": sec * 1e6, "tflops": flops / sec / 1e12,
            "weight_gbs": weight_bytes(g.n, g.k, g.experts) / sec / 1e9, "cores": 1, "kind": "oracle",
            "sample": "rows of experts 0..%d (%d of %d rows), time scaled by the row count"
                      % (e - 1, r1, g.rows)}


def cpu_baselines(wl):
    """The oracle on every dense workload and the grouped one: configs 1-3 in
    full; prefill on 64 sampled rows; grouped on the rows of 16 experts."""
    out = {}
    out["tiny_m7_n130_k256"] = oracle_dense(wl["tiny"], 0.5)
    out["decode_m1_n5120_k2048"] = oracle_dense(wl["decode1"], 1.0)
    out["decode_m16_n5120_k2048"] = oracle_dense(wl["decode16"], 1.0)
    out["mid_m128_n2048_k4096"] = oracle_dense(wl["mid"], 0.5)
    out["mid_m128_n130_k4096_bias"] = oracle_dense(wl["mid130"], 0.5)
    rng = np.random.default_rng(7)
    pre = wl["prefill"]
    rows = np.unique(np.concatenate([np.arange(32), [pre.m - 1], rng.choice(pre.m, 31, replace=False)]))
    out["prefill_m8192_n8192_k8192"] = oracle_dense(pre, 0.0, rows=rows)
    out["grouped_t256_e128_top8_n1536_k2048"] = oracle_grouped(wl["grouped"], 16)
    return out


def headline_cpu_baseline(d, budget_s):
    """The contract line's baseline: the oracle on the full decode call (all
    16 tokens x all 5120 weight rows), repeated for about budget_s."""
    import oracle
    wq, wsf = oracle.quantize_rows(d.w)
    sec, n = _timed(lambda: oracle.linear(d.x, wq, wsf, d.bias), budget_s)
    res = {"value": weight_bytes(d.n, d.k) / sec / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "the full decode call (M=16, N=5120, K=2048) %d times, %.1f s" % (n, sec * n)}
    res.update(host_description())
    return res


def compact(v):
    """Floats to 4 significant digits (keeps the printed lines short)."""
    if isinstance(v, float):
        return float("%.4g" % v)
    if isinstance(v, dict):
        return {k: compact(x) for k, x in v.items()}
    if isinstance(v, (list, tuple)):
        return [compact(x) for x in v]
    return v


# ------------------------------------------------------------------- main
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def step_roofline(d, wb, launches_per_step, ms_step, ms_gemm, peak_gbs, traffic, act_sf_bytes):
    """Roofline of the dominant kernel of the timed step.  When the schedule
    fuses the activation quantization, the step is that one GEMM launch:
    its algorithmic bytes (BF16 x, weights and scales, bias, y) over the
    step's time.  Otherwise the GEMM (quantized x and its scales, weights and
    scales, bias, y) over its own per-launch time, measured alone.  The
    other one is reported beside it."""
    fused_bytes = 2 * d.m * d.k + wb + 2 * d.n + 2 * d.m * d.n
    gemm_bytes = d.m * d.k + act_sf_bytes + wb + 2 * d.n + 2 * d.m * d.n
    gemm_alone = {"us_per_launch": ms_gemm * 1e3, "alg_bytes_per_launch": gemm_bytes,
                  "achieved": gemm_bytes / (ms_gemm * 1e-3) / 1e9}
    if launches_per_step == 1:
        ms, nbytes = ms_step, fused_bytes
        kernel = "mxfp8_gemm_kernel<16> (quantization fused; the step's only launch)"
    else:
        ms, nbytes = ms_gemm, gemm_bytes
        kernel = "mxfp8_gemm_kernel<16>"
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
            "frac": achieved / peak_gbs, "traffic": traffic, "kernel": kernel,
            "us_per_launch": ms * 1e3, "alg_bytes_per_launch": nbytes,
            "gemm_prequantized_alone": gemm_alone}


def max_over_ranks(x, ws, device="cuda"):
    """The largest x over all ranks (the slowest rank's time); x itself on
    one rank.  The process group must be initialised when ws > 1."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ws, seconds):
    """Units all ranks processed over the slowest rank's time."""
    return ws * units_per_rank / seconds


def run_reference(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import workloads
    d = workloads.decode(m=16)
    import oracle
    wq, wsf = oracle.quantize_rows(d.w)
    total = args.steps + args.warmup
    # each step: all 16 tokens for a block of weight rows, sized so the whole
    # run stays within ~90 s of CPU time
    t0 = time.perf_counter()
    oracle.linear(d.x, wq[:8], wsf[:8], d.bias[:8])
    per_row = (time.perf_counter() - t0) / 8
    nb = int(max(1, min(d.n, 90.0 / max(1, total) / max(per_row, 1e-9))))
    for i in range(args.warmup):
        c0 = (i * nb) % d.n
        oracle.linear(d.x, wq[c0:c0 + nb], wsf[c0:c0 + nb], d.bias[c0:c0 + nb])
    done = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        c0 = (i * nb) % d.n
        c1 = min(d.n, c0 + nb)
        oracle.linear(d.x, wq[c0:c1], wsf[c0:c1], d.bias[c0:c1])
        done += c1 - c0
    el = time.perf_counter() - t0
    value = done * (d.k + d.k // 32) / el / 1e9
    sample = "per step all %d tokens x %d weight rows of N=%d, K=%d" % (d.m, nb, d.n, d.k)
    line = {"impl": "reference", "metric": "MXFP8 linear weight GB/s (decode M=16, N=5120, K=2048)",
            "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": d.name, "m": d.m, "n": d.n, "k": d.k,
                                            "bias": True},
            "cpu_baseline": dict({"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": sample}, **host_description()),
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def large_m_block(cfgs, peaks):
    """The large-M half of the metric: the 8x4 prefill layer and its GEMM
    alone against the FP8 tensor peak (measured BF16 x the nominal ratio)."""
    p = cfgs.get("prefill_m8192_n8192_k8192")
    if not p:
        return None
    fp8 = peaks["bf16_tflops"] * FP8_PER_BF16
    return {"workload": "prefill_m8192_n8192_k8192", "us_per_call": p["us_per_call"], "tflops": p["tflops"],
            "frac": p["tflops"] / fp8, "gemm_us": p["gemm_us"], "gemm_tflops": p["gemm_tflops"],
            "gemm_frac": p["gemm_tflops"] / fp8, "peak_tflops": fp8,
            "peak": "fp8 = 2 x bf16 %s" % peaks["source"]}


def build_workloads():
    import workloads
    return {"tiny": workloads.tiny(), "decode1": workloads.decode(m=1), "decode16": workloads.decode(m=16),
            "mid": workloads.mid(), "mid130": workloads.mid(n=130, bias=True), "prefill": workloads.prefill(),
            "grouped": workloads.grouped()}


def measure_configs(mx, wl, peaks):
    """Every workload of the layer on the GPU (time per call, TFLOP/s, GB/s,
    roofline), each timed as CUDA-graph replays over rotating copies."""
    cfgs = {}
    cfgs["tiny_m7_n130_k256"] = measure_config(mx, "tiny", wl["tiny"], peaks, 2000)
    cfgs["decode_m1_n5120_k2048"] = measure_config(mx, "d1", wl["decode1"], peaks, 4000)
    cfgs["decode_m16_n5120_k2048"] = measure_config(mx, "d16", wl["decode16"], peaks, 4000)
    cfgs["mid_m128_n2048_k4096"] = measure_config(mx, "mid", wl["mid"], peaks, 2000)
    cfgs["mid_m128_n130_k4096_bias"] = measure_config(mx, "mid130", wl["mid130"], peaks, 2000)
    cfgs["prefill_m8192_n8192_k8192"] = measure_config(mx, "prefill", wl["prefill"], peaks, 40)
    cfgs["prefill_m8192_n8192_k8192_128x4"] = measure_128x4(mx, wl["prefill"], peaks, 40)
    cfgs["grouped_t256_e128_top8_n1536_k2048"] = measure_grouped(mx, peaks, 200, g=wl["grouped"])
    cfgs["moe_mlp_t256_e128_top8_h2048_i768"] = measure_moe(mx, peaks, 200)
    cfgs["decode_m16_n5120_k2048_autotuned"] = measure_config(mx, "d16", wl["decode16"], peaks, 4000, tune=True)
    cfgs["mid_m128_n2048_k4096_autotuned"] = measure_config(mx, "mid", wl["mid"], peaks, 2000, tune=True)
    for name, v in cfgs.items():
        v["peaks"] = "of %s" % peaks["source"]
        # DRAM bytes of one GEMM launch from the committed ncu capture of this
        # workload (None when absent or captured on other kernel sources)
        v["traffic"] = load_traffic("gemm", name)
    return cfgs


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    barrier = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier
    import mxfp8_block_scaled_x4_gb300 as mx
    mx.library()
    import workloads
    peaks = load_peaks()
    peak_src = "of %s" % peaks["source"]
    if args.workload != "decode16":
        builders = {"decode1": lambda: workloads.decode(m=1), "tiny": workloads.tiny,
                    "mid": workloads.mid, "mid130": lambda: workloads.mid(n=130, bias=True),
                    "prefill": workloads.prefill}
        if args.workload == "grouped":
            res = measure_grouped(mx, peaks, args.steps)
        elif args.workload == "moe":
            res = measure_moe(mx, peaks, args.steps)
        elif args.workload == "prefill128x4":
            res = measure_128x4(mx, workloads.prefill(), peaks, args.steps)
        else:
            res = measure_config(mx, args.workload, builders[args.workload](), peaks, args.steps)
        res["workload"] = args.workload
        res["peaks"] = peak_src
        print(json.dumps(res), flush=True)
        return

    d = workloads.decode(m=16)
    wb = weight_bytes(d.n, d.k)
    nbytes = dense_bytes(d.m, d.n, d.k, True)
    setup = DenseSetup(mx, d, copies_for(nbytes))

    # ---- headline: K timed steps of the whole layer
    clocks = ClockSampler(local)
    clocks.start()
    ms = time_steps(setup.linear, args.steps, max(3, args.warmup), barrier=barrier)
    clk = clocks.stop()
    # kernels per call of the timed schedule: the GEMM, plus the activation
    # quantizer unless the GEMM quantizes its own tile
    launches_per_step = 1 if mx.last_schedule()["fused"] else 2
    t_max = max_over_ranks(ms, ws)
    value = whole_job_rate(args.steps * wb, ws, t_max * 1e-3) / 1e9

    # ---- the GEMM on pre-quantized activations, timed alone per launch
    g_steps = min(args.steps, 20000)
    ms_g = time_steps(setup.gemm, g_steps, 100) / g_steps
    roof = step_roofline(d, wb, launches_per_step, t_max / args.steps, ms_g, peaks["hbm_gbs"],
                         load_traffic("gemm", d.name), mx.act_scale_bytes(d.m, d.k))
    roof["peak_source"] = peak_src
    roof.pop("gemm_prequantized_alone", None)

    # ---- e2e through the public API with host buffers
    # its own step count (steady state over four streams), independent of K
    e2e = measure_e2e(mx, setup, steps=E2E_STEPS)
    if ws > 1:  # whole job: every rank's steps over the slowest rank's time
        e2e["us_per_step"] = max_over_ranks(e2e["us_per_step"], ws)
        e2e["value"] = whole_job_rate(wb, ws, e2e["us_per_step"] * 1e-6) / 1e9

    out = {"metric": "MXFP8 linear weight GB/s (decode M=16, N=5120, K=2048)",
           "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
           "data": "synthetic",
           "config": {"workload": d.name, "m": d.m, "n": d.n, "k": d.k, "bias": True,
                      "parallelism": "replicas" if ws > 1 else "single",
                      "l2": "inputs larger than L2: %d rotating copies (%.0f MB)" % (setup.R, setup.R * nbytes / 1e6),
                      "timing": "CUDA-graph replays; " + timing_method()},
           "roofline": roof,
           "gpu_launches": launches_per_step * args.steps,
           "clocks": clk,
           "e2e": e2e}
    gemm_alone_us = ms_g * 1e3
    del setup
    torch.cuda.empty_cache()
    try:  # auxiliary: a failure here must not cost the contract line
        out["weight_prep"] = measure_prepare(mx, d, peaks)
    except Exception as exc:  # noqa: BLE001
        out["weight_prep"] = {"error": repr(exc)}
    torch.cuda.empty_cache()

    if rank == 0:
        wl = build_workloads() if not args.no_configs else {}
        cfgs = {}
        if not args.no_configs:
            cfgs = measure_configs(mx, wl, peaks)
        cpu = {}
        if not args.no_configs:
            try:
                cpu = cpu_baselines(wl)
            except Exception as exc:  # noqa: BLE001
                cpu = {"error": {"error": repr(exc)}}
        # one compact line per workload before the contract line
        for name, v in cfgs.items():
            line = {"bench_config": name}
            line.update(v)
            if name in cpu:
                line["cpu_baseline"] = cpu[name]
            print(json.dumps(compact(line)), flush=True)
        for name, v in cpu.items():
            if name not in cfgs:
                print(json.dumps(compact({"bench_config": name, "cpu_baseline": v})), flush=True)
        lm = large_m_block(cfgs, peaks)
        if lm:
            out["large_m"] = lm
        out["kernel_us"] = {"linear_call": t_max / args.steps * 1e3, "gemm_prequantized": gemm_alone_us}
        out["cpu_baseline"] = headline_cpu_baseline(d, args.cpu_seconds)
        print(json.dumps(compact(out)), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_e2e(mx, setup, steps):
    """Per step: one mxfp8_linear_host call on page-locked host buffers, which
    enqueues the copy of x in, the layer and the copy of y out.  Steps
    alternate over E2E_STREAMS streams, each with its own workspace and host
    output (that many independent requests in flight, so one request's copies
    overlap the others' kernels); the single-stream time is reported beside
    it."""
    import torch
    d = setup.d
    nreq = E2E_STREAMS
    xh = [torch.from_numpy(d.x).to(torch.bfloat16).pin_memory() for _ in range(2)]
    yh = [torch.empty((d.m, d.n), dtype=torch.bfloat16).pin_memory() for _ in range(nreq)]
    ws = [torch.empty((mx.linear_host_workspace_bytes(d.m, d.n, d.k),), dtype=torch.uint8, device="cuda")
          for _ in range(nreq)]
    s0 = torch.cuda.current_stream()
    others = [torch.cuda.Stream() for _ in range(nreq - 1)]
    pws = setup.pws
    b = setup.bias

    # The public C entry point, called with its arguments prepared once (the
    # Python wrapper's checks would add host time to every step).
    import ctypes
    lib = mx.library()
    fn = lib.mxfp8_linear_host
    cvp = ctypes.c_void_p
    b_ptr = None if b is None else cvp(b.data_ptr())

    def args(i, j, streams):
        return (cvp(xh[i % 2].data_ptr()), d.m, ctypes.byref(pws[i % len(pws)].c), b_ptr, cvp(yh[j].data_ptr()),
                cvp(ws[j].data_ptr()), ctypes.c_size_t(ws[j].numel()), cvp(streams[j].cuda_stream))

    def run(nstreams, n):
        streams = ([s0] + others)[:nstreams]
        calls = [args(i, i % nstreams, streams) for i in range(nstreams * len(pws))]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s0)
        for so in streams[1:]:
            so.wait_event(e0)
        for i in range(n):
            st = fn(*calls[i % len(calls)])
            if st != 0:
                raise mx.Mxfp8Error(st, "mxfp8_linear_host")
        for so in streams[1:]:
            done = torch.cuda.Event()
            done.record(so)
            s0.wait_event(done)
        e1.record(s0)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run(nreq, 10)
    run(1, 10)
    ms = run(nreq, steps)
    ms1 = run(1, steps)
    wb = weight_bytes(d.n, d.k)
    return {"value": steps * wb / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": d.m * d.k * 2, "d2h_bytes_per_step": d.m * d.n * 2,
            "us_per_step": ms * 1e3 / steps, "steps": steps,
            "single_stream_us_per_step": ms1 * 1e3 / steps,
            "requests_in_flight": nreq,
            "note": "mxfp8_linear_host via ctypes, one stream per request in flight"}


def code_sha(path):
    """sha256 prefix (16 hex digits) of a C/CUDA source with its comments
    removed, runs of blanks outside string and character literals collapsed
    to one, lines stripped and empty lines dropped: a capture stays valid
    across comment-only edits of the file and no longer across any edit of
    its code."""
    src = open(path, encoding="utf-8").read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in " \t":
            if not out or out[-1] != " ":
                out.append(" ")
            i += 1
        else:
            out.append(c)
            i += 1
    body = "\n".join(ln.strip() for ln in "".join(out).splitlines() if ln.strip())
    return hashlib.sha256(body.encode("utf-8")).hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, valid only while
    the kernel source's code (code_sha) is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        table = json.load(open(path))
        ent = table[kernel][workload]
        src = os.path.join(ROOT, "mxfp8_block_scaled_x4_gb300", "csrc", ent.get("source", "gemm.cu"))
        if ent.get("code_sha") != code_sha(src):
            return None
        return ent["dram_bytes_per_launch"]
    except Exception:  # noqa: BLE001
        return None


if __name__ == "__main__":
    main()
