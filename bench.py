#!/usr/bin/env python3
"""Benchmark of the int8 quantized projection hot path on GB300.

Default workload (the headline): the batch-1 decode GEMV sweep -- q8_0
quantization of the activation, then Q8_0 GEMVs (n, k) = (12288, 7168),
(96, 7168), (512, 128) -- reported as algorithmic HBM GB/s.  The same JSON
line carries a ``prefill`` object: the qwen2-7B-shaped prefill chain
(3325 tokens, d = 3584, nf = 18944: rmsnorm_quant -> gate and up GEMMs ->
swiglu_quant -> down GEMM) with the GEMMs' int8-op throughput.

Inputs are seeded synthetic tensors (no dataset); weights rotate through
copies totalling more than 4x the 129 MB L2 (decode), and the prefill step's
own working set is about 1.2 GB, so no step reads the previous step's data
from L2.

``--impl reference`` times the plain CPU oracle on the host cores on a
bounded sample of the same workload and prints the same line with
``"impl": "reference"``.  Under torchrun every rank runs an independent
replica (the path has no exchange step) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
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

from int8_quantized_projection_gb300 import synthetic as syn  # noqa: E402

METRIC = "Q8_0 GEMV HBM GB/s (b=1) and prefill int8 GEMM TOPS, as % of GB300 roofline"
L2_BYTES = 129 * 1000 * 1000
DECODE_SHAPES = [(12288, 7168), (96, 7168), (512, 128)]
PREFILL = dict(tokens=3325, d=3584, nf=18944, eps=1e-6)

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of a kernel, from
# the ncu capture summarised under profiles/; None until taken, and reset to
# None whenever that kernel changes (the figure would describe old code).
NCU_TRAFFIC_BYTES = {"gemv_fused 12288x7168+96x7168": 97_632_512,      # profiles/gemv_fused_quant_12288x7168_plus_96x7168.md
                     "gemm_tc 18944x3584 t=3325": 396_982_272,         # profiles/gemm_tc_18944x3584_t3325.md
                     "gemv_small 12288x7168 t=16": 97_616_896,         # profiles/gemv_small_12288x7168_t16.md
                     "gemv_staged_q4a 12288x7168": 55_090_176}         # profiles/gemv_staged_q4a_12288x7168.md


# ---------------------------------------------------------------------------
# algorithmic bytes / ops per call (counted with the true token count)
# ---------------------------------------------------------------------------
def bytes_quantize(rows, k):
    return 4 * rows * k + rows * k + 4 * rows * (k // 32)


def bytes_gemv(n, k):
    return n * (k // 32) * 34 + k + 4 * (k // 32) + 4 * n


def bytes_rmsnorm_quant(rows, d, write_y=True):
    # x read, the weight vector, the plane written, and the f32 output unless it is dead (mode 2)
    return (8 if write_y else 4) * rows * d + 4 * d + rows * d + 4 * rows * (d // 32)


def bytes_swiglu_quant(rows, nf, write_y=True):
    # gate + up read, the plane written, and the f32 output unless it is dead (mode 2)
    return (12 if write_y else 8) * rows * nf + rows * nf + 4 * rows * (nf // 32)


def ops_gemm(t, n, k):
    return 2 * t * n * k


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.window = None

    def mark(self, begin):
        """Record the host time at which the timed region begins / ends."""
        if begin:
            self.window = [time.time(), None]
        elif self.window is not None:
            self.window[1] = time.time()

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # let the sampler reach its steady cadence before the timed region
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        # keep the samples taken during the timed region, widened by one
        # sampling interval on each side so that short regions still get some
        if self.window and self.window[1]:
            lo, hi = self.window[0] - 0.06, self.window[1] + 0.06
            kept = []
            for r in rows:
                try:
                    ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float(
                        "0." + r[0].split(".")[1]) if "." in r[0] else 0.0
                except (ValueError, IndexError):
                    ts = None
                if ts is None or lo <= ts <= hi:
                    kept.append(r)
            rows = kept or rows[-2:]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(torch, values, device):
    """Element-wise maximum of a list of floats over all ranks (one all-reduce).

    Each replica times its own steps; a job is as slow as its slowest rank."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


GRAPH_STEPS = 60  # steps per timed CUDA graph (rounded to a multiple of the weight copies)
E2E_MIN_STEPS = 300  # steps the end-to-end loops time at least


def hold_device(torch, launches):
    """Keep the stream busy (a device-side sleep, before the start event) while
    the host enqueues `launches` graph replays, so that the timed region
    measures the device and not the host's launch latency."""
    torch.cuda._sleep(int(2_000_000 + 40_000 * launches))  # cycles: ~1 ms + ~20 us per replay


def gpu_smi_id(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev)


# ---------------------------------------------------------------------------
# decode workload (headline)
# ---------------------------------------------------------------------------
def decode_inputs():
    g = syn.rng(1, 0)
    xs = {k: syn.activations(g, 1, k, sigma=1.5, outlier_frac=0.01) for k in (7168, 128)}
    ws = [syn.q8_0_weights(syn.rng(1, 1 + i), n, k)[0] for i, (n, k) in enumerate(DECODE_SHAPES)]
    return xs, ws


def decode_bytes(fused=False):
    """Algorithmic bytes of one decode step.  fused: the k = 7168 activation is
    quantized inside the grouped GEMV (q8_0_gemv_fused), so it is read once as
    f32 and no plane is written or read; the k = 128 chain is unchanged."""
    side = bytes_quantize(1, 128) + bytes_gemv(*DECODE_SHAPES[2])
    if fused:
        return bytes_gemv_fused(7168, [DECODE_SHAPES[0][0], DECODE_SHAPES[1][0]], "quant") + side
    return bytes_quantize(1, 7168) + sum(bytes_gemv(n, k) for n, k in DECODE_SHAPES[:2]) + side


def run_decode(torch, q8p, steps, warmup, dev, sampler):
    xs_h, ws_h = decode_inputs()
    per_copy = sum(w.nbytes for w in ws_h)
    copies = max(2, -(-4 * L2_BYTES // per_copy))
    ws = [[torch.from_numpy(w).to(dev) for w in ws_h] for _ in range(copies)]
    # the step's inputs and outputs each live in one buffer (16-byte aligned
    # views), so the end-to-end step moves them with one copy each way
    x_all = torch.cat([torch.from_numpy(xs_h[7168]), torch.from_numpy(xs_h[128])], dim=1).to(dev)
    xs = {7168: x_all[:, :7168], 128: x_all[:, 7168:]}
    planes = {k: q8p.empty_plane(1, k, dev) for k in xs}
    y_all = torch.empty(sum(n for n, _ in DECODE_SHAPES), dtype=torch.float32, device=dev)
    ys = list(torch.split(y_all, [n for n, _ in DECODE_SHAPES]))
    stream = torch.cuda.current_stream(dev)

    # every launch pre-marshalled once (one ctypes call per launch in the loop)
    # The two k = 7168 projections share one activation: one grouped launch
    # ("Part 4 - Lecture 05", sec. 2.5) that also quantizes it (sec. 4: producer
    # and consumer in one launch); the k = 128 one (4 blocks per row, not a
    # staged shape) has its own quantize and plane.
    def main_call(wset, stream_=None):
        return q8p.q8_0_gemv_fused([(wset[0], DECODE_SHAPES[0][0], ys[0]), (wset[1], DECODE_SHAPES[1][0], ys[1])],
                                   7168, q8p.PRODUCER_QUANT, xs[7168][0], stream=stream_, bind=True)

    quant128 = q8p.quantize_q8_0(xs[128], *planes[128], bind=True)
    gemvs = [[main_call(wset), q8p.q8_0_gemv(wset[2], *DECODE_SHAPES[2], *planes[128], ys[2], bind=True)]
             for wset in ws]

    def step(i, ev=None):
        g = gemvs[i % copies]
        if ev is not None:
            ev[0].record(stream)
        g[0]()
        if ev is not None:
            ev[1].record(stream)
        quant128()
        g[1]()

    for i in range(warmup):
        step(i)
    q8p.q8_check()
    # The headline region replays CUDA graphs of decode steps (the weight
    # copies in turn): a step's launches are a few microseconds of GPU work
    # each, so issuing them one by one from the host measures the host.  The
    # captured launches keep their programmatic-dependent-launch edges, and
    # nothing is recorded between them (an event between two launches would
    # keep the next kernel from starting while the previous one drains).  The
    # k = 128 chain (its quantize, then its GEMV) shares no data with the
    # k = 7168 chain, so the graph runs it as a parallel branch: its small
    # CTAs sit beside the grouped GEMV's one CTA per SM instead of adding two
    # launch latencies to every step.
    cap, side = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    quant_side = q8p.quantize_q8_0(xs[128], *planes[128], stream=side, bind=True)
    gemvs_c = [[main_call(wset, cap),
                q8p.q8_0_gemv(wset[2], *DECODE_SHAPES[2], *planes[128], ys[2], stream=side, bind=True)] for wset in ws]
    # the same step with the k = 7168 quantize as its own launch (for comparison)
    quant_main = q8p.quantize_q8_0(xs[7168], *planes[7168], stream=cap, bind=True)
    grouped_c = [q8p.q8_0_gemv_grouped([(wset[0], DECODE_SHAPES[0][0], ys[0]), (wset[1], DECODE_SHAPES[1][0], ys[1])],
                                       7168, *planes[7168], stream=cap, bind=True) for wset in ws]

    def steps_main(n):  # the fused k = 7168 GEMV alone, n launches on weight copies 0, 1, ... in turn
        for i in range(n):
            gemvs_c[i % copies][0]()

    def steps_part(n, fused=True):  # n decode steps on weight copies 0, 1, ... in turn
        side.wait_stream(cap)  # fork
        for i in range(n):
            c = i % copies
            if fused:
                gemvs_c[c][0]()
            else:
                quant_main()
                grouped_c[c]()
            quant_side()
            gemvs_c[c][1]()
        cap.wait_stream(side)  # join

    def capture(fn):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=cap):
            fn()
        return g_

    # K timed steps = reps replays of a graph of G steps (G a multiple of the
    # copy count, so the weight copies keep rotating), then one replay of a
    # graph of the remaining K mod G steps: every timed step is a graph
    # replay, whatever K is.  The host enqueues the replays behind a device
    # sleep (outside the events), so no host launch latency lands inside the
    # timed region.
    G = copies * max(1, GRAPH_STEPS // copies)
    reps, rem = divmod(steps, G)
    cap.wait_stream(stream)
    steps_part(copies)  # the same launches once outside the capture
    steps_part(copies, False)
    graph = capture(lambda: steps_part(G))
    graph_rem = capture(lambda: steps_part(rem)) if rem else None
    graph_two = capture(lambda: steps_part(G, False))
    graph_two_rem = capture(lambda: steps_part(rem, False)) if rem else None
    graph_main = capture(lambda: steps_main(G))
    graph_main_rem = capture(lambda: steps_main(rem)) if rem else None
    stream.wait_stream(cap)

    def timed(g_full, g_rem, sample=False):
        g_full.replay()  # warm
        torch.cuda.synchronize(dev)
        if sample:
            sampler.start()
            sampler.mark(True)
        hold_device(torch, reps + (g_rem is not None))
        t0.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        if sample:
            sampler.mark(False)
        q8p.q8_check()
        return t0.elapsed_time(t1)

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = timed(graph, graph_rem, sample=True)
    clocks = sampler.stop()
    ms_two = timed(graph_two, graph_two_rem) / steps
    # The roofline's kernel duration: the fused k = 7168 GEMV alone, K launches
    # back to back from graphs built like the step's (one launch per weight
    # copy in turn, programmatic dependent launch between them, as in the
    # step), CUDA events around the K launches, the mean per launch.
    kern_ms = timed(graph_main, graph_main_rem) / steps
    # The same launches each bracketed by its own events (no overlap with its
    # neighbours): reported beside it as the isolated launch time.
    nev = min(steps, 4 * copies)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nev)]
    torch.cuda.synchronize(dev)
    for i in range(nev):
        step(warmup + i, evs[i])
    torch.cuda.synchronize(dev)
    q8p.q8_check()
    iso_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)

    # end to end through the public API with host buffers (weights resident).
    # A serving loop records its step once -- the host-to-device copy of the
    # inputs from pinned memory, the library calls, the device-to-host copy of
    # the outputs -- as a CUDA graph and replays it every step.  Independent
    # requests let it keep several steps in flight: consecutive steps use three
    # sets of device buffers on three streams, so one step's copies and its
    # launch's ramp and tail overlap the other steps' kernels, and the host
    # enqueues step i, then waits for step i-5 and reads its outputs; the six
    # host buffers rotate, so a step never writes the buffer the host is
    # reading (`e2e_s`).  `e2e_serial_s` waits
    # for every step before enqueuing the next (one buffer set);
    # `e2e_eager_s` also issues the step call by call.
    nbuf, nsets = 6, 3
    xh = [x_all.cpu().pin_memory() for _ in range(nbuf)]
    yh = [torch.empty(y_all.shape, dtype=torch.float32).pin_memory() for _ in range(nbuf)]

    def make_set(k):  # device buffers, streams and bound calls of buffer set k
        if k == 0:
            xa, ya, pl, cp_, sd_ = x_all, y_all, planes[128], cap, side
        else:
            xa, ya = torch.empty_like(x_all), torch.empty_like(y_all)
            pl, cp_, sd_ = q8p.empty_plane(1, 128, dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        yv = list(torch.split(ya, [n for n, _ in DECODE_SHAPES]))
        mains = [q8p.q8_0_gemv_fused([(wset[0], DECODE_SHAPES[0][0], yv[0]), (wset[1], DECODE_SHAPES[1][0], yv[1])],
                                     7168, q8p.PRODUCER_QUANT, xa[0, :7168], stream=cp_, bind=True) for wset in ws]
        q128 = q8p.quantize_q8_0(xa[:, 7168:], *pl, stream=sd_, bind=True)
        g128 = [q8p.q8_0_gemv(wset[2], *DECODE_SHAPES[2], *pl, yv[2], stream=sd_, bind=True) for wset in ws]
        return dict(x=xa, y=ya, cap=cp_, side=sd_, mains=mains, q128=q128, g128=g128, launch=torch.cuda.Stream(dev))

    sets = [make_set(k) for k in range(nsets)]

    def e2e_body(st, i, par):  # on set st's capture streams: the inputs in, one step, the outputs out
        st["x"].copy_(xh[par], non_blocking=True)
        st["side"].wait_stream(st["cap"])
        st["mains"][i]()
        st["q128"]()
        st["g128"][i]()
        st["cap"].wait_stream(st["side"])
        yh[par].copy_(st["y"], non_blocking=True)

    e2e_graphs = []  # [weight copy][host buffer]; host buffer h runs on buffer set h % nsets
    for st_i, st in enumerate(sets):
        st["cap"].wait_stream(stream)
        with torch.cuda.stream(st["cap"]):
            for i in range(copies):  # once outside the capture
                e2e_body(st, i, st_i)
        stream.wait_stream(st["cap"])
    for i in range(copies):
        row = []
        for par in range(nbuf):
            st = sets[par % nsets]
            gi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gi, stream=st["cap"]):
                e2e_body(st, i, par)
            row.append(gi)
        e2e_graphs.append(row)
    torch.cuda.synchronize(dev)
    done = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_run(n, start):  # up to nbuf - 1 steps in flight, alternating buffer sets and streams
        for j in range(n):
            i = start + j
            h = i % nbuf
            ls = sets[h % nsets]["launch"]
            with torch.cuda.stream(ls):
                e2e_graphs[i % copies][h].replay()
                done[h].record(ls)
            if j >= nbuf - 1:
                done[(i - nbuf + 1) % nbuf].synchronize()  # that step's outputs are in yh[(i - nbuf + 1) % nbuf]
        for j in range(max(0, n - nbuf + 1), n):
            done[(start + j) % nbuf].synchronize()

    def e2e_serial_run(n, start):
        for j in range(n):
            i = start + j
            e2e_graphs[i % copies][0].replay()
            stream.synchronize()

    def e2e_eager_run(n, start):
        for j in range(n):
            x_all.copy_(xh[0], non_blocking=True)
            step(start + j)
            yh[0].copy_(y_all, non_blocking=True)
            stream.synchronize()

    # the end-to-end loops run at least E2E_MIN_STEPS steps, so that filling and
    # draining the steps in flight does not dominate a short run
    e2e_steps = max(steps, E2E_MIN_STEPS)
    res = {}
    for name, fn in (("e2e_s", e2e_run), ("e2e_serial_s", e2e_serial_run), ("e2e_eager_s", e2e_eager_run)):
        fn(warmup, 0)
        torch.cuda.synchronize(dev)
        e0 = time.perf_counter()
        fn(e2e_steps, warmup)
        res[name] = (time.perf_counter() - e0) * steps / e2e_steps  # seconds for `steps` steps at that rate
        q8p.q8_check()
    e2e_s, e2e_serial_s, e2e_eager_s = res["e2e_s"], res["e2e_serial_s"], res["e2e_eager_s"]
    return dict(ms=ms, kern_ms=kern_ms, iso_ms=iso_ms, clocks=clocks, e2e_steps=e2e_steps, e2e_s=e2e_s, e2e_serial_s=e2e_serial_s, e2e_eager_s=e2e_eager_s,
                copies=copies, ms_two=ms_two,
                h2d=sum(v.nbytes for v in xs_h.values()), d2h=4 * sum(n for n, _ in DECODE_SHAPES))


# ---------------------------------------------------------------------------
# tiny GEMV (one 256 x 512 projection, batch 1): latency-bound
# ---------------------------------------------------------------------------
TINY = dict(n=256, k=512)


def tiny_inputs():
    n, k = TINY["n"], TINY["k"]
    x = syn.activations(syn.rng(0, 0), 1, k)
    w = syn.q8_0_weights(syn.rng(0, 1), n, k)[0]
    return x, w


def bytes_tiny():
    n, k = TINY["n"], TINY["k"]
    return bytes_quantize(1, k) + bytes_gemv(n, k)


def graph_schedule(torch, cap, issue, steps, copies, per_graph=600):
    """CUDA graphs that together issue steps 0..steps-1 (step i on weight copy
    i mod copies) and the order to replay them in.  A graph holds at most
    `per_graph` steps; graphs are shared between runs of steps that start on
    the same copy."""
    graphs, order, i = {}, [], 0
    G = max(1, min(per_graph, steps))
    while i < steps:
        ln = min(G, steps - i)
        key = (i % copies, ln)
        if key not in graphs:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=cap):
                for j in range(ln):
                    issue(i + j)
            graphs[key] = g_
        order.append(graphs[key])
        i += ln
    return order


def run_tiny(torch, q8p, steps, warmup, dev):
    """The quantize of a 1 x 512 activation and the 256 x 512 projection per
    step, timed two ways: one q8_0_gemv_fused launch (the quantize inside the
    GEMV) and quantize_q8_0 -> q8_0_gemv (two launches).  The weights rotate
    through copies totalling > 4 x L2; every timed step is a graph replay."""
    n, k = TINY["n"], TINY["k"]
    x_h, w_h = tiny_inputs()
    copies = -(-4 * L2_BYTES // w_h.nbytes)
    wall = torch.from_numpy(w_h).to(dev).repeat(copies)
    ws = [wall[i * w_h.nbytes:(i + 1) * w_h.nbytes] for i in range(copies)]
    x = torch.from_numpy(x_h).to(dev)
    plane = q8p.empty_plane(1, k, dev)
    y = torch.empty(n, dtype=torch.float32, device=dev)
    cap = torch.cuda.Stream(dev)
    quant = q8p.quantize_q8_0(x, *plane, stream=cap, bind=True)
    gemvs = [q8p.q8_0_gemv(w, n, k, *plane, y, stream=cap, bind=True) for w in ws]
    fused = [q8p.q8_0_gemv_fused([(w, n, y)], k, q8p.PRODUCER_QUANT, x[0], stream=cap, bind=True) for w in ws]

    def issue_two(i):
        quant()
        gemvs[i % copies]()

    def issue_fused(i):
        fused[i % copies]()

    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, issue in (("fused", issue_fused), ("two", issue_two)):
        cap.wait_stream(stream)
        for i in range(max(warmup, 1)):
            issue(i)
        q8p.q8_check()
        order = graph_schedule(torch, cap, issue, steps, copies)
        stream.wait_stream(cap)
        for g_ in order[:1]:
            g_.replay()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, len(order))
        t0.record(stream)
        for g_ in order:
            g_.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        res[name] = 1e3 * t0.elapsed_time(t1) / steps
        del order
    return dict(us=res["fused"], us_two=res["two"], copies=copies, steps=steps)


# ---------------------------------------------------------------------------
# prefill chain
# ---------------------------------------------------------------------------
def prefill_inputs():
    T, d, nf = PREFILL["tokens"], PREFILL["d"], PREFILL["nf"]
    g = syn.rng(3, 0)
    x = syn.activations(g, T, d)
    w = syn.uniform(g, d, 0.5, 1.5)
    wg = syn.q8_0_weights(syn.rng(3, 1), nf, d)[0]
    wu = syn.q8_0_weights(syn.rng(3, 2), nf, d)[0]
    wd = syn.q8_0_weights(syn.rng(3, 3), d, nf)[0]
    return x, w, wg, wu, wd


def run_prefill(torch, q8p, steps, warmup, dev):
    T, d, nf, eps = PREFILL["tokens"], PREFILL["d"], PREFILL["nf"], PREFILL["eps"]
    x_h, w_h, wg_h, wu_h, wd_h = prefill_inputs()
    x, w, wg, wu, wd = (torch.from_numpy(a).to(dev) for a in (x_h, w_h, wg_h, wu_h, wd_h))
    tp = q8p.q8_plane_rows(T)
    pa = q8p.empty_plane(tp, d, dev)
    G = torch.empty((T, nf), dtype=torch.float32, device=dev)
    U = torch.empty((T, nf), dtype=torch.float32, device=dev)
    pb = q8p.empty_plane(tp, nf, dev)
    O = torch.empty((T, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = ["rmsnorm_quant", "gemm_gate", "gemm_up", "swiglu_quant", "gemm_down"]
    ws_d = q8p.gemm_workspace(nf, T, d, dev)    # gate and up: same shapes, ordered on one stream
    ws_f = q8p.gemm_workspace(d, T, nf, dev)    # down
    # mode 2 for both producers: the GEMMs read only the planes, so the f32
    # outputs of the norm and of SwiGLU are dead
    calls = [q8p.rmsnorm_quant(x, w, eps, None, *pa, bind=True),
             q8p.q8_0_gemm(wg, nf, d, *pa, T, G, workspace=ws_d, bind=True),
             q8p.q8_0_gemm(wu, nf, d, *pa, T, U, workspace=ws_d, bind=True),
             q8p.swiglu_quant(G, U, None, *pb, bind=True),
             q8p.q8_0_gemm(wd, d, nf, *pb, T, O, workspace=ws_f, bind=True)]

    def step(ev=None):
        for i, call in enumerate(calls):
            if ev is not None:
                ev[i].record(stream)
            call()
        if ev is not None:
            ev[5].record(stream)

    for _ in range(warmup):
        step()
    q8p.q8_check()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    q8p.q8_check()
    per = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, nm in enumerate(names)}

    def chain_back_to_back():
        """Mean time of one chain with `steps` chains issued back to back
        between one pair of events (each call's start under the previous
        call's tail, as a prefill of several layers runs)."""
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, 5 * steps)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        return e0.elapsed_time(e1) / steps

    b2b_chain = {"chain": chain_back_to_back()}
    # the standalone prepass of the same activation (not part of the chain, whose
    # producers are fused): quantize_q8_0 of x into the d-wide plane, timed alone
    quant = q8p.quantize_q8_0(x, *pa, bind=True)
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for a, b in qev:
        a.record(stream)
        quant()
        b.record(stream)
    torch.cuda.synchronize(dev)
    q8p.q8_check()
    per["quantize_q8_0 (standalone, not in the chain)"] = statistics.mean(a.elapsed_time(b) for a, b in qev)
    # each producer back to back (as in a chain of layers, the next call's start
    # under the previous one's tail): 20 calls between one pair of events, the
    # f32 inputs rotating over copies that together exceed L2
    xs = [x] + [x.clone() for _ in range(-(-L2_BYTES // (4 * x.numel())))]  # > L2 together
    b2b = {}
    for nm, cl in (("rmsnorm_quant", [q8p.rmsnorm_quant(xc, w, eps, None, *pa, bind=True) for xc in xs]),
                   ("swiglu_quant", [q8p.swiglu_quant(G, U, None, *pb, bind=True)]),
                   ("quantize_q8_0", [q8p.quantize_q8_0(xc, *pa, bind=True) for xc in xs])):
        for i in range(max(3, warmup)):
            cl[i % len(cl)]()
        q8p.q8_check()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, 20)
        e0.record(stream)
        for i in range(20):
            cl[i % len(cl)]()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        b2b[nm] = e0.elapsed_time(e1) / 20
    del xs
    # the same chain on weights prepared once per matrix (q8_0_gemm_prepare_weights,
    # outside the timed region): the GEMMs skip their per-call weight pre-pass
    wg_p, wu_p = (q8p.q8_0_gemm_prepare_weights(m, nf, d) for m in (wg, wu))
    wd_p = q8p.q8_0_gemm_prepare_weights(wd, d, nf)
    wsp_d = torch.empty(q8p.q8_0_gemm_prepared_workspace_bytes(nf, T, d), dtype=torch.uint8, device=dev)
    wsp_f = torch.empty(q8p.q8_0_gemm_prepared_workspace_bytes(d, T, nf), dtype=torch.uint8, device=dev)
    calls[1] = q8p.q8_0_gemm_prepared(None, wg_p, nf, d, *pa, T, G, workspace=wsp_d, bind=True)
    calls[2] = q8p.q8_0_gemm_prepared(None, wu_p, nf, d, *pa, T, U, workspace=wsp_d, bind=True)
    calls[4] = q8p.q8_0_gemm_prepared(None, wd_p, d, nf, *pb, T, O, workspace=wsp_f, bind=True)
    for _ in range(warmup):
        step()
    q8p.q8_check()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    q8p.q8_check()
    prepared = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, nm in enumerate(names)}
    b2b_chain["chain_prepared"] = chain_back_to_back()
    b2b.update(b2b_chain)
    return per, prepared, b2b


# ---------------------------------------------------------------------------
# small-batch decode: one projection for a few tokens, weights read once
# ---------------------------------------------------------------------------
SMALL = {"n": 12288, "k": 7168, "tokens": 16}


def bytes_small(n, k, t):
    return n * (k // 32) * 34 + t * (k + 4 * (k // 32)) + 4 * t * n


def time_calls(torch, q8p, calls, steps, warmup, dev):
    """Mean device time of one launch, two ways: each launch bracketed by its
    own pair of events (`us`, no overlap with its neighbours), and all `steps`
    launches back to back under one pair (`us_b2b`, the prologue of each
    overlapping the tail of the previous one as in a decode stream).  Launch i
    uses weight copy i mod copies, so consecutive launches read different
    memory (together > 4 x L2)."""
    copies = len(calls)
    for i in range(warmup):
        calls[i % copies]()
    q8p.q8_check()
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        evs[i][0].record(stream)
        calls[(warmup + i) % copies]()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        calls[(warmup + i) % copies]()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    q8p.q8_check()
    return dict(us=1e3 * statistics.mean(a.elapsed_time(b) for a, b in evs), us_b2b=1e3 * e0.elapsed_time(e1) / steps,
                copies=copies)


def run_small(torch, q8p, steps, warmup, dev):
    n, k, t = SMALL["n"], SMALL["k"], SMALL["tokens"]
    w_h = syn.q8_0_weights(syn.rng(4, 1), n, k)[0]
    copies = max(2, -(-4 * L2_BYTES // w_h.nbytes))
    ws = [torch.from_numpy(w_h).to(dev) for _ in range(copies)]
    x = torch.from_numpy(syn.activations(syn.rng(4, 0), t, k, sigma=1.5, outlier_frac=0.01)).to(dev)
    plane = q8p.empty_plane(q8p.q8_plane_rows(t), k, dev)
    q8p.quantize_q8_0(x, *plane)
    y = torch.empty((t, n), dtype=torch.float32, device=dev)
    calls = [q8p.q8_0_gemv_batched(w, n, k, *plane, t, y, bind=True) for w in ws]
    return time_calls(torch, q8p, calls, steps, warmup, dev)


# ---------------------------------------------------------------------------
# asymmetric 4-bit weights (value d*nib - m), batch 1: the ssum consumer
# ---------------------------------------------------------------------------
ASYM = {"n": 12288, "k": 7168}


def bytes_q4a_gemv(n, k):
    return n * (k // 32) * 20 + k + 4 * (k // 32) + 4 * n


def run_asym(torch, q8p, steps, warmup, dev):
    n, k = ASYM["n"], ASYM["k"]
    w_h = syn.q4a_weights(syn.rng(5, 1), n, k)[0]
    copies = max(2, -(-4 * L2_BYTES // w_h.nbytes))
    ws = [torch.from_numpy(w_h).to(dev) for _ in range(copies)]
    x = torch.from_numpy(syn.activations(syn.rng(5, 0), 1, k, sigma=1.5, outlier_frac=0.01)).to(dev)
    plane = q8p.empty_plane(1, k, dev)
    q8p.quantize_q8_0(x, *plane)
    y = torch.empty(n, dtype=torch.float32, device=dev)
    calls = [q8p.q4a_gemv(w, n, k, *plane, y, bind=True) for w in ws]
    return time_calls(torch, q8p, calls, steps, warmup, dev)


# ---------------------------------------------------------------------------
# shared-activation decode: one RMSNorm-quantized activation feeding four
# projections (q, k, v, gate) in one grouped launch
# ---------------------------------------------------------------------------
SHARED = dict(d=7168, ns=[3072, 512, 512, 3072], eps=1e-6)


def bytes_shared(fused=False):
    d = SHARED["d"]
    if fused:
        return bytes_gemv_fused(d, SHARED["ns"], "rmsnorm")
    return bytes_rmsnorm_quant(1, d, False) + bytes_gemv_group(d, SHARED["ns"])


def run_shared(torch, q8p, steps, warmup, dev):
    """RMSNorm + q8_0 quantize feeding the four projections, timed two ways:
    one q8_0_gemv_fused launch per step (the norm computed inside the grouped
    GEMV), and rmsnorm_quant (mode 2) -> q8_0_gemv_grouped (two launches).
    Each is recorded as a CUDA graph of about GRAPH_STEPS steps (the weight
    copies in turn, together > 4 x L2), as the decode step is."""
    d, ns, eps = SHARED["d"], SHARED["ns"], SHARED["eps"]
    g = syn.rng(2, 0)
    x = torch.from_numpy(syn.activations(g, 1, d)).to(dev)
    nw = torch.from_numpy(syn.uniform(g, d, 0.5, 1.5)).to(dev)
    host = [syn.q8_0_weights(syn.rng(2, 1 + i), n, d)[0] for i, n in enumerate(ns)]
    per_copy = sum(w.nbytes for w in host)
    copies = max(2, -(-4 * L2_BYTES // per_copy))
    ws = [[torch.from_numpy(w).to(dev) for w in host] for _ in range(copies)]
    plane = q8p.empty_plane(1, d, dev)
    ys = [torch.empty(n, dtype=torch.float32, device=dev) for n in ns]
    cap = torch.cuda.Stream(dev)
    norm = q8p.rmsnorm_quant(x, nw, eps, None, *plane, stream=cap, bind=True)
    gemvs = [q8p.q8_0_gemv_grouped(list(zip(wset, ns, ys)), d, *plane, stream=cap, bind=True) for wset in ws]
    fused = [q8p.q8_0_gemv_fused(list(zip(wset, ns, ys)), d, q8p.PRODUCER_RMSNORM, x[0], None, nw, eps,
                                 stream=cap, bind=True) for wset in ws]
    steps_two = [[norm, gm] for gm in gemvs]  # one step per weight copy
    steps_fused = [[fu] for fu in fused]
    stream = torch.cuda.current_stream(dev)
    per_graph = copies * max(1, GRAPH_STEPS // copies)  # steps per graph, as the decode step's graphs
    reps = max(1, steps // per_graph)
    res = {}
    for name, per_copy_calls in (("fused", steps_fused), ("two", steps_two)):
        cap.wait_stream(stream)
        for i in range(max(copies, warmup)):
            for c in per_copy_calls[i % copies]:
                c()
        q8p.q8_check()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(per_graph):
                for c in per_copy_calls[i % copies]:
                    c()
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, reps)
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        res[name] = 1e3 * t0.elapsed_time(t1) / (reps * per_graph)
        del graph
    return dict(us=res["fused"], us_two=res["two"], copies=copies, steps=reps * per_graph, per_graph=per_graph)


# ---------------------------------------------------------------------------
# layer-stack decode: every projection of a 28-layer d = 3584 model and its
# LM head for one token (batch 1), recorded as one CUDA graph
# ---------------------------------------------------------------------------
LAYERS = dict(layers=28, d=3584, nf=18944, q=3584, kv=512, vocab=152064, eps=1e-6)
# The layer stack's headline launch plan, the set that measured fastest in
# the chain: RMSNorm -> q/k/v, quantize -> o and the final RMSNorm -> LM head
# inside their GEMV launch (q8_0_gemv_fused), and gate/up as one
# q8_0_gemv_gate_up launch on rmsnorm_quant's plane whose epilogue writes the
# SwiGLU output's plane for down ("gu_pair").  Fusing SwiGLU into down instead
# is slower (every CTA recomputes the 18944-wide row), and so, in the chain,
# is RMSNorm inside the gate/up launch.
LAYER_FUSED = ("qkv", "o", "gu_pair", "head")


def layer_groups():
    """One layer's launches of projections: (activation width k, [rows of each projection])."""
    L = LAYERS
    d, nf = L["d"], L["nf"]
    return [(d, [L["q"], L["kv"], L["kv"]]), (d, [d]), (d, [nf, nf]), (nf, [d])]


def bytes_gemv_group(k, ns):
    # every projection's weights and outputs, the shared activation read once
    return sum(n * (k // 32) * 34 + 4 * n for n in ns) + k + 4 * (k // 32)


def bytes_gemv_fused(k, ns, producer):
    # every projection's weights and outputs, and the producer's f32 inputs read
    # once (x; x and the norm weight; gate and up): no plane is written or read
    f32_in = {"quant": 4 * k, "rmsnorm": 8 * k, "swiglu": 8 * k}[producer]
    return sum(n * (k // 32) * 34 + 4 * n for n in ns) + f32_in


def bytes_layer_stack(fused=(), layers=None):
    """Algorithmic bytes of one token; `fused` = the producers computed inside
    their consumer's launch (of "qkv", "o", "gu", "down", "head")."""
    L = dict(LAYERS, layers=layers or LAYERS["layers"])
    d, nf = L["d"], L["nf"]
    (_, qkv), (_, o), (_, gu), (_, down) = layer_groups()
    steps = [("qkv", d, qkv, "rmsnorm"), ("o", d, o, "quant"), ("gu", d, gu, "rmsnorm"), ("down", nf, down, "swiglu")]

    def one(name, k, ns, producer):
        if name in fused:
            return bytes_gemv_fused(k, ns, producer)
        prod = {"rmsnorm": bytes_rmsnorm_quant(1, k, False), "quant": bytes_quantize(1, k),
                "swiglu": bytes_swiglu_quant(1, k, False)}[producer]
        return prod + bytes_gemv_group(k, ns)
    if "gu_pair" in fused:  # gate/up on the norm's plane, writing the SwiGLU plane; down reads it
        plane = lambda k: k + 4 * (k // 32)  # noqa: E731
        pair = (bytes_rmsnorm_quant(1, d, False) + sum(n * (d // 32) * 34 for n in gu) + plane(d) + plane(nf)
                + bytes_gemv(down[0], nf))
        steps = steps[:2]
    else:
        pair = 0
    per_layer = sum(one(*st) for st in steps) + pair
    return L["layers"] * per_layer + one("head", d, [L["vocab"]], "rmsnorm")


def run_layers(torch, q8p, steps, warmup, dev, layer_count=LAYERS["layers"]):
    """Per layer: RMSNorm -> q/k/v (one grouped launch); quantize of the
    attention output -> o; RMSNorm -> gate/up (one grouped launch); SwiGLU of
    their outputs -> down.  Then the final norm and the LM head.  Timed three
    ways, each as one CUDA graph per token: the producers of LAYER_FUSED
    inside their consumer's launch (q8_0_gemv_fused) and the others as their
    own launches in mode 2 (the headline); every producer as its own launch
    (rmsnorm_quant / quantize_q8_0 / swiglu_quant, then the GEMV on the plane:
    8 launches per layer); every producer fused (4 launches per layer).
    Layer 0's matrices are drawn from the synthetic recipe; layers 1..27 are
    device copies of them (the same bytes, distinct memory, so every token
    streams all 7.5 GB from HBM)."""
    L = dict(LAYERS, layers=layer_count)
    d, nf, eps = L["d"], L["nf"], L["eps"]
    g = syn.rng(4, 0)
    shapes = [(n, k) for k, ns in layer_groups() for n in ns]  # q k v o gate up down
    host, head_h = stack_weights_host()
    layers = [[torch.from_numpy(w).to(dev) for w in host] for _ in range(L["layers"])]
    head = torch.from_numpy(head_h).to(dev)
    x = torch.from_numpy(syn.activations(g, 1, d)).to(dev)        # hidden state entering each layer
    attn = torch.from_numpy(syn.activations(g, 1, d)).to(dev)     # attention output
    h = torch.from_numpy(syn.activations(g, 1, d)).to(dev)        # hidden state after attention
    nw1, nw2, nwf = (torch.from_numpy(syn.uniform(g, d, 0.5, 1.5)).to(dev) for _ in range(3))
    pd, pf = q8p.empty_plane(1, d, dev), q8p.empty_plane(1, nf, dev)
    ys = [torch.empty((1, n), dtype=torch.float32, device=dev) for n, _ in shapes]
    logits = torch.empty(L["vocab"], dtype=torch.float32, device=dev)
    cap = torch.cuda.Stream(dev)
    P_Q, P_R, P_S = q8p.PRODUCER_QUANT, q8p.PRODUCER_RMSNORM, q8p.PRODUCER_SWIGLU

    def token(fuse):
        """One token's launches; `fuse` = the producers computed inside their
        consumer's launch, of {"qkv", "o", "gu", "down", "head"}, or "gu_pair"
        (gate/up with the SwiGLU plane written by its epilogue)."""
        c = []
        for wq, wk, wv, wo, wg, wu, wd in layers:
            qkv = [(wq, L["q"], ys[0]), (wk, L["kv"], ys[1]), (wv, L["kv"], ys[2])]
            gu = [(wg, nf, ys[4]), (wu, nf, ys[5])]
            c += ([q8p.q8_0_gemv_fused(qkv, d, P_R, x[0], None, nw1, eps, stream=cap, bind=True)] if "qkv" in fuse
                  else [q8p.rmsnorm_quant(x, nw1, eps, None, *pd, stream=cap, bind=True),
                        q8p.q8_0_gemv_grouped(qkv, d, *pd, stream=cap, bind=True)])
            c += ([q8p.q8_0_gemv_fused([(wo, d, ys[3])], d, P_Q, attn[0], stream=cap, bind=True)] if "o" in fuse
                  else [q8p.quantize_q8_0(attn, *pd, stream=cap, bind=True),
                        q8p.q8_0_gemv(wo, d, d, *pd, ys[3], stream=cap, bind=True)])
            if "gu_pair" in fuse:  # SwiGLU + quantize in the gate/up launch's epilogue, down on its plane
                c += [q8p.rmsnorm_quant(h, nw2, eps, None, *pd, stream=cap, bind=True),
                      q8p.q8_0_gemv_gate_up(wg, wu, nf, d, *pf, qs=pd[0], ds=pd[1], stream=cap, bind=True),
                      q8p.q8_0_gemv(wd, d, nf, *pf, ys[6], stream=cap, bind=True)]
                continue
            c += ([q8p.q8_0_gemv_fused(gu, d, P_R, h[0], None, nw2, eps, stream=cap, bind=True)] if "gu" in fuse
                  else [q8p.rmsnorm_quant(h, nw2, eps, None, *pd, stream=cap, bind=True),
                        q8p.q8_0_gemv_grouped(gu, d, *pd, stream=cap, bind=True)])
            c += ([q8p.q8_0_gemv_fused([(wd, d, ys[6])], nf, P_S, ys[4][0], ys[5][0], stream=cap, bind=True)]
                  if "down" in fuse else
                  [q8p.swiglu_quant(ys[4], ys[5], None, *pf, stream=cap, bind=True),
                   q8p.q8_0_gemv(wd, d, nf, *pf, ys[6], stream=cap, bind=True)])
        c += ([q8p.q8_0_gemv_fused([(head, L["vocab"], logits)], d, P_R, x[0], None, nwf, eps, stream=cap,
                                   bind=True)] if "head" in fuse
              else [q8p.rmsnorm_quant(x, nwf, eps, None, *pd, stream=cap, bind=True),
                    q8p.q8_0_gemv(head, L["vocab"], d, *pd, logits, stream=cap, bind=True)])
        return c

    variants = {"mixed": token(LAYER_FUSED), "two": token(()), "fused": token(("qkv", "o", "gu", "down", "head"))}
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, calls in variants.items():
        cap.wait_stream(stream)
        for _ in range(max(1, warmup)):  # eager, outside the capture
            for c in calls:
                c()
        q8p.q8_check()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for c in calls:
                c()
        stream.wait_stream(cap)
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, steps)
        t0.record(stream)
        for _ in range(steps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        res[name] = t0.elapsed_time(t1) / steps
        del graph
    return dict(ms=res["mixed"], ms_two=res["two"], ms_fused=res["fused"],
                launches=len(variants["mixed"]), launches_two=len(variants["two"]),
                launches_fused=len(variants["fused"]),
                weight_bytes=sum(w.numel() for w in layers[0]) * L["layers"] + head.numel())


# ---------------------------------------------------------------------------
# layer-stack prefill / small-batch sweep: every projection of the 28-layer
# stack and the LM head through q8_0_gemm at T tokens
# ---------------------------------------------------------------------------
STACK_TOKENS = (16, 512, 2048, 3325)


_STACK_HOST = {}


def stack_weights_host():
    """Layer 0's seven projection blobs and the LM head blob (host, generated once)."""
    if not _STACK_HOST:
        L = LAYERS
        shapes = [(n, k) for k, ns in layer_groups() for n in ns]  # q k v o gate up down
        _STACK_HOST["layer"] = [syn.q8_0_weights(syn.rng(4, 0, i), n, k)[0] for i, (n, k) in enumerate(shapes)]
        _STACK_HOST["head"] = syn.q8_0_weights(syn.rng(4, 0, len(shapes)), L["vocab"], L["d"])[0]
    return _STACK_HOST["layer"], _STACK_HOST["head"]


def stack_shapes():
    """(name, rows n, width k) of one layer's projections, in call order."""
    L = LAYERS
    d, nf = L["d"], L["nf"]
    return [("q", L["q"], d), ("k", L["kv"], d), ("v", L["kv"], d), ("o", d, d), ("gate", nf, d), ("up", nf, d),
            ("down", d, nf)]


def bytes_stack_call(t, n, k):
    # weights, the plane rows read, the f32 outputs
    return n * (k // 32) * 34 + t * (k + 4 * (k // 32)) + 4 * t * n


def run_stack_tokens(torch, q8p, reps, warmup, dev, tokens=STACK_TOKENS, layer_count=LAYERS["layers"]):
    """Per token count T: one pass = every projection of every layer and the
    LM head, each one q8_0_gemm call (28 x 7 + 1 = 197 calls) on a q8_0 plane
    of T tokens per activation width (3584 and 18944), quantized on the GPU
    from seeded f32 ~N(0,1).  Timed two ways: `reps` whole passes between one
    pair of CUDA events (the stack time), and one pass with events around
    every call (per-shape time, averaged over the layers).  Layers 1..27 are
    device copies of layer 0's matrices (distinct memory; 7.5 GB of weights
    per pass)."""
    L = LAYERS
    d, nf, V = L["d"], L["nf"], L["vocab"]
    shapes = stack_shapes()
    host, head_h = stack_weights_host()
    layers = [[torch.from_numpy(w).to(dev) for w in host] for _ in range(layer_count)]
    head = torch.from_numpy(head_h).to(dev)
    tmax = max(tokens)
    g = syn.rng(4, 1)
    planes = {}
    for k in (d, nf):
        x = torch.from_numpy(syn.activations(g, tmax, k)).to(dev)
        planes[k] = q8p.empty_plane(q8p.q8_plane_rows(tmax), k, dev)
        q8p.quantize_q8_0(x, *planes[k])
        del x
    all_shapes = shapes + [("head", V, d)]
    ws_bytes = max(q8p.q8_0_gemm_workspace_bytes(n, T, k) for T in tokens for (_, n, k) in all_shapes)
    ws = torch.empty(max(ws_bytes, 1024), dtype=torch.uint8, device=dev)
    Y = torch.empty(tmax * V, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for T in tokens:
        calls = []
        for lw in layers:
            for (name, n, k), w in zip(shapes, lw):
                calls.append((name, q8p.q8_0_gemm(w, n, k, *planes[k], T, Y, workspace=ws, bind=True)))
        calls.append(("head", q8p.q8_0_gemm(head, V, d, *planes[d], T, Y, workspace=ws, bind=True)))
        for _ in range(max(1, warmup // 3)):
            for _, c in calls:
                c()
        q8p.q8_check()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, 8 * len(calls))
        t0.record(stream)
        for _ in range(reps):
            for _, c in calls:
                c()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        stack_ms = t0.elapsed_time(t1) / reps
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
        hold_device(torch, 8 * len(calls))
        for (_, c), (a, b) in zip(calls, evs):
            a.record(stream)
            c()
            b.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        per = {}
        for (name, _), (a, b) in zip(calls, evs):
            per.setdefault(name, []).append(a.elapsed_time(b))
        out[T] = dict(stack_ms=stack_ms, per_ms={nm: statistics.mean(v) for nm, v in per.items()}, reps=reps)
    # at T <= 16 the same pass with the projections of one activation grouped:
    # q, k, v one launch, gate and up one launch (4 launches per layer + head)
    for T in [T for T in tokens if T <= q8p.GEMV_MAX_TOKENS]:
        Yg = [torch.empty(T * n, dtype=torch.float32, device=dev) for (_, n, _) in shapes]
        calls = []
        for lw in layers:
            pj = [(w, n, y) for ((_, n, _), w, y) in zip(shapes, lw, Yg)]
            calls.append(q8p.q8_0_gemv_batched_grouped(pj[0:3], d, *planes[d], T, bind=True))
            calls.append(q8p.q8_0_gemm(lw[3], d, d, *planes[d], T, Y, workspace=ws, bind=True))
            calls.append(q8p.q8_0_gemv_batched_grouped(pj[4:6], d, *planes[d], T, bind=True))
            calls.append(q8p.q8_0_gemm(lw[6], d, nf, *planes[nf], T, Y, workspace=ws, bind=True))
        calls.append(q8p.q8_0_gemm(head, V, d, *planes[d], T, Y, workspace=ws, bind=True))
        for _ in range(max(1, warmup // 3)):
            for c in calls:
                c()
        q8p.q8_check()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch, 8 * len(calls))
        t0.record(stream)
        for _ in range(reps):
            for c in calls:
                c()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        q8p.q8_check()
        out[T]["stack_ms_grouped"] = t0.elapsed_time(t1) / reps
        out[T]["grouped_calls"] = len(calls)
        del Yg
    # the same passes on weights prepared once per matrix (f16 codes + d_w,
    # q8_0_gemm_prepare_weights outside the timed region), for the token counts
    # that take the tcgen05 GEMM
    big = [T for T in tokens if q8p.q8_0_gemm_prepared_workspace_bytes(d, T, d) > 0]
    if big:
        prep = [[q8p.q8_0_gemm_prepare_weights(w, n, k) for (_, n, k), w in zip(shapes, lw)] for lw in layers]
        head_p = q8p.q8_0_gemm_prepare_weights(head, V, d)
        wsb = max(q8p.q8_0_gemm_prepared_workspace_bytes(n, T, k) for T in big for (_, n, k) in all_shapes)
        wsp = torch.empty(max(wsb, 1024), dtype=torch.uint8, device=dev)
        for T in big:
            calls = [q8p.q8_0_gemm_prepared(None, wp, n, k, *planes[k], T, Y, workspace=wsp, bind=True)
                     for pl in prep for (_, n, k), wp in zip(shapes, pl)]
            calls.append(q8p.q8_0_gemm_prepared(None, head_p, V, d, *planes[d], T, Y, workspace=wsp, bind=True))
            for _ in range(max(1, warmup // 3)):
                for c in calls:
                    c()
            q8p.q8_check()
            torch.cuda.synchronize(dev)
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_device(torch, 8 * len(calls))
            t0.record(stream)
            for _ in range(reps):
                for c in calls:
                    c()
            t1.record(stream)
            torch.cuda.synchronize(dev)
            q8p.q8_check()
            out[T]["stack_ms_prepared"] = t0.elapsed_time(t1) / reps
        del prep, head_p, wsp
    return out


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_decode_sample(budget_s):
    import oracle

    xs, ws = decode_inputs()
    reps, t0 = 0, time.perf_counter()
    while True:
        planes = {k: oracle.quantize(v) for k, v in xs.items()}
        for (n, k), wb in zip(DECODE_SHAPES, ws):
            oracle.gemv(wb, n, k, *planes[k])
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return dict(value=decode_bytes() * reps / el / 1e9, unit="GB/s", cores=oracle.num_threads(), kind="oracle",
                sample=f"{reps} full decode steps (quantize + 3 GEMVs of the sweep) in {el:.1f} s")


def _oracle_time(fn, budget_s):
    """Mean wall time of fn() over repeated calls filling about budget_s (at least one call)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / reps, reps, el


def oracle_leg_samples(budget_s, legs):
    """cpu_baseline objects of the non-headline legs: the oracle as it stands,
    timed on the host cores, each on the leg's own inputs or a stated slice
    of them, the rate extrapolated linearly to the leg's whole workload."""
    import oracle

    cores = oracle.num_threads()
    out = {}

    def obj(value, unit, sample):
        return dict(value=round(value, 4), unit=unit, cores=cores, kind="oracle", sample=sample)

    if "tiny" in legs:
        n, k = TINY["n"], TINY["k"]
        x, w = tiny_inputs()
        dt, reps, el = _oracle_time(lambda: oracle.gemv(w, n, k, *oracle.quantize(x)), budget_s)
        out["tiny"] = obj(bytes_gemv_fused(k, [n], "quant") / dt / 1e9, "GB/s",
                          f"{reps} full steps (quantize 1x{k} + GEMV {n}x{k}) in {el:.1f} s")
    if "shared" in legs:
        d, ns, eps = SHARED["d"], SHARED["ns"], SHARED["eps"]
        g = syn.rng(2, 0)
        x, nw = syn.activations(g, 1, d), syn.uniform(g, d, 0.5, 1.5)
        wb = [syn.q8_0_weights(syn.rng(2, 1 + i), n, d)[0] for i, n in enumerate(ns)]

        def shared_step():
            y = oracle.rmsnorm(x, nw, eps).astype(np.float32)
            qs, ds = oracle.quantize(y)
            for w, n in zip(wb, ns):
                oracle.gemv(w, n, d, qs, ds)
        dt, reps, el = _oracle_time(shared_step, budget_s)
        out["shared"] = obj(bytes_shared(fused=True) / dt / 1e9, "GB/s",
                            f"{reps} full steps (RMSNorm, quantize, 4 GEMVs) in {el:.1f} s")
    if "prefill" in legs:
        T, d, nf, eps = PREFILL["tokens"], PREFILL["d"], PREFILL["nf"], PREFILL["eps"]
        x, w, wg, wu, wd = prefill_inputs()
        ts = 4
        ti = np.arange(ts)

        def chain():
            qa = oracle.quantize(oracle.rmsnorm(x[:ts], w, eps).astype(np.float32))
            gt = oracle.gemm(wg, nf, d, *qa, t_idx=ti)[0].astype(np.float32)
            ut = oracle.gemm(wu, nf, d, *qa, t_idx=ti)[0].astype(np.float32)
            qb = oracle.quantize(oracle.swiglu(gt, ut).astype(np.float32))
            oracle.gemm(wd, d, nf, *qb, t_idx=ti)
        dt, reps, el = _oracle_time(chain, budget_s)
        ops = 3 * ops_gemm(ts, nf, d)
        out["prefill"] = obj(ops / dt / 1e12, "TOPS",
                             f"{reps} chains on the first {ts} of {T} tokens (rmsnorm, gate/up, swiglu, down, all rows) "
                             f"in {el:.1f} s; int8-op rate extrapolated linearly to {T} tokens "
                             f"(chain ~{dt * T / ts:.0f} s)")
    if "layers" in legs:
        L = LAYERS
        d, nf, eps = L["d"], L["nf"], L["eps"]
        shapes = stack_shapes()
        wb, head = stack_weights_host()
        g = syn.rng(4, 0)
        x, attn, h = (syn.activations(g, 1, d) for _ in range(3))
        nw = syn.uniform(g, d, 0.5, 1.5)
        hrows = L["vocab"] // 16
        head_s = head[: hrows * (d // 32) * 34]

        def layer():
            qa = oracle.quantize(oracle.rmsnorm(x, nw, eps).astype(np.float32))
            for (_, n, k), w in zip(shapes[:3], wb[:3]):
                oracle.gemv(w, n, k, *qa)
            oracle.gemv(wb[3], d, d, *oracle.quantize(attn))
            qh = oracle.quantize(oracle.rmsnorm(h, nw, eps).astype(np.float32))
            gt = oracle.gemv(wb[4], nf, d, *qh)[0].astype(np.float32)[None]
            ut = oracle.gemv(wb[5], nf, d, *qh)[0].astype(np.float32)[None]
            oracle.gemv(wb[6], d, nf, *oracle.quantize(oracle.swiglu(gt, ut).astype(np.float32)))
        dl, rl, el1 = _oracle_time(layer, budget_s * 0.7)
        dh, rh, el2 = _oracle_time(lambda: oracle.gemv(head_s, hrows, d, *oracle.quantize(x)), budget_s * 0.3)
        tok = L["layers"] * dl + 16 * dh
        out["layers"] = obj(bytes_layer_stack(LAYER_FUSED) / tok / 1e9, "GB/s",
                            f"{rl} passes of one layer (producers + 7 GEMVs) in {el1:.1f} s and {rh} passes of the LM "
                            f"head's first {hrows} rows in {el2:.1f} s; extrapolated to {L['layers']} layers + the "
                            f"whole head (~{tok:.2f} s per token)")
    for T in legs.get("stack", ()):
        L = LAYERS
        d, V = L["d"], L["vocab"]
        shapes = stack_shapes() + [("head", V, d)]
        wl_, hd_ = stack_weights_host()
        wb = list(wl_) + [hd_]
        ts, rows = min(T, 4), 256
        g = syn.rng(4, 1)
        pl = {k: oracle.quantize(syn.activations(g, ts, k)) for k in (d, L["nf"])}
        ni = np.arange(rows)
        times = []
        for (_, n, k), w in zip(shapes, wb):
            dt, _, _ = _oracle_time(lambda: oracle.gemm(w, n, k, *pl[k], t_idx=np.arange(ts), n_idx=ni),
                                    budget_s / len(shapes))
            times.append(dt * (T / ts) * (n / rows))
        full = L["layers"] * sum(times[:-1]) + times[-1]
        ops = L["layers"] * sum(ops_gemm(T, n, k) for _, n, k in shapes[:-1]) + ops_gemm(T, V, d)
        byts = L["layers"] * sum(bytes_stack_call(T, n, k) for _, n, k in shapes[:-1]) + bytes_stack_call(T, V, d)
        samp = (f"each projection shape timed on {ts} tokens x its first {rows} rows, extrapolated linearly to "
                f"{T} tokens x all rows, 28 layers + LM head (~{full:.0f} s per pass)")
        out[f"stack_{T}"] = (obj(byts / full / 1e9, "GB/s", samp) if T <= 16 else obj(ops / full / 1e12, "TOPS", samp))
    if "small" in legs:
        n, k, t = SMALL["n"], SMALL["k"], SMALL["tokens"]
        w = syn.q8_0_weights(syn.rng(4, 1), n, k)[0]
        qs, ds = oracle.quantize(syn.activations(syn.rng(4, 0), t, k, sigma=1.5, outlier_frac=0.01))
        rows = 768
        dt, reps, el = _oracle_time(lambda: oracle.gemm(w, n, k, qs, ds, n_idx=np.arange(rows)), budget_s)
        out["small"] = obj(bytes_small(n, k, t) / (dt * n / rows) / 1e9, "GB/s",
                           f"{reps} passes over the first {rows} of {n} rows, {t} tokens, in {el:.1f} s; "
                           "extrapolated linearly to all rows")
    if "asym" in legs:
        n, k = ASYM["n"], ASYM["k"]
        w = syn.q4a_weights(syn.rng(5, 1), n, k)[0]
        qs, ds = oracle.quantize(syn.activations(syn.rng(5, 0), 1, k, sigma=1.5, outlier_frac=0.01))
        dt, reps, el = _oracle_time(lambda: oracle.q4a_gemv(w, n, k, qs, ds), budget_s)
        out["asym"] = obj(bytes_q4a_gemv(n, k) / dt / 1e9, "GB/s", f"{reps} full q4a_gemv calls in {el:.1f} s")
    return out


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    xs, ws = decode_inputs()
    t_full = []
    for _ in range(args.warmup):
        t0 = time.perf_counter()
        planes = {k: oracle.quantize(v) for k, v in xs.items()}
        for (n, k), wb in zip(DECODE_SHAPES, ws):
            oracle.gemv(wb, n, k, *planes[k])
        t_full.append(time.perf_counter() - t0)
    # Each timed step is the decode step on a prefix of every weight matrix's
    # rows, sized so that K steps take about a minute (all rows when K is small).
    frac = min(1.0, 60.0 / (args.steps * statistics.median(t_full)))
    rows = [max(1, int(frac * n)) for n, _ in DECODE_SHAPES]
    subs = [wb[: r * (k // 32) * 34] for wb, r, (_, k) in zip(ws, rows, DECODE_SHAPES)]
    step_bytes = (bytes_quantize(1, 7168) + bytes_quantize(1, 128) +
                  sum(bytes_gemv(r, k) for r, (_, k) in zip(rows, DECODE_SHAPES)))
    per = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        planes = {k: oracle.quantize(v) for k, v in xs.items()}
        for r, (_, k), wb in zip(rows, DECODE_SHAPES, subs):
            oracle.gemv(wb, r, k, *planes[k])
        per.append(time.perf_counter() - t0)
    tot = sum(per)
    value = step_bytes * args.steps / tot / 1e9
    sample = (f"{args.steps} decode steps of the sweep, each timed" if frac >= 1.0 else
              f"{args.steps} decode steps of the sweep on the first {rows} rows of each weight matrix "
              f"({100 * frac:.1f}% of the rows, bounded to ~60 s), each timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": decode_config(None),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def decode_config(copies):
    return {"workload": "decode GEMV sweep b=1: q8_0 quantize + Q8_0 GEMV (n,k) in {(12288,7168),(96,7168),(512,128)}",
            "activation": "f32 ~N(0,1.5), 1% outliers x20, seed 1", "weights": "Q8_0, d~U(0.002,0.02), q~U{-127..127}",
            "l2": (f"weights rotate through {copies} copies ({copies} x 94.4 MB > 4 x L2)" if copies else "n/a (CPU)"),
            "launch": ("timed steps replayed from a CUDA graph of one step per weight copy; per step the k = 7168 "
                       "pair is one q8_0_gemv_fused launch (quantize inside) and the k = 128 chain (quantize_q8_0 -> "
                       "q8_0_gemv) a parallel graph branch" if copies else "n/a (CPU)"),
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 6000 decode steps keep the timed region ~0.2 s long, so the clock sampler
    # (50 ms) sees it; the prefill chain runs steps // 6 times (~3.4 s)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--layer-count", type=int, default=LAYERS["layers"],
                    help="layers of the layer-stack leg (a shorter stack for profiling runs)")
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode", "prefill", "small", "asym", "shared", "layers", "tiny", "stack"],
                    help="decode and/or prefill legs (profiling runs select one)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--cpu-leg-budget", type=float, default=1.5,
                    help="seconds of oracle time for each other leg's cpu_baseline")
    ap.add_argument("--stack-tokens", default=",".join(str(t) for t in STACK_TOKENS),
                    help="token counts of the layer-stack sweep through q8_0_gemm")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import torch

    import int8_quantized_projection_gb300 as q8p
    from int8_quantized_projection_gb300 import build as b

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    if rank == 0:
        b.build()
    if world > 1:
        torch.distributed.barrier()
    q8p.lib()

    wl = args.workload
    stack_tokens = tuple(int(v) for v in args.stack_tokens.split(",") if v)
    cpu, cpu_legs = None, {}
    if rank == 0:  # oracle baselines before any GPU work is timed (host cores only)
        if wl in ("all", "decode"):
            cpu = oracle_decode_sample(args.cpu_budget)
        legs = {k: True for k in ("tiny", "shared", "small", "asym", "layers") if wl in ("all", k)}
        if wl == "all" and not args.no_prefill or wl == "prefill":
            legs["prefill"] = True
        if wl in ("all", "stack"):
            legs["stack"] = stack_tokens
        cpu_legs = oracle_leg_samples(args.cpu_leg_budget, legs)

    sampler = ClockSampler(gpu_smi_id(torch, dev))
    if world > 1:
        torch.distributed.barrier()
    dec = None
    if args.workload in ("all", "decode"):
        dec = run_decode(torch, q8p, args.steps, args.warmup, dev, sampler)

    pre = None
    if args.workload == "prefill" or (args.workload == "all" and not args.no_prefill):
        pre = run_prefill(torch, q8p, args.steps if dec is None else max(3, args.steps // 6), args.warmup, dev)

    small = None
    if args.workload in ("all", "small"):
        small = run_small(torch, q8p, args.steps if dec is None and pre is None else max(20, args.steps // 30),
                          args.warmup, dev)

    asym = None
    if args.workload in ("all", "asym"):
        asym = run_asym(torch, q8p, args.steps if args.workload == "asym" else max(20, args.steps // 30),
                        args.warmup, dev)

    shr = None
    if args.workload in ("all", "shared"):
        shr = run_shared(torch, q8p, args.steps if args.workload == "shared" else max(60, args.steps // 10),
                         args.warmup, dev)

    lay = None
    if args.workload in ("all", "layers"):
        lay = run_layers(torch, q8p, args.steps if args.workload == "layers" else max(10, args.steps // 200),
                         args.warmup, dev,
                         args.layer_count)

    tiny = None
    if args.workload in ("all", "tiny"):
        tiny = run_tiny(torch, q8p, args.steps, args.warmup, dev)

    stk = None
    if args.workload in ("all", "stack"):
        stk = run_stack_tokens(torch, q8p, 3 if args.workload == "all" else max(1, min(args.steps, 20)), args.warmup,
                               dev, stack_tokens, args.layer_count)

    if world > 1:  # every duration becomes the slowest rank's (same legs on every rank)
        vals = (([dec["ms"], dec["e2e_s"], dec["kern_ms"], dec["e2e_eager_s"], dec["e2e_serial_s"], dec["ms_two"],
                  dec["iso_ms"]] if dec else [])
                + (list(pre[0].values()) + list(pre[1].values()) + list(pre[2].values()) if pre else [])
                + ([small["us"], small["us_b2b"]] if small else []) + ([asym["us"], asym["us_b2b"]] if asym else [])
                + ([lay["ms"], lay["ms_two"], lay["ms_fused"]] if lay else [])
                + ([shr["us"], shr["us_two"]] if shr else [])
                + ([tiny["us"], tiny["us_two"]] if tiny else [])
                + ([v for T in sorted(stk) for v in [stk[T]["stack_ms"]] + [stk[T]["per_ms"][nm] for nm in
                                                                             sorted(stk[T]["per_ms"])]
                    + ([stk[T]["stack_ms_prepared"]] if "stack_ms_prepared" in stk[T] else [])
                    + ([stk[T]["stack_ms_grouped"]] if "stack_ms_grouped" in stk[T] else [])] if stk else []))
        red = max_over_ranks(torch, vals, dev)
        if dec:
            (dec["ms"], dec["e2e_s"], dec["kern_ms"], dec["e2e_eager_s"], dec["e2e_serial_s"], dec["ms_two"],
             dec["iso_ms"]) = red[:7]
            red = red[7:]
        if pre:
            n0, n1, n2 = len(pre[0]), len(pre[1]), len(pre[2])
            pre = (dict(zip(pre[0].keys(), red[:n0])), dict(zip(pre[1].keys(), red[n0:n0 + n1])),
                   dict(zip(pre[2].keys(), red[n0 + n1:n0 + n1 + n2])))
            red = red[n0 + n1 + n2:]
        if small:
            small["us"], small["us_b2b"] = red.pop(0), red.pop(0)
        if asym:
            asym["us"], asym["us_b2b"] = red.pop(0), red.pop(0)
        if lay:
            lay["ms"], lay["ms_two"], lay["ms_fused"] = red.pop(0), red.pop(0), red.pop(0)
        if shr:
            shr["us"], shr["us_two"] = red.pop(0), red.pop(0)
        if tiny:
            tiny["us"], tiny["us_two"] = red.pop(0), red.pop(0)
        if stk:
            for T in sorted(stk):
                stk[T]["stack_ms"] = red.pop(0)
                for nm in sorted(stk[T]["per_ms"]):
                    stk[T]["per_ms"][nm] = red.pop(0)
                if "stack_ms_prepared" in stk[T]:
                    stk[T]["stack_ms_prepared"] = red.pop(0)
                if "stack_ms_grouped" in stk[T]:
                    stk[T]["stack_ms_grouped"] = red.pop(0)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peaks = measured_peaks()
    line = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic"}
    if dec is not None:
        ms = dec["ms"]
        step_bytes = decode_bytes(fused=True)
        value = world * step_bytes * args.steps / (ms / 1e3) / 1e9
        big = bytes_gemv_fused(7168, [DECODE_SHAPES[0][0], DECODE_SHAPES[1][0]], "quant")
        achieved = big / (dec["kern_ms"] / 1e3) / 1e9
        line.update({
            "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms / args.steps, 5),
            "config": decode_config(dec["copies"]),
            "roofline": {"kernel": "q8_0_gemv_fused 12288x7168 + 96x7168, quantize inside (gemv_staged_kernel)",
                         "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                         "traffic": NCU_TRAFFIC_BYTES["gemv_fused 12288x7168+96x7168"],
                         "algorithmic_bytes": big, "avg_launch_us": round(dec["kern_ms"] * 1e3, 3),
                         "timing": "the fused GEMV alone, K launches back to back from CUDA graphs (weight copies "
                                   "in turn, programmatic dependent launch as in the step), CUDA events around them",
                         "isolated_launch_us": round(dec["iso_ms"] * 1e3, 3)},
            "two_launch": {"calls": "quantize_q8_0 (k = 7168) -> q8_0_gemv_grouped, the k = 128 chain unchanged",
                           "ms_per_step": round(dec["ms_two"], 5),
                           "gbs": round(world * decode_bytes() / (dec["ms_two"] / 1e3) / 1e9, 2)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * step_bytes * args.steps / dec["e2e_s"] / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": dec["h2d"], "d2h_bytes_per_step": dec["d2h"],
                    "launch": "per step: one CUDA graph replay (pinned-memory copy in, the library calls, copy out; "
                              "recorded once); consecutive steps on three device buffer sets and streams, so "
                              "independent steps overlap on the device (one step's copies and its launch's ramp and "
                              "tail under the others' kernels: this can exceed `value`, whose steps run one after "
                              "another on one stream); up to five steps in flight: the host reads step i-5's outputs "
                              "after enqueuing step i (six host buffers rotate)",
                    "steps_timed": dec["e2e_steps"],
                    "serial_value": round(world * step_bytes * args.steps / dec["e2e_serial_s"] / 1e9, 2),
                    "eager_value": round(world * step_bytes * args.steps / dec["e2e_eager_s"] / 1e9, 2)},
            "clocks": dec["clocks"],
            "gpu_launches": 3 * args.steps,
        })
    if pre is not None:
        T, d, nf = PREFILL["tokens"], PREFILL["d"], PREFILL["nf"]
        pre, pre_prep, pre_b2b = pre
        gemm_ms = pre["gemm_gate"] + pre["gemm_up"] + pre["gemm_down"]
        tops = 3 * ops_gemm(T, nf, d) / (gemm_ms / 1e3) / 1e12
        gemm_ms_p = pre_prep["gemm_gate"] + pre_prep["gemm_up"] + pre_prep["gemm_down"]
        tops_p = 3 * ops_gemm(T, nf, d) / (gemm_ms_p / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        pobj = {
            "workload": f"prefill chain T={T} d={d} nf={nf}: rmsnorm_quant, gate/up GEMM, swiglu_quant, down GEMM "
                        "(both producers in mode 2: the plane only, no f32 output)",
            "ms_per_chain": round(sum(v for k_, v in pre.items() if not k_.startswith("quantize_q8_0")), 4),
            "ms_per_chain_back_to_back": round(pre_b2b["chain"], 4),
            "back_to_back_timing": "chains issued back to back between one pair of CUDA events (programmatic "
                                       "dependent launch across every call); `ms_per_chain` adds the calls timed "
                                       "one at a time",
            "ms": {k: round(v, 4) for k, v in pre.items()},
            "gemm_tops": round(tops, 2), "unit": "int8 TOPS (2*T*N*K per GEMM)",
            "roofline_gemm": {"kernel": "q8_0_gemm (gemm_tc_kernel)", "bound": "tensor", "achieved": round(tops, 2),
                              "peak": peak, "unit": "TFLOP/s", "frac": round(tops / peak, 4),
                              "traffic": NCU_TRAFFIC_BYTES["gemm_tc 18944x3584 t=3325"],
                              "peak_note": f"sustained dense bf16/f16 tensor peak ({peaks['source']}); sm_103a has "
                                           "no int8 tcgen05 kind"},
            "quantize_gbs": {"rmsnorm_quant_mode2": round(bytes_rmsnorm_quant(T, d, False) / pre["rmsnorm_quant"] / 1e6,
                                                          1),
                             "swiglu_quant_mode2": round(bytes_swiglu_quant(T, nf, False) / pre["swiglu_quant"] / 1e6,
                                                         1),
                             "quantize_q8_0": round(bytes_quantize(T, d) /
                                                    pre["quantize_q8_0 (standalone, not in the chain)"] / 1e6, 1),
                             "timing": "each call bracketed by its own CUDA events (no overlap with its neighbours)",
                             "peak": peaks["hbm_gbs"],
                             "back_to_back": {
                                 "rmsnorm_quant_mode2": round(bytes_rmsnorm_quant(T, d, False)
                                                              / pre_b2b["rmsnorm_quant"] / 1e6, 1),
                                 "swiglu_quant_mode2": round(bytes_swiglu_quant(T, nf, False)
                                                             / pre_b2b["swiglu_quant"] / 1e6, 1),
                                 "quantize_q8_0": round(bytes_quantize(T, d) / pre_b2b["quantize_q8_0"] / 1e6, 1),
                                 "us": {k: round(1e3 * v, 2) for k, v in pre_b2b.items() if not k.startswith("chain")},
                                 "timing": "20 calls back to back between one pair of CUDA events (programmatic "
                                           "dependent launch: each call's start overlaps the previous one's tail), "
                                           "f32 inputs rotating over copies that together exceed L2"}},
            "l2": "step working set ~1.2 GB > L2",
            "prepared_weights": {
                "calls": "the same chain with q8_0_gemm_prepared: each weight matrix widened to f16 once "
                         "(q8_0_gemm_prepare_weights, outside the timed region), so a GEMM call runs its "
                         "activation pre-pass and the tcgen05 kernel only",
                "ms_per_chain": round(sum(pre_prep.values()), 4),
                "ms_per_chain_back_to_back": round(pre_b2b["chain_prepared"], 4),
                "ms": {k: round(v, 4) for k, v in pre_prep.items()},
                "gemm_tops": round(tops_p, 2), "frac": round(tops_p / peak, 4)},
        }
        if dec is None:  # prefill-only run: the GEMM throughput (all replicas) is the headline
            line.update({"value": round(world * pobj["gemm_tops"], 2), "unit": "TOPS",
                         "ms_per_step": pobj["ms_per_chain"],
                         "config": {"workload": pobj["workload"], "l2": pobj["l2"], "parallelism": "replicas"},
                         "roofline": pobj["roofline_gemm"], "gpu_launches": 5 * args.steps})
        pobj["cpu_baseline"] = cpu_legs.get("prefill")
        line["prefill"] = pobj
    if small is not None:
        n, k, t = SMALL["n"], SMALL["k"], SMALL["tokens"]
        gbs = bytes_small(n, k, t) / (small["us"] / 1e6) / 1e9
        sobj = {"workload": f"small-batch decode: q8_0_gemv_batched {n}x{k}, t={t} tokens, weights read once",
                "us_per_call": round(small["us"], 2), "gbs": round(gbs, 1),
                "us_back_to_back": round(small["us_b2b"], 2),
                "gbs_back_to_back": round(bytes_small(n, k, t) / (small["us_b2b"] / 1e6) / 1e9, 1),
                "roofline": {"kernel": "q8_0_gemv_batched (gemv_small_kernel)", "bound": "hbm",
                             "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(gbs / peaks["hbm_gbs"], 4),
                             "traffic": NCU_TRAFFIC_BYTES["gemv_small 12288x7168 t=16"],
                             "algorithmic_bytes": bytes_small(n, k, t)},
                "l2": f"weights rotate through {small['copies']} copies (> 4 x L2)"}
        if dec is None and pre is None:
            line.update({"value": round(world * sobj["gbs"], 1), "unit": "GB/s",
                         "ms_per_step": round(small["us"] / 1e3, 5),
                         "config": {"workload": sobj["workload"], "l2": sobj["l2"], "parallelism": "replicas"},
                         "roofline": sobj["roofline"], "gpu_launches": 2 * args.steps})
        sobj["cpu_baseline"] = cpu_legs.get("small")
        line["small_batch"] = sobj
    if asym is not None:
        n, k = ASYM["n"], ASYM["k"]
        gbs = bytes_q4a_gemv(n, k) / (asym["us"] / 1e6) / 1e9
        aobj = {"workload": f"asymmetric 4-bit weights (d*nib - m, min term from the plane's ssum): q4a_gemv "
                            f"{n}x{k}, batch 1",
                "us_per_call": round(asym["us"], 2), "gbs": round(gbs, 1),
                "us_back_to_back": round(asym["us_b2b"], 2),
                "gbs_back_to_back": round(bytes_q4a_gemv(n, k) / (asym["us_b2b"] / 1e6) / 1e9, 1),
                "roofline": {"kernel": "q4a_gemv (gemv_staged_kernel<FmtQ4A>)", "bound": "hbm", "achieved": round(gbs, 1),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                             "traffic": NCU_TRAFFIC_BYTES["gemv_staged_q4a 12288x7168"],
                             "algorithmic_bytes": bytes_q4a_gemv(n, k)},
                "l2": f"weights rotate through {asym['copies']} copies (> 4 x L2)"}
        if args.workload == "asym":
            line.update({"value": round(world * aobj["gbs"], 1), "unit": "GB/s",
                         "ms_per_step": round(asym["us"] / 1e3, 5),
                         "config": {"workload": aobj["workload"], "l2": aobj["l2"], "parallelism": "replicas"},
                         "roofline": aobj["roofline"], "gpu_launches": 2 * args.steps})
        aobj["cpu_baseline"] = cpu_legs.get("asym")
        line["asym_gemv"] = aobj
    if shr is not None:
        byts = bytes_shared(fused=True)
        gbs = byts / (shr["us"] / 1e6) / 1e9
        byts2 = bytes_shared()
        sobj2 = {"workload": f"shared-activation decode b=1: RMSNorm (d={SHARED['d']}) + q8_0 quantize feeding "
                             f"q/k/v/gate {'/'.join(str(n) for n in SHARED['ns'])} in one q8_0_gemv_fused launch "
                             "(the norm computed inside the grouped GEMV)",
                 "us_per_step": round(shr["us"], 2), "gbs": round(gbs, 1), "algorithmic_bytes": byts,
                 "launches_per_step": 1,
                 "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": round(gbs / peaks["hbm_gbs"], 4)},
                 "two_launch": {"calls": "rmsnorm_quant (mode 2) -> q8_0_gemv_grouped",
                                "us_per_step": round(shr["us_two"], 2),
                                "gbs": round(byts2 / (shr["us_two"] / 1e6) / 1e9, 1), "algorithmic_bytes": byts2,
                                "launches_per_step": 2},
                 "launch": f"CUDA graphs of {shr['per_graph']} steps (the {shr['copies']} weight copies in turn, "
                           "> 4 x L2), replayed; programmatic dependent launch between steps, as the decode step"}
        if args.workload == "shared":
            line.update({"value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": round(shr["us"] / 1e3, 5),
                         "config": {"workload": sobj2["workload"], "l2": f"{shr['copies']} weight copies > 4 x L2",
                                    "parallelism": "replicas"},
                         "roofline": sobj2["roofline"], "gpu_launches": shr["steps"]})
        sobj2["cpu_baseline"] = cpu_legs.get("shared")
        line["shared_activation"] = sobj2
    if lay is not None:
        L = dict(LAYERS, layers=args.layer_count)
        byts = bytes_layer_stack(LAYER_FUSED, args.layer_count)
        gbs = byts / (lay["ms"] / 1e3) / 1e9
        byts2 = bytes_layer_stack((), args.layer_count)
        byts3 = bytes_layer_stack(("qkv", "o", "gu", "down", "head"), args.layer_count)
        lobj = {"workload": f"layer-stack decode b=1: {L['layers']} layers (d={L['d']}, nf={L['nf']}; q {L['q']}, "
                            f"k/v {L['kv']}, o, gate/up, down) + LM head {L['vocab']}x{L['d']}; per layer RMSNorm "
                            "-> grouped q/k/v and quantize -> o inside their GEMV launch (q8_0_gemv_fused), "
                            "rmsnorm_quant -> gate/up with SwiGLU + quantize in its epilogue (q8_0_gemv_gate_up) -> "
                            "down on that plane; the final RMSNorm inside the LM head's launch",
                "ms_per_token": round(lay["ms"], 4), "tokens_per_s": round(1e3 / lay["ms"], 1),
                "gbs": round(gbs, 1), "algorithmic_bytes": byts, "weight_bytes": lay["weight_bytes"],
                "launches_per_token": lay["launches"],
                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(gbs / peaks["hbm_gbs"], 4)},
                "two_launch": {"calls": "every producer as its own launch (mode 2), then the GEMV on its plane",
                               "ms_per_token": round(lay["ms_two"], 4),
                               "gbs": round(byts2 / (lay["ms_two"] / 1e3) / 1e9, 1), "algorithmic_bytes": byts2,
                               "launches_per_token": lay["launches_two"]},
                "all_fused": {"calls": "every producer inside its GEMV launch (q8_0_gemv_fused)",
                              "ms_per_token": round(lay["ms_fused"], 4),
                              "gbs": round(byts3 / (lay["ms_fused"] / 1e3) / 1e9, 1), "algorithmic_bytes": byts3,
                              "launches_per_token": lay["launches_fused"]},
                "launch": f"one CUDA graph per token, replayed; layers 1..{L['layers'] - 1} are device copies of layer "
                          f"0's matrices (distinct memory: {lay['weight_bytes'] / 1e9:.2f} GB streamed per token, > L2)"}
        if args.workload == "layers":
            line.update({"value": round(world * gbs, 1), "unit": "GB/s", "ms_per_step": lobj["ms_per_token"],
                         "config": {"workload": lobj["workload"],
                                    "l2": f"{lay['weight_bytes'] / 1e9:.2f} GB of weights per token > L2",
                                    "parallelism": "replicas"},
                         "roofline": lobj["roofline"], "gpu_launches": lay["launches"] * args.steps})
        lobj["cpu_baseline"] = cpu_legs.get("layers")
        line["layer_stack"] = lobj
    if tiny is not None:
        n, k = TINY["n"], TINY["k"]
        tbytes = bytes_gemv_fused(k, [n], "quant")
        gbs = tbytes / (tiny["us"] / 1e6) / 1e9
        tobj = {"workload": f"tiny GEMV b=1: q8_0 quantize of 1x{k} inside the {n}x{k} q8_0_gemv_fused launch "
                            "(weights d~U(0.002,0.02), activation f32 ~N(0,1), seed 0)",
                "us_per_step": round(tiny["us"], 3), "gbs": round(gbs, 2), "algorithmic_bytes": tbytes,
                "launches_per_step": 1,
                "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(gbs / peaks["hbm_gbs"], 5),
                             "note": "141 KB per step: bound by one launch's latency, not by bandwidth"},
                "two_launch": {"calls": "quantize_q8_0 -> q8_0_gemv", "us_per_step": round(tiny["us_two"], 3),
                               "gbs": round(bytes_tiny() / (tiny["us_two"] / 1e6) / 1e9, 2),
                               "algorithmic_bytes": bytes_tiny()},
                "launch": f"CUDA graphs of up to 600 steps replayed; weights rotate through {tiny['copies']} copies "
                          "(> 4 x L2)",
                "cpu_baseline": cpu_legs.get("tiny")}
        if args.workload == "tiny":
            line.update({"value": round(world * gbs, 2), "unit": "GB/s", "ms_per_step": round(tiny["us"] / 1e3, 6),
                         "config": {"workload": tobj["workload"], "l2": tobj["launch"], "parallelism": "replicas"},
                         "roofline": tobj["roofline"], "gpu_launches": args.steps,
                         "cpu_baseline": tobj["cpu_baseline"]})
        line["tiny"] = tobj
    if stk is not None:
        L = dict(LAYERS, layers=args.layer_count)
        shapes = stack_shapes() + [("head", L["vocab"], L["d"])]
        sw = {}
        for T in sorted(stk):
            r = stk[T]
            ops = L["layers"] * sum(ops_gemm(T, n, k) for _, n, k in shapes[:-1]) + ops_gemm(T, *shapes[-1][1:])
            byts = (L["layers"] * sum(bytes_stack_call(T, n, k) for _, n, k in shapes[:-1])
                    + bytes_stack_call(T, *shapes[-1][1:]))
            per = {}
            for nm, n, k in shapes:
                ms_ = r["per_ms"][nm]
                per[f"{nm} {n}x{k}"] = {"ms": round(ms_, 4), "tops": round(ops_gemm(T, n, k) / ms_ / 1e9, 2),
                                        "gbs": round(bytes_stack_call(T, n, k) / ms_ / 1e6, 1)}
            tops = ops / (r["stack_ms"] / 1e3) / 1e12
            gbs = byts / (r["stack_ms"] / 1e3) / 1e9
            if T <= 16:
                roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs / peaks["hbm_gbs"], 4)}
            else:
                roof = {"bound": "tensor", "achieved": round(tops, 2), "peak": peaks["bf16_tflops_sustained"],
                        "unit": "TFLOP/s", "frac": round(tops / peaks["bf16_tflops_sustained"], 4),
                        "peak_note": "sustained dense bf16/f16 tensor peak; the int8 codes run on kind::f16 "
                                     "(sm_103a has no int8 tcgen05 kind)"}
            sw[str(T)] = {"tokens": T, "ms_per_pass": round(r["stack_ms"], 4), "tops": round(tops, 2),
                          "gbs": round(gbs, 1), "int8_ops": ops, "algorithmic_bytes": byts, "roofline": roof,
                          "per_shape": per, "cpu_baseline": cpu_legs.get(f"stack_{T}"), "passes_timed": r["reps"]}
            if "stack_ms_prepared" in r:
                tp = ops / (r["stack_ms_prepared"] / 1e3) / 1e12
                sw[str(T)]["prepared_weights"] = {
                    "ms_per_pass": round(r["stack_ms_prepared"], 4), "tops": round(tp, 2),
                    "frac": round(tp / peaks["bf16_tflops_sustained"], 4),
                    "calls": "q8_0_gemm_prepared on weights widened once per matrix (outside the timed region)"}
            if "stack_ms_grouped" in r:
                gg = byts / (r["stack_ms_grouped"] / 1e3) / 1e9
                sw[str(T)]["grouped"] = {
                    "ms_per_pass": round(r["stack_ms_grouped"], 4), "gbs": round(gg, 1),
                    "frac": round(gg / peaks["hbm_gbs"], 4), "launches": r["grouped_calls"],
                    "calls": "q8_0_gemv_batched_grouped for q/k/v and for gate/up of each layer, q8_0_gemm for o, "
                             "down and the head"}
        sobj3 = {"workload": f"layer-stack sweep through q8_0_gemm: {L['layers']} layers x (q {L['q']}, k/v {L['kv']}, "
                             f"o {L['d']}, gate/up {L['nf']} at k={L['d']}; down {L['d']} at k={L['nf']}) + LM head "
                             f"{L['vocab']}x{L['d']}, one call per projection ({7 * L['layers'] + 1} calls per pass) on "
                             "one q8_0 plane of T tokens per width",
                 "tokens": sw,
                 "launch": "calls issued eagerly behind a device-side sleep; per-shape times from a second pass with "
                           "CUDA events around every call (mean over layers); 7.5 GB of weights per pass (> L2)"}
        if args.workload == "stack":
            top = sw[str(max(stk))]
            line.update({"value": round(world * top["tops"], 2), "unit": "TOPS", "ms_per_step": top["ms_per_pass"],
                         "config": {"workload": sobj3["workload"] + f", T={max(stk)}",
                                    "l2": "7.5 GB of weights per pass > L2", "parallelism": "replicas"},
                         "roofline": top["roofline"], "cpu_baseline": top["cpu_baseline"]})
        line["layer_stack_tokens"] = sobj3
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
