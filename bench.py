#!/usr/bin/env python3
"""Decode-step benchmark of the Q4_0 x Q8_0 GEMV path with fused RMSNorm -> Q8_0.

One step = one batch-1 decode pass of an 8B-shaped Llama layer stack's
projections: fused RMSNorm*gamma -> Q8_0 (or plain Q8_0) for each activation,
then one GEMV per projection (q, k, v, o, gate, up, down, vocab head).  The
weights (419 MB of Q4_0 per step) exceed the 129 MB L2, so every step streams
them from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  ``value`` is the step's algorithmic bytes (weights,
activations, outputs) over device time with inputs resident; ``e2e`` repeats
the step through the same C-ABI calls with the step's inputs copied from
pinned host memory and all outputs stored into pinned host memory inside
the timed region.  The
step is replayed from a CUDA graph (one graph per input set).  ``roofline``
is the GEMV kernel's achieved bandwidth from per-launch CUDA events; the peak
is the measured copy bandwidth of this GPU model.  ``cpu_baseline`` times the
CPU oracle on a bounded sample.  ``--impl reference`` times that oracle alone
as the reference arm.

Multi-GPU: replicas only (each rank runs the whole step on its own GPU; the
product shards with no exchange); the per-rank time is max-reduced.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_decode_gemv_rms_gb300 import synth, workloads  # noqa: E402

METRIC = "Q4_0×Q8_0 GEMV HBM GB/s (fraction of GB300 peak) and µs/call at batch 1"
UNIT = "GB/s"
N_INPUT_SETS = 4
FUSED_SEG_MAX_K = 16384     # the segment-layout fused kernel stages x and gamma whole
# The fused route fuses groups up to this K and splits larger ones.  Measured on GB300: at K = 14336
# every CTA quantizing all 448 blocks costs 14.7 us per call against 7.6 us for the split GEMV, and the
# step takes 90.4 us with down fused against 85.1 us with down split.
FUSED_ROUTE_MAX_K = 8192
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0}, "fallback"


def source_hash(*paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_file: str, workload: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or
    None when the summary is missing, was taken on a different source, or on
    another workload (the per-launch bytes belong to the captured shapes)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel_file}:{workload}")
    if not e or e.get("source_sha") != source_hash(os.path.join("quantized_decode_gemv_rms_gb300", "csrc",
                                                                 kernel_file)):
        return None
    return e


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.dev = device_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        win = [r for r in rows if self.t0 is not None and self.t0 - 0.15 <= r[0] <= (self.t1 or r[0]) + 0.15]
        use = win if win else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for i, n in enumerate(names):
                if r[3][5 + i].lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in use]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if win else "whole run (no sample fell inside the timed region)"}


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- workload bytes
def step_bytes(wl):
    """Algorithmic bytes of one decode step -- what it must move at least once:
    every projection's Q4_0 weights and fp32 outputs, every fp32 activation
    vector and every gamma.  The same count serves the fused and the unfused
    route (the unfused one also writes and reads the Q8_0 vectors, ~0.01%)."""
    total = 0
    for m in wl.matrices:
        total += workloads.q4_0_bytes(m.rows, m.cols) + 4 * m.rows
    for tag, K in wl.activations.items():
        norm = any(m.source == f"norm:{tag}" for m in wl.matrices)
        total += 4 * K + (4 * K if norm else 0)
    return total


def fused_launch_bytes(m):
    """Algorithmic bytes of one fused norm+GEMV launch: W, x, gamma (if any), y."""
    norm = m.source.startswith("norm:")
    return workloads.q4_0_bytes(m.rows, m.cols) + 4 * m.cols * (2 if norm else 1) + 4 * m.rows


def activation_kinds(wl):
    kinds = {}
    for m in wl.matrices:
        kind, tag = m.source.split(":", 1)
        kinds[tag] = kind
    return kinds


# ---------------------------------------------------------------- CPU oracle leg
def oracle_decode_sample(wl, row_frac, threads, inputs, Wq_rows):
    """One oracle pass: quantize every activation, then the sampled rows of
    every matrix.  Returns the algorithmic bytes it covered."""
    import oracle
    kinds = activation_kinds(wl)
    xq = {}
    nbytes = 0
    for tag, K in wl.activations.items():
        gam = inputs["gamma"].get(tag) if kinds[tag] == "norm" else None
        xq[tag] = oracle.quantize_q8_0(inputs["x"][tag], gam, wl.eps)
        nbytes += 4 * K + (4 * K if gam is not None else 0) + workloads.q8_0_bytes(1, K)
    for m in wl.matrices:
        tag = m.source.split(":", 1)[1]
        Wq = Wq_rows[m.name]
        oracle.matvec(Wq, xq[tag], m.cols, threads=threads)
        nbytes += Wq.nbytes + workloads.q8_0_bytes(1, m.cols) + 4 * Wq.shape[0]
    return nbytes


def oracle_setup(wl, row_frac):
    """Sampled rows of every matrix (every 1/row_frac-th row), quantized by the oracle."""
    import oracle
    Wq_rows = {}
    for m in wl.matrices:
        step = max(1, int(round(1.0 / row_frac)))
        rows = np.arange(0, m.rows, step)
        Wq_rows[m.name] = oracle.quantize_q4_0(synth.weight_rows(wl.seed, m.name, m.rows, m.cols, rows))
    kinds = activation_kinds(wl)
    inputs = {"x": {}, "gamma": {}}
    for tag, K in wl.activations.items():
        inputs["x"][tag] = synth.activations(wl.seed, f"x:{tag}:0", 1, K, outlier_frac=wl.outlier_frac)
        if kinds[tag] == "norm":
            inputs["gamma"][tag] = synth.gamma(wl.seed, tag, K)
    return Wq_rows, inputs


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(wl, budget_s, row_frac, steps=None, warmup=1, threads=None):
    cores = threads or cpu_cores()
    Wq_rows, inputs = oracle_setup(wl, row_frac)
    for _ in range(max(1, warmup)):
        oracle_decode_sample(wl, row_frac, cores, inputs, Wq_rows)  # untimed
    t0 = time.perf_counter()
    done = 0
    nbytes = 0
    while True:
        nbytes += oracle_decode_sample(wl, row_frac, cores, inputs, Wq_rows)
        done += 1
        el = time.perf_counter() - t0
        if steps is not None and done >= steps:
            break
        if steps is None and el >= budget_s:
            break
    el = time.perf_counter() - t0
    return nbytes / el / 1e9, cores, done, el, nbytes


def oracle_leg(wl, seconds, threads=None):
    """The oracle timed by the reference arm's own code in a fresh process,
    so that the benchmark process (its CUDA context, pinned buffers and
    threads) does not weigh on it and both legs measure the same thing.
    Returns the reference arm's JSON line."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", wl.name,
           "--steps", "1", "--warmup", "3", "--oracle-seconds", str(seconds)]
    if threads:
        cmd += ["--oracle-threads", str(threads)]
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"oracle leg failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------- GPU leg
class DecodeStep:
    def __init__(self, wl, device, layout="seg", copies=1):
        import torch
        from quantized_decode_gemv_rms_gb300 import qdg
        self.qdg = qdg
        self.torch = torch
        self.wl = wl
        self.kinds = activation_kinds(wl)
        self.W = {}
        for m in wl.matrices:
            Wq = torch.empty(qdg.q4_0_nbytes(m.rows, m.cols), dtype=torch.uint8, device=device)
            chunk = 16384
            for r in range(0, m.rows, chunk):
                r1 = min(m.rows, r + chunk)
                w = torch.from_numpy(synth.weights(wl.seed, m.name, m.rows, m.cols, row_begin=r, row_end=r1))
                wd = w.to(device)
                qdg.quantize_q4_0(wd, Wq[r * (m.cols // 32) * 18:r1 * (m.cols // 32) * 18], O=r1 - r, K=m.cols)
                del wd
            self.W[m.name] = Wq
        # the segment layout of every matrix (repacked once, at load); the split
        # route's GEMV reads it when layout == "seg", the per-launch timings always
        self.layout = layout
        self.Wr = {}
        for m in wl.matrices:
            Wr = torch.empty(qdg.q4_0_seg_nbytes(m.rows, m.cols), dtype=torch.uint8, device=device)
            qdg.q4_0_repack_seg(self.W[m.name], Wr, m.rows, m.cols)
            self.Wr[m.name] = Wr
        # weight copies the step rotates through (copy c of every matrix, in
        # the layout given here): a workload whose weights fit in L2 needs
        # several, so that every step reads its weights from HBM
        self.copies = copies
        self.copies_layout = layout
        src = self.Wr if layout == "seg" else self.W
        self.Wcopies = [src] + [{n: t.clone() for n, t in src.items()} for _ in range(copies - 1)]
        torch.cuda.synchronize()
        self.gamma = {tag: torch.from_numpy(synth.gamma(wl.seed, tag, K)).to(device)
                      for tag, K in wl.activations.items() if self.kinds[tag] == "norm"}
        # input sets: host (pinned) and device copies
        # input sets: one pinned host buffer and one device buffer per set, holding every
        # activation vector back to back (one copy moves a step's inputs); outputs likewise
        xoff, off = {}, 0
        for tag, K in wl.activations.items():
            xoff[tag] = (off, K)
            off += K
        self.x_host_flat, self.x_dev_flat, self.x_host, self.x_dev = [], [], [], []
        for p in range(N_INPUT_SETS):
            hf = torch.empty(off, dtype=torch.float32).pin_memory()
            for tag, (o, K) in xoff.items():
                hf[o:o + K] = torch.from_numpy(synth.activations(wl.seed, f"x:{tag}:{p}", 1, K,
                                                                 outlier_frac=wl.outlier_frac)[0])
            df = hf.to(device)
            self.x_host_flat.append(hf)
            self.x_dev_flat.append(df)
            self.x_host.append({tag: hf[o:o + K] for tag, (o, K) in xoff.items()})
            self.x_dev.append({tag: df[o:o + K] for tag, (o, K) in xoff.items()})
        self.xq = {tag: torch.empty(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device=device)
                   for tag, K in wl.activations.items()}
        ytotal = sum(m.rows for m in wl.matrices)
        self.y_flat = torch.empty(ytotal, dtype=torch.float32, device=device)
        self.y_host_flat = torch.empty(ytotal, dtype=torch.float32).pin_memory()
        self.y, self.y_host, off = {}, {}, 0
        for m in wl.matrices:
            self.y[m.name] = self.y_flat[off:off + m.rows]
            self.y_host[m.name] = self.y_host_flat[off:off + m.rows]
            off += m.rows
        # consecutive projections with the same input (and K) form one launch
        self.groups = []
        for m in wl.matrices:
            if (self.groups and self.groups[-1][0].source == m.source and self.groups[-1][0].cols == m.cols
                    and len(self.groups[-1]) < 4):
                self.groups[-1].append(m)
            else:
                self.groups.append([m])
        # the chain route's workspace (zeroed once; every chain launch leaves its counters zero)
        self.chain_ws = torch.zeros(qdg.q4_0s_gemv_chain_workspace_bytes(), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()      # release the fp32 staging of the weights

    def fusable(self, grp, layout=None, route=True):
        """Whether the fused kernel can serve this group (segment layout: it
        stages the input whole, K <= FUSED_SEG_MAX_K); with route=True,
        whether the fused route uses it (K <= FUSED_ROUTE_MAX_K)."""
        limit = FUSED_ROUTE_MAX_K if route else FUSED_SEG_MAX_K
        return (layout or self.layout) == "plain" or grp[0].cols <= limit

    def launches_per_step(self, route="split"):
        if route == "chain":
            return 1
        return sum(1 if route == "fused" and self.fusable(g) else 2 for g in self.groups)

    def run_group(self, grp, xs, Ws=None, layout=None, out=None):
        """One fused launch for projections that read the same activation."""
        layout = layout or self.layout
        tag = grp[0].source.split(":", 1)[1]
        g = self.gamma.get(tag) if self.kinds[tag] == "norm" else None
        out = out if out is not None else self.y
        ys, Os = [out[m.name] for m in grp], [m.rows for m in grp]
        if layout == "seg":
            Ws = Ws if Ws is not None else [self.Wr[m.name] for m in grp]
            self.qdg.q4_0s_gemv_rmsnorm_group(Ws, ys, Os, xs[tag], g, self.wl.eps, grp[0].cols)
        else:
            Ws = Ws if Ws is not None else [self.W[m.name] for m in grp]
            self.qdg.q4_0_gemv_rmsnorm_group(Ws, ys, Os, xs[tag], g, self.wl.eps, grp[0].cols)

    def copy_weights(self, grp, copy):
        """The matrices of a group in weight copy `copy` (None = the layout's own)."""
        if copy == 0:
            return None
        assert self.layout == self.copies_layout, "weight copies exist for one layout only"
        return [self.Wcopies[copy][m.name] for m in grp]

    def chain_stages(self, xs, copy=0, out=None):
        """The step as chain stages: one per group, in dependency order."""
        out = out if out is not None else self.y
        stages = []
        for grp in self.groups:
            tag = grp[0].source.split(":", 1)[1]
            Ws = self.copy_weights(grp, copy) or [self.Wr[m.name] for m in grp]
            stages.append({"x": xs[tag], "gamma": self.gamma.get(tag) if self.kinds[tag] == "norm" else None,
                           "K": grp[0].cols, "Ws": Ws, "ys": [out[m.name] for m in grp],
                           "Os": [m.rows for m in grp], "xq_out": self.xq[tag]})
        return stages

    def run(self, xs, events=None, fused=True, copy=0, route=None, out=None):
        """One decode step in dependency order.  route "chain": one launch
        runs every group (norm/quantize, then the grouped GEMV), each group
        after the previous one's outputs; for each group of projections
        sharing an input -- "fused": one launch (RMSNorm*gamma -> Q8_0 ->
        GEMV); "split": the quantize kernel, then one grouped GEMV launch.
        Without a route, `fused` picks between the last two.  `copy` picks the
        weight copy the step reads; `out` maps projections to their output
        buffers (default: the device outputs)."""
        qdg = self.qdg
        route = route or ("fused" if fused else "split")
        if route == "chain":
            assert self.layout == "seg", "the chain reads the segment layout"
            qdg.q4_0s_gemv_chain(self.chain_stages(xs, copy, out), self.wl.eps, self.chain_ws)
            return
        fused = route == "fused"
        for grp in self.groups:
            Ws = self.copy_weights(grp, copy)
            if fused and self.fusable(grp):
                self.run_group(grp, xs, Ws=Ws, out=out)
                continue
            tag = grp[0].source.split(":", 1)[1]
            K = grp[0].cols
            g = self.gamma.get(tag) if self.kinds[tag] == "norm" else None
            qdg.qnorm_quantize_q8_0(xs[tag], g, self.wl.eps, self.xq[tag], K=K, N=1)
            self.gemv_group(grp, self.xq[tag], Ws=Ws, out=out)

    def gemv_group(self, grp, xq, Ws=None, layout=None, out=None):
        """The grouped GEMV of one group on its prepared Q8_0 vector."""
        layout = layout or self.layout
        K = grp[0].cols
        out = out if out is not None else self.y
        ys, Os = [out[m.name] for m in grp], [m.rows for m in grp]
        if layout == "seg":
            Ws = Ws if Ws is not None else [self.Wr[m.name] for m in grp]
            self.qdg.q4_0s_q8_0_gemv_group(Ws, ys, Os, xq, K)
        else:
            Ws = Ws if Ws is not None else [self.W[m.name] for m in grp]
            self.qdg.q4_0_q8_0_gemv_group(Ws, ys, Os, xq, K)

def capture(fn, side, count=1):
    """CUDA graph of `count` calls of fn (on the side stream)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(count):
            fn()
    return g


def bench_ours(args, wl, world, rank, local):
    import torch
    from quantized_decode_gemv_rms_gb300 import qdg
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    qdg.lib()
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 1 if args.pdl else 0)
    # A step whose weights fit three times in L2 rotates through weight
    # copies (a multiple of the input sets), so every step streams from HBM.
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    wbytes = sum(workloads.q4_0_bytes(m.rows, m.cols) for m in wl.matrices)
    need = -(-3 * l2 // wbytes)                      # ceil(3 L2 / weight bytes)
    wcopies = 1 if wbytes > 3 * l2 else N_INPUT_SETS * -(-need // N_INPUT_SETS)
    spg = max(N_INPUT_SETS, wcopies)                 # steps per graph: every input set and copy once
    step = DecodeStep(wl, device, layout=args.layout, copies=wcopies)
    stream = torch.cuda.current_stream()
    nbytes = step_bytes(wl)
    route = args.route
    routes = [route] + [r for r in ("chain", "split", "fused") if r != route and (r != "chain" or args.layout == "seg")]
    L = step.launches_per_step(route)

    # eager warm-up of every route (also sets kernel attributes before capture)
    for r in routes:
        for i in range(3):
            step.run(step.x_dev[i % N_INPUT_SETS], route=r)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK

    # graphs: one per input set and route; the launch counters, read around the
    # capture of the timed route, tell which kernels the step consists of
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graphs = {}
    counts = {}
    # One graph holds spg consecutive steps (input set k % N_INPUT_SETS,
    # weight copy k % wcopies), as a multi-layer forward pass would:
    # programmatic dependent launch chains the kernels inside a graph, while
    # consecutive graph launches serialise.
    NC = 12                                         # launch counters of the library
    with torch.cuda.stream(side):
        for r in routes:
            before = [qdg.qdg_launch_count(i) for i in range(NC)]

            def steps(r=r):
                for k in range(spg):
                    step.run(step.x_dev[k % N_INPUT_SETS], route=r, copy=k % wcopies)
            graphs[r] = capture(steps, side)
            after = [qdg.qdg_launch_count(i) for i in range(NC)]
            counts[r] = [(after[i] - before[i]) // spg for i in range(NC)]
    stream.wait_stream(side)
    torch.cuda.synchronize()
    ng = len(step.groups)
    gk = 6 if args.layout == "seg" else 1          # launch counter of the split route's GEMV
    fk = 9 if args.layout == "seg" else 5          # and of the fused kernel
    nf = sum(1 for g in step.groups if step.fusable(g))
    if "fused" in counts:
        c = counts["fused"]
        assert c[fk] == nf and c[0] == ng - nf and c[gk] == ng - nf and c[11] == 0, counts
    if "split" in counts:
        c = counts["split"]
        assert c[0] == ng and c[gk] == ng and c[fk] == 0 and c[11] == 0, counts
    if "chain" in counts:
        c = counts["chain"]
        assert c[11] == 1 and sum(c) == 1, counts
    for c in counts.values():
        assert c[7 - gk] == 0 and c[14 - fk] == 0, counts
    sfx = "_seg" if args.layout == "seg" else ""
    fusion = {"route": route,
              "per_step_launches": {"chain": counts[route][11], "fused_norm_gemv" + sfx: counts[route][fk],
                                    "quantize": counts[route][0], "gemv" + sfx: counts[route][gk]}}

    def run_steps(n, r=route):
        """n decode steps: whole graphs of spg steps, the remainder eagerly."""
        if not args.graph:
            for k in range(n):
                step.run(step.x_dev[k % N_INPUT_SETS], route=r, copy=k % wcopies)
            return
        for _ in range(n // spg):
            graphs[r].replay()
        for k in range(n % spg):
            step.run(step.x_dev[k % N_INPUT_SETS], route=r, copy=k % wcopies)

    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        smi_id = str(local)
    sampler = ClockSampler(smi_id)
    sampler.start()
    t_end = time.time() + 0.6                       # pre-roll: clocks under this load
    while time.time() < t_end:
        run_steps(200)
        torch.cuda.synchronize()
    run_steps(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    e0.record(stream)
    run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    status = qdg.qdg_device_status()
    if status != qdg.QDG_OK:
        raise RuntimeError(f"device status after timed region: {qdg.status_string(status)}")
    t_end = time.time() + 0.3                       # post-roll
    while time.time() < t_end:
        run_steps(200)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()

    # ---- spread of the step time: events around each of R graph replays
    # (spg steps each), outside the timed region above
    dist = None
    if args.graph:
        reps = max(20, min(200, args.steps // spg))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        evs[0].record(stream)
        for i in range(reps):
            graphs[route].replay()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per = sorted(evs[i].elapsed_time(evs[i + 1]) * 1e3 / spg for i in range(reps))
        pick = lambda q: per[min(reps - 1, int(round(q * (reps - 1))))]
        dist = {"p10": round(pick(0.1), 2), "p50": round(pick(0.5), 2), "p90": round(pick(0.9), 2),
                "samples": reps, "unit": "us per step",
                "how": f"CUDA events around each replay of the {spg}-step graph"}

    # ---- the other routes, same number of steps, for comparison
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    ms_other = {}
    for r in routes[1:]:
        run_steps(args.warmup, r)
        torch.cuda.synchronize()
        f0.record(stream)
        run_steps(args.steps, r)
        f1.record(stream)
        torch.cuda.synchronize()
        ms_other[r] = f0.elapsed_time(f1) / args.steps

    # ---- per-launch cost of each group's launch (GEMV alone on a prepared Q8_0
    # vector, and the fused launch): a graph of C back-to-back launches, each on
    # its own copy of the weights (C copies exceed three L2 sizes, so every
    # launch streams its weights from HBM)
    kinds = ["gemv", "gemv_seg", "fused", "fused_seg"]
    per_call = {k: {} for k in kinds}
    spread_kind = "gemv_seg" if args.layout == "seg" else "gemv"
    per_call_spread = {}
    launch_bytes = {k: {} for k in kinds}
    for p_ in range(1):
        step.run(step.x_dev[0], fused=False)          # the Q8_0 vectors of input set 0
    torch.cuda.synchronize()
    for grp in step.groups:
        name = "+".join(m.name for m in grp)
        tag = grp[0].source.split(":", 1)[1]
        K = grp[0].cols
        gbytes = sum(workloads.q4_0_bytes(m.rows, m.cols) for m in grp)
        copies = int(min(160, max(2, -(-3 * l2 // gbytes))))
        for kind in kinds:
            if kind == "fused_seg" and not step.fusable(grp, "seg", route=False):
                continue
            src = step.Wr if kind.endswith("_seg") else step.W
            Wc = [[src[m.name] for m in grp]] + [[src[m.name].clone() for m in grp] for _ in range(copies - 1)]

            def one(c, kind=kind, Wc=Wc):
                if kind.startswith("fused"):
                    step.run_group(grp, step.x_dev[0], Ws=Wc[c], layout="seg" if kind == "fused_seg" else "plain")
                else:
                    step.gemv_group(grp, step.xq[tag], Ws=Wc[c], layout="seg" if kind == "gemv_seg" else "plain")
            with torch.cuda.stream(side):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=side):
                    for c in range(copies):
                        one(c)
                gr.replay()
                side.synchronize()
                # events around every replay: the mean per launch, and for the
                # timed kernel kind also the spread over the replays
                reps = 21 if kind == spread_kind else 3
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
                evs[0].record(side)
                for r in range(reps):
                    gr.replay()
                    evs[r + 1].record(side)
                side.synchronize()
            per_call[kind][name] = evs[0].elapsed_time(evs[reps]) * 1e3 / (reps * copies)
            if kind == spread_kind:
                per = sorted(evs[r].elapsed_time(evs[r + 1]) * 1e3 / copies for r in range(reps))
                per_call_spread[name] = {"p10": round(per[2], 2), "p50": round(per[10], 2), "p90": round(per[18], 2),
                                         "replays": reps, "launches_per_replay": copies}
            del gr, Wc
            torch.cuda.empty_cache()
        xbytes = 4 * K * (2 if grp[0].source.startswith("norm:") else 1)
        launch_bytes["fused"][name] = gbytes + xbytes + sum(4 * m.rows for m in grp)
        launch_bytes["gemv"][name] = gbytes + workloads.q8_0_bytes(1, K) + sum(4 * m.rows for m in grp)
        launch_bytes["gemv_seg"][name] = launch_bytes["gemv"][name]
        launch_bytes["fused_seg"][name] = launch_bytes["fused"][name]
    torch.cuda.synchronize()
    gbs_per_call = {kind: {n: launch_bytes[kind][n] / (per_call[kind][n] * 1e-6) / 1e9 for n in per_call[kind]}
                    for kind in per_call}

    # ---- end to end through the same calls, inputs from pinned host memory:
    # every step moves its input vectors host -> device (one copy), runs, and
    # moves every output device -> host.  The headline copies the inputs with
    # the library's copy kernel (qdg_stage_copy) and lets the GEMVs store the
    # outputs straight into the mapped pinned buffer; a second staging copy
    # for the outputs, and copy-engine copies, are measured beside it.  With graphs, the copies are nodes of the same graph
    # as the kernels (spg steps per graph).
    n_e2e = spg * max(3, min(args.steps, 500) // spg)
    h2d = sum(t.numel() * 4 for t in step.x_host[0].values())
    d2h = sum(t.numel() * 4 for t in step.y_host.values())

    def measure_e2e(staging):
        e2e_graph = None
        if args.graph:
            def e2e_steps():
                for k in range(spg):
                    _e2e_step(step, None, k, route=route, staging=staging, copy=k % wcopies)
            with torch.cuda.stream(side):
                e2e_graph = capture(e2e_steps, side)
            stream.wait_stream(side)
            torch.cuda.synchronize()

        def run_e2e(n):
            if e2e_graph is not None:
                for _ in range(n // spg):
                    e2e_graph.replay()
            else:
                for k in range(n):
                    _e2e_step(step, None, k, route=route, staging=staging, copy=k % wcopies)
        run_e2e(spg)
        torch.cuda.synchronize()
        barrier(world)
        f0.record(stream)
        run_e2e(n_e2e)
        f1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(f0.elapsed_time(f1) / n_e2e, world, device)
    ms_e2e = measure_e2e("direct")
    ms_e2e_kernel = measure_e2e("kernel")
    ms_e2e_engine = measure_e2e("engine")

    peaks, peak_src = measured_peaks()
    if route == "chain":
        # one launch is the whole step: its algorithmic bytes over the average
        # launch time of the timed region (events on the launching stream)
        kernel = "gemv_chain_kernel (q4_0s_gemv_chain)"
        kern_bytes, launches = nbytes, 1
        achieved = nbytes / (ms * 1e-3) / 1e9
        traffic = ncu_traffic("gemv_chain.cu", wl.name)
    else:
        def main_kind(grp):
            if args.layout == "seg":
                return "fused_seg" if route == "fused" and step.fusable(grp) else "gemv_seg"
            return "fused" if route == "fused" else "gemv"
        mk = {"+".join(m.name for m in g): main_kind(g) for g in step.groups}
        kern_bytes, launches = sum(launch_bytes[k][n] for n, k in mk.items()), len(step.groups)
        # the dominant kernel's average launch from the per-launch graphs above
        achieved = kern_bytes / (sum(per_call[k][n] for n, k in mk.items()) * 1e-6) / 1e9
        names = {"fused": "gemv_kernel<fused> (q4_0_gemv_rmsnorm_group)",
                 "gemv": "gemv_kernel (q4_0_q8_0_gemv_group)",
                 "gemv_seg": "gemv_seg_kernel (q4_0s_q8_0_gemv_group)",
                 "fused_seg": "gemv_seg_kernel<fused> (q4_0s_gemv_rmsnorm_group)"}
        kernel = " + ".join(sorted({names[k] for k in mk.values()}))
        used = set(mk.values())
        traffic = (ncu_traffic("gemv_seg.cu", wl.name) if used == {"gemv_seg"} else
                   ncu_traffic("gemv.cu", wl.name) if used == {"gemv"} else None)
    roof = {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_source": ("measured: MEASURED_PEAKS.json hbm_gbs (copy bandwidth)" if peak_src == "measured"
                            else "fallback 6.8 TB/s"),
            "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
            "traffic_source": (traffic.get("what") if traffic else
                               "no ncu capture of this source on this workload"),
            "algorithmic_bytes_per_launch": round(kern_bytes / launches),
            "launches_of_this_kernel_per_step": launches,
            "achieved_over_whole_step": round(kern_bytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_nominal_8TB": round(achieved / 8000.0, 4)}
    result = {
        "metric": METRIC, "value": round(nbytes * world / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i32 (int4 x int8 block sums) + f32 scaling",
        "data": ("synthetic (seeded N(0,0.02) weights, N(0,1) activations" +
                 (f" with {wl.outlier_frac:.0%} x{wl.outlier_mult:g} outliers)" if wl.outlier_frac else ")")),
        "config": {"workload": wl.name, "batch": 1, "matrices": {m.name: [m.rows, m.cols] for m in wl.matrices},
                   "bytes_per_step": nbytes,
                   "l2": (f"inputs larger than L2 ({wbytes / 1e6:.0f} MB of weights per step vs "
                          f"{l2 / 1e6:.0f} MB L2)" if wcopies == 1 else
                          f"weights rotate through {wcopies} copies ({wcopies * wbytes / 1e6:.0f} MB, more than "
                          f"three times the {l2 / 1e6:.0f} MB L2), so every step reads its weights from HBM"),
                   "route": ({"chain": "chain: one launch per step (every group's RMSNorm->Q8_0 and grouped GEMV, "
                                       "each group after the previous group's outputs)",
                              "fused": "fused: one RMSNorm->Q8_0->GEMV launch per group" +
                                       (f" (K <= {FUSED_ROUTE_MAX_K}; split for larger K)" if args.layout == "seg"
                                        else ""),
                              "split": "split: quantize kernel + grouped GEMV launch per group"}[route]) +
                            ("; weights in the segment layout (repacked at load)" if args.layout == "seg"
                             else "; weights in plain Q4_0 blocks") +
                            "; groups " + ", ".join("+".join(m.name for m in g) for g in step.groups) +
                            " in dependency order",
                   "launch": ((f"cuda graph of {spg} steps" if args.graph else "eager") +
                              (" + PDL" if args.pdl else "")),
                   "parallelism": f"replicas x{world}"},
        "us_per_step": round(ms * 1e3, 2),
        "us_per_step_spread": dist,
        "us_per_call": {k: {n: round(v, 2) for n, v in d.items()} for k, d in per_call.items()},
        "us_per_call_spread": {"kind": spread_kind, "groups": per_call_spread,
                               "how": "mean launch time within each of 21 graph replays; p10/p50/p90 over replays"},
        "gbs_per_call": {k: {n: round(v, 1) for n, v in d.items()} for k, d in gbs_per_call.items()},
        "per_call_note": ("one launch per group of projections sharing an input (gemv: on a prepared Q8_0 vector; "
                          "gemv_seg: the same on weights in the segment layout; "
                          "fused: norm+quantize+GEMV; fused_seg: the same on the segment layout, K <= 16384); "
                          "graph of back-to-back launches on distinct weight copies "
                          "(> 3 x L2), PDL as configured"),
        "other_routes": {r: {"us_per_step": round(v * 1e3, 2), "value": round(nbytes / (v * 1e-3) / 1e9, 1)}
                         for r, v in ms_other.items()},
        "fusion_check": fusion,
        "roofline": roof,
        "e2e": {"value": round(nbytes * world / (ms_e2e * 1e-3) / 1e9, 1), "unit": UNIT,
                "ms_per_step": round(ms_e2e, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": ("every step: one host-to-device copy of its input vectors from pinned memory by the "
                        "library's staging kernel (qdg_stage_copy), the step through the C ABI, and every output "
                        "stored by the GEMVs straight into the mapped pinned host buffer (the device-to-host move "
                        "of the step's result is those stores)" +
                        (f"; copies and kernels in one CUDA graph of {spg} steps" if args.graph else "")),
                "staging_kernel": {"value": round(nbytes * world / (ms_e2e_kernel * 1e-3) / 1e9, 1),
                                   "ms_per_step": round(ms_e2e_kernel, 5),
                                   "how": "the same with the outputs written to device memory and moved to the "
                                          "pinned buffer by a second staging-kernel copy"},
                "copy_engine": {"value": round(nbytes * world / (ms_e2e_engine * 1e-3) / 1e9, 1),
                                "ms_per_step": round(ms_e2e_engine, 5),
                                "how": "the same with stream-ordered copy-engine copies in both directions"}},
        "gpu_launches": int(L * args.steps),
        "clocks": clocks,
    }
    return result, step


def bench_extras(args, device):
    """Small-N (N = 2, 4, 8) and prefill GEMM timings: CUDA events around each
    call, after warm-up.  The small-N weights rotate through enough copies to
    exceed three L2 sizes, so every call reads HBM."""
    import torch
    from quantized_decode_gemv_rms_gb300 import qdg
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    peaks, _ = measured_peaks()
    out = {"small_n": {}, "prefill": {}}

    def timed(fn, reps, warm=5):
        for i in range(warm):
            fn(i)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i, (a, b) in enumerate(evs):
            a.record()
            fn(i)
            b.record()
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in evs])) * 1e3

    side = torch.cuda.Stream(device)

    def timed_graph(fn, count, replays=3):
        """Per-call time from a CUDA graph of `count` back-to-back calls
        fn(0..count-1) (PDL as configured), replayed `replays` times."""
        for i in range(count):
            fn(i)
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=side):
                for i in range(count):
                    fn(i)
            gr.replay()
            side.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(side)
            for _ in range(replays):
                gr.replay()
            a1.record(side)
            side.synchronize()
        return a0.elapsed_time(a1) * 1e3 / (replays * count)

    def make_w(seed, name, O, K):
        Wq = torch.empty(qdg.q4_0_nbytes(O, K), dtype=torch.uint8, device=device)
        for r in range(0, O, 8192):
            r1 = min(O, r + 8192)
            w = torch.from_numpy(synth.weights(seed, name, O, K, row_begin=r, row_end=r1)).to(device)
            qdg.quantize_q4_0(w, Wq[r * (K // 32) * 18:r1 * (K // 32) * 18], O=r1 - r, K=K)
        return Wq

    for (O, K) in (workloads.SMALL_N_SHAPES if args.only in (None, "small_n") else ()):
        Wq = make_w(workloads.SMALL_N_SEED, f"smalln-{O}x{K}", O, K)
        copies = max(2, -(-3 * l2 // Wq.numel()))
        Ws = [Wq] + [Wq.clone() for _ in range(copies - 1)]
        res = {}
        for N in workloads.SMALL_N_COLS:
            x = torch.from_numpy(synth.activations(workloads.SMALL_N_SEED, f"smalln-x-{K}", N, K)).to(device)
            g = torch.from_numpy(synth.gamma(workloads.SMALL_N_SEED, f"smalln-g-{K}", K)).to(device)
            xq = torch.empty(qdg.q8_0_nbytes(N, K), dtype=torch.uint8, device=device)
            qdg.qnorm_quantize_q8_0(x, g, 1e-6, xq)
            y = torch.empty((N, O), dtype=torch.float32, device=device)
            us = timed_graph(lambda i: qdg.q4_0_q8_0_gemm_small_n(Ws[i % copies], xq, y, O, O, K, N), copies)
            nbytes = workloads.gemv_algorithmic_bytes(O, K, N)
            res[f"N{N}"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                            "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
        # every N on the segment layout (N = 2: dp4a with one unpack for both
        # vectors; N >= 3: the MMA kernel with lanes loading straight into registers)
        Wr = torch.empty(qdg.q4_0_seg_nbytes(O, K), dtype=torch.uint8, device=device)
        qdg.q4_0_repack_seg(Wq, Wr, O, K)
        Wrs = [Wr] + [Wr.clone() for _ in range(copies - 1)]
        for N in workloads.SMALL_N_COLS:
            x = torch.from_numpy(synth.activations(workloads.SMALL_N_SEED, f"smalln-x-{K}", N, K)).to(device)
            xq = torch.empty(qdg.q8_0_nbytes(N, K), dtype=torch.uint8, device=device)
            qdg.qnorm_quantize_q8_0(x, g, 1e-6, xq)
            y = torch.empty((N, O), dtype=torch.float32, device=device)
            us = timed_graph(lambda i: qdg.q4_0s_q8_0_gemm_small_n(Wrs[i % copies], xq, y, O, O, K, N), copies)
            nbytes = workloads.gemv_algorithmic_bytes(O, K, N)
            res[f"N{N}_seg"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                                "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4)}
        del Wrs, Wr
        out["small_n"][f"{O}x{K}"] = dict(res, weight_copies=copies,
                                          timing="graph of back-to-back launches over the weight copies; "
                                                 "N<n> = plain Q4_0 layout, N<n>_seg = the same on the segment layout")
        del Ws, Wq
        torch.cuda.empty_cache()
    for (O, K, T) in (workloads.PREFILL_SHAPES if args.only in (None, "prefill") else ()):
        Wq = make_w(workloads.PREFILL_SEED, f"prefill-{O}x{K}", O, K)
        x = torch.from_numpy(synth.activations(workloads.PREFILL_SEED, f"prefill-{O}x{K}-x", T, K)).to(device)
        xq = torch.empty(qdg.q8_0_nbytes(T, K), dtype=torch.uint8, device=device)
        qdg.qnorm_quantize_q8_0(x, None, 0.0, xq)
        y = torch.empty((T, O), dtype=torch.float32, device=device)
        ws = torch.empty(qdg.q4_0_q8_0_gemm_workspace_bytes(K, T), dtype=torch.uint8, device=device)
        us = timed(lambda i: qdg.q4_0_q8_0_gemm(Wq, xq, y, O, O, K, T, ws), 30)
        tflops = 2.0 * O * K * T / (us * 1e-6) / 1e12
        out["prefill"][f"{O}x{K}x{T}"] = {"us": round(us, 2), "tflops": round(tflops, 1),
                                          "frac_fp16_peak": round(tflops / peaks["bf16_tflops"], 4)}
        del Wq, x, xq, y, ws
        torch.cuda.empty_cache()
    # Q8_0 weights (batch-1 GEMV): gate-shaped and down-shaped matrices, rotating weight copies
    out["q8_0_weights"] = {}
    for (O, K) in (workloads.SMALL_N_SHAPES if args.only in (None, "q8w") else ()):
        W8 = torch.empty(O * (K // 32) * 34, dtype=torch.uint8, device=device)
        for r in range(0, O, 8192):
            r1 = min(O, r + 8192)
            w = torch.from_numpy(synth.weights(workloads.SMALL_N_SEED, f"q8w-{O}x{K}", O, K, row_begin=r,
                                               row_end=r1)).to(device)
            qdg.qnorm_quantize_q8_0(w, None, 0.0, W8[r * (K // 32) * 34:r1 * (K // 32) * 34], K=K, N=r1 - r)
        copies = max(2, -(-3 * l2 // W8.numel()))
        Ws = [W8] + [W8.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(synth.activations(workloads.SMALL_N_SEED, f"q8w-x-{K}", 1, K)).to(device)
        xq = torch.empty(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device=device)
        qdg.qnorm_quantize_q8_0(x, None, 0.0, xq)
        y = torch.empty(O, dtype=torch.float32, device=device)
        us = timed_graph(lambda i: qdg.q8_0_q8_0_gemv(Ws[i % copies], xq, y, O, K), copies)
        nbytes = O * (K // 32) * 34 + (K // 32) * 34 + 4 * O
        out["q8_0_weights"][f"{O}x{K}"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                                           "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                                           "weight_copies": copies}
        del Ws, W8
        torch.cuda.empty_cache()
    # the quantize kernel alone on the decode step's activation shapes (one
    # vector, with and without the norm): a graph of back-to-back launches
    out["qnorm"] = {}
    for (K, norm) in (((4096, True), (14336, False)) if args.only in (None, "qnorm") else ()):
        x = torch.from_numpy(synth.activations(workloads.SMALL_N_SEED, f"qn-x-{K}", 1, K)).to(device)
        g = torch.from_numpy(synth.gamma(workloads.SMALL_N_SEED, f"qn-g-{K}", K)).to(device) if norm else None
        xq = torch.empty(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device=device)
        us = timed_graph(lambda i: qdg.qnorm_quantize_q8_0(x, g, 1e-6, xq), 20)
        out["qnorm"][f"K{K}{'_norm' if norm else '_plain'}"] = {"us": round(us, 2)}
    # k-quant weights (batch-1 GEMV): Q4_K (144-byte super-blocks) and Q5_K
    # (176-byte), the same shapes, quantized on the GPU at load time,
    # rotating weight copies
    kquants = (("q4k", "q4_k_weights", 144, qdg.quantize_q4_k, qdg.q4_k_q8_0_gemv),
               ("q5k", "q5_k_weights", 176, qdg.quantize_q5_k, qdg.q5_k_q8_0_gemv))
    for tag, key, sb, quantize, gemv in kquants:
        out[key] = {}
        for (O, K) in (workloads.SMALL_N_SHAPES if args.only in (None, tag) else ()):
            Wk = torch.empty(O * (K // 256) * sb, dtype=torch.uint8, device=device)
            for r in range(0, O, 8192):
                r1 = min(O, r + 8192)
                w = torch.from_numpy(synth.weights(workloads.SMALL_N_SEED, f"{tag}-{O}x{K}", O, K, row_begin=r,
                                                   row_end=r1)).to(device)
                quantize(w, Wk[r * (K // 256) * sb:r1 * (K // 256) * sb], O=r1 - r, K=K)
                del w
            copies = max(2, -(-3 * l2 // Wk.numel()))
            Ws = [Wk] + [Wk.clone() for _ in range(copies - 1)]
            x = torch.from_numpy(synth.activations(workloads.SMALL_N_SEED, f"{tag}-x-{K}", 1, K)).to(device)
            xq = torch.empty(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device=device)
            qdg.qnorm_quantize_q8_0(x, None, 0.0, xq)
            y = torch.empty(O, dtype=torch.float32, device=device)
            us = timed_graph(lambda i: gemv(Ws[i % copies], xq, y, O, K), copies)
            nbytes = O * (K // 256) * sb + (K // 32) * 34 + 4 * O
            out[key][f"{O}x{K}"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                                    "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                                    "weight_copies": copies}
            del Ws, Wk
            torch.cuda.empty_cache()
    out["peak_note"] = ("small-N against the measured HBM copy bandwidth; prefill against the measured dense "
                        "bf16 burst peak (the fp16 tensor rate is the same nominal 2.25 PFLOP/s)")
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return out


def _e2e_step(step, graphs, k, fused=True, staging="direct", copy=0, route=None):
    """One step from host buffers: every input vector in (one copy), the step,
    every output out.  staging="direct": the library's staging kernel copies
    the inputs in from the mapped pinned buffer, and the GEMVs store their
    outputs straight into the mapped pinned output buffer (the device-to-host
    move is the kernels' own stores); "kernel": the staging kernel for both
    directions (the outputs land in device memory first); "engine":
    stream-ordered copy-engine copies for both."""
    p = k % N_INPUT_SETS
    if staging in ("kernel", "direct"):
        step.qdg.qdg_stage_copy(step.x_dev_flat[p], step.x_host_flat[p])
    else:
        step.x_dev_flat[p].copy_(step.x_host_flat[p], non_blocking=True)
    step.run(step.x_dev[p], fused=fused, copy=copy, route=route,
             out=step.y_host if staging == "direct" else None)
    if staging == "kernel":
        step.qdg.qdg_stage_copy(step.y_host_flat, step.y_flat)
    elif staging == "engine":
        step.y_host_flat.copy_(step.y_flat, non_blocking=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.LLAMA_8B.name, choices=sorted(workloads.ALL))
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--route", choices=["chain", "split", "fused"], default="split",
                    help="the timed main line: split = quantize kernel + grouped GEMV per group (default); "
                         "fused = one norm+quantize+GEMV launch per group; chain = one persistent launch per step")
    ap.add_argument("--layout", choices=["seg", "plain"], default="seg",
                    help="weight layout the split route's GEMV reads: seg = segment layout repacked at load "
                         "(default), plain = Q4_0 blocks as stored")
    ap.add_argument("--pdl", action="store_true", default=True)
    ap.add_argument("--no-pdl", dest="pdl", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--oracle-seconds", type=float, default=0.0,
                    help="reference arm: time the oracle for this many seconds instead of --steps passes")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="reference arm: host threads for the oracle (default: every core this process may use)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the small-N and prefill timings")
    ap.add_argument("--only", choices=["small_n", "prefill", "q8w", "q4k", "q5k", "qnorm"], default=None,
                    help="time only that product (one JSON object with its numbers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = workloads.ALL[args.workload]
    world, rank, local = dist_setup(args)

    if args.impl == "reference":
        if rank != 0:
            return
        row_frac = 1.0 / 16
        rate, cores, done, el, nb = time_oracle(wl, args.oracle_seconds, row_frac,
                                                steps=None if args.oracle_seconds > 0 else args.steps,
                                                warmup=args.warmup, threads=args.oracle_threads or None)
        line = {"impl": "reference", "metric": METRIC, "value": round(rate, 4), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / done * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64 (oracle: dequantize-then-dot)", "data": "synthetic",
                "config": {"workload": wl.name, "batch": 1},
                "cpu_baseline": {"value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": f"every 16th row of each matrix + all activations; {done} passes "
                                           f"in {el:.1f} s ({nb / 1e9:.2f} GB)"},
                "e2e": {"value": round(rate, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.only in ("small_n", "prefill", "q8w", "q4k", "q5k", "qnorm"):
        import torch
        torch.cuda.set_device(local)
        ex = bench_extras(args, torch.device("cuda", local))
        key = {"q8w": "q8_0_weights", "q4k": "q4_k_weights", "q5k": "q5_k_weights"}.get(args.only, args.only)
        if rank == 0:
            print(json.dumps({"only": args.only, key: ex[key]}))
        return
    result, step = bench_ours(args, wl, world, rank, local)
    if args.extras and rank == 0:
        import torch
        del step
        torch.cuda.empty_cache()
        result["extras"] = bench_extras(args, torch.device("cuda", local))
    if rank == 0 and world == 1 and args.cpu_baseline:
        # the reference arm's code in a fresh process, on every core, then on one
        # thread (its rows are independent, so both give the same bits)
        ref = oracle_leg(wl, args.cpu_budget)
        result["cpu_baseline"] = dict(ref["cpu_baseline"], how="bench.py --impl reference in a fresh process")
        ref1 = oracle_leg(wl, max(1.0, args.cpu_budget / 4), threads=1)
        result["cpu_baseline"]["single_thread"] = {k: ref1["cpu_baseline"][k] for k in ("value", "unit", "cores",
                                                                                        "sample")}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
