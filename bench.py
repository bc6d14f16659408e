"""Benchmark of the shared-base, per-request LoRA projection on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path (planner, shrink, fused base+expand) over one
batch of the workload: one lora_linear_forward call (for the 24-layer sweep, 96 calls: 4
projections x 24 layers). Inputs are seeded synthetic bf16 tensors already resident in
HBM; three copies of the weights rotate between steps so that W is not L2-resident, and
X alone is larger than the 129 MB L2 for the prefill workloads.

Prints one JSON line (rank 0). `value` is useful TFLOP/s of the whole job (all ranks);
`e2e` is the same metric through the host-buffer entry point (X copied in, Y copied
out every step); `roofline` is the projection kernel against the roof that binds it (CUDA
events around each launch, on the launch stream): useful TFLOP/s against the measured bf16
peak, or algorithmic GB/s against the measured copy bandwidth for batches that stream W
(`roofline_other` holds the other roof); `cpu_baseline` is the fp64 oracle timed on a
bounded sample on the host cores. The default run (the 16k prefill) also times the
decode-sized batch (48 chat rows, gate_up) in the same process, under `decode`.

Multi-GPU: launched under torchrun, every rank runs an independent replica (the
projection's rows need no exchange); the timed region is bracketed by barriers and the
slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-linear TFLOP/s & tokens/s at 1 GB300; % of bf16 tensor peak / HBM BW"
SWEEP = "sweep_24_layers"
SWEEP_MULTI = "sweep_24_layers_multi"   # the same stack with three adapters (ids 1, 2, 3)
DECODE_SWEEP = "decode_24_layers"        # one decode step of six chats (48 rows) through the same stack


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def _code_only(text: str) -> str:
    """Source text without its comments and blank lines: what the compiler reads (the device
    sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (line.split("//", 1)[0].rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line.strip())


def _kernel_hash(w4: bool = False):
    """Hash of the code the GPU runs for the measured kernel: the device part of its source file
    (up to the end of its device namespace; the host launch code after it does not count), the
    device helpers and the parameter headers it compiles from (lora_internal.h, and lora_w4.h
    for the 4-bit kernel), each without comments and blank lines, so that an edit of a comment
    does not retire a capture of the same code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixed_lora_projection_gb300", "csrc")
    with open(os.path.join(csrc, "kernels_w4.cu" if w4 else "kernels.cu")) as fh:
        text = fh.read()
    h.update(_code_only(text[:text.index("}  // namespace dev")]).encode())
    for f in ("dev_common.cuh", "lora_internal.h") + (("lora_w4.h",) if w4 else ()):
        with open(os.path.join(csrc, f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _profiled_traffic(workload: str):
    """dram bytes per fused launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    kh = _kernel_hash(workload.endswith("+w4"))
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[1] == kh:
                return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle samples in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        self.index = index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed"
        if not inside:
            inside, window = rows, "whole run"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# --------------------------------------------------------------------------- workloads

def _workloads(name):
    from mixed_lora_projection_gb300.synth import (SWEEP_LAYERS, SWEEP_PROJECTIONS, WORKLOADS, decode_workload,
                                                   sweep_workload)
    if name in (SWEEP, SWEEP_MULTI):
        return [(sweep_workload(p, name == SWEEP_MULTI), layer, i) for layer in range(SWEEP_LAYERS)
                for i, (p, _, _) in enumerate(SWEEP_PROJECTIONS)]
    if name == DECODE_SWEEP:
        return [(decode_workload(p), layer, i) for layer in range(SWEEP_LAYERS)
                for i, (p, _, _) in enumerate(SWEEP_PROJECTIONS)]
    return [(WORKLOADS[name], 0, 0)]


def _flops_of(items):
    return sum(w.useful_flops() for w, _, _ in items)


def _tokens_of(items):
    return items[0][0].T


def _fused_flops(w):
    """Algorithmic FLOPs of the fused base+expand kernel: 2 T d_in d_out + 2 T_a r d_out."""
    return 2.0 * w.T * w.d_in * w.d_out + 2.0 * w.adapter_rows * w.rank * w.d_out


L2_BYTES = 129e6   # GB300 L2


def _alg_bytes(w, w4=False):
    """Algorithmic bytes of one call: bf16 X, W, Y and the named adapters; with a 4-bit base, W
    counts as its packed nibbles (half a byte per weight) plus its bf16 group scales."""
    b = w.algorithmic_bytes()
    if w4:
        b += -2.0 * w.d_out * w.d_in + 0.5 * w.d_out * w.d_in + 2.0 * w.d_out * w.d_in / 128
    return b


def _l2_note(items, n_copies, w4=False):
    """What keeps the timed steps from running out of L2 (129 MB), for this workload."""
    if len(items) > 1:
        wb = sum(2.0 * w.d_in * w.d_out for w, _, _ in items)
        return f"{len(items)} distinct weight sets per step ({wb / 1e9:.1f} GB), each read once per step"
    w = items[0][0]
    xb = 2.0 * w.T * w.d_in
    wb = (0.5 + 2.0 / 128) * w.d_in * w.d_out if w4 else 2.0 * w.d_in * w.d_out
    wdesc = f"{n_copies} rotating weight copies of {wb / 1e6:.0f} MB ({n_copies * wb / 1e6:.0f} MB in all)"
    if xb > L2_BYTES:
        return f"X ({xb / 1e6:.0f} MB) larger than L2; {wdesc}"
    if wb > L2_BYTES:
        return f"X ({xb / 1e6:.1f} MB) fits in L2; each step reads a weight copy ({wb / 1e6:.0f} MB) larger than L2"
    return f"X ({xb / 1e6:.1f} MB) fits in L2; {wdesc}, larger than L2 together"


def _rooflines(items, w4, fused_flops, avg_fused_ms, traffic, peak_burst, hbm, src, shrink_n, peak_sust=None):
    """(binding roof, other roof) of the timed kernel: the tensor roof (algorithmic FLOPs against
    the measured bf16 burst) and the HBM roof (algorithmic bytes against the measured copy
    bandwidth); the one that takes longer at its peak binds. The tensor roof also gives the
    fraction of the measured sustained bf16 rate (cuBLAS back to back for seconds, at the power
    limit), the figure for lines whose timed region runs long enough to reach that limit."""
    alg = sum(_alg_bytes(w, w4) for w, _, _ in items)
    kernel = ("lora_w4_kernel (4-bit base + expand; shrink on lora_gemm_kernel before it)" if w4
              else "lora_gemm_kernel (shrink + base + expand, one launch per call)" if not shrink_n
              else "lora_gemm_kernel (fused base + expand launch)")
    achieved_tf = fused_flops / (avg_fused_ms * 1e-3) / 1e12 if avg_fused_ms else None
    achieved_gbs = alg / (avg_fused_ms * 1e-3) / 1e9 if avg_fused_ms else None
    tensor = {"bound": "tensor", "achieved": round(achieved_tf, 2) if achieved_tf else None, "peak": peak_burst,
              "unit": "TFLOP/s", "frac": round(achieved_tf / peak_burst, 4) if achieved_tf else None,
              "traffic": traffic, "peak_source": f"{src} bf16 burst", "kernel": kernel,
              "algorithmic_flops_per_step": fused_flops}
    if peak_sust:
        tensor["peak_sustained"] = peak_sust
        tensor["frac_of_sustained"] = round(achieved_tf / peak_sust, 4) if achieved_tf else None
    mem = {"bound": "hbm", "achieved": round(achieved_gbs, 1) if achieved_gbs else None, "peak": hbm,
           "unit": "GB/s", "frac": round(achieved_gbs / hbm, 4) if achieved_gbs else None, "traffic": traffic,
           "peak_source": f"{src} copy bandwidth", "kernel": kernel, "algorithmic_bytes_per_step": alg}
    if alg / (hbm * 1e9) > fused_flops / (peak_burst * 1e12):
        return mem, tensor
    return tensor, mem


def decode_line(dev, steps, warmup):
    """The decode-sized batch (the 48 chat rows of the mixed batch, gate_up 5120 -> 34816, no
    adapter rows) timed in the same process as the headline: its kernel streams W, so the HBM
    roof binds. Three weight copies of 356 MB rotate, so W never stays in L2."""
    import torch
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    from mixed_lora_projection_gb300.synth import WORKLOADS, make_inputs
    w = WORKLOADS["mixed_decode"]
    copies = [make_inputs(w, dev, proj_index=4 * c, with_x=(c == 0)) for c in range(3)]
    y = torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, len(w.seg_ids), dev) as ll:
        def f(i):
            c = copies[i % 3]
            ll.forward(copies[0].x, w.seg_offsets, w.seg_ids, c.w, c.a, c.b, c.scales, y=y, stream=stream)
        for i in range(warmup):
            f(i)
        torch.cuda.synchronize()
        assert ll.status() == 0
        ll.set_option(L.OPT_TIMING, 1)
        n0 = ll.timing(1)[2]
        sampler = ClockSampler(dev.index)
        sampler.start()
        time.sleep(0.2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.time()
        e0.record(stream)
        for i in range(steps):
            f(i)
        e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        time.sleep(0.1)
        sampler.stop()
        kernel_ms, n_timed, n_all = ll.timing(1)
        ll.set_option(L.OPT_TIMING, 0)
        assert ll.status() == 0, "a kernel's bounded wait ran out"
        shape = ll.describe(w.T, w.seg_offsets, w.seg_ids)
    ms = e0.elapsed_time(e1) / steps
    k_ms = kernel_ms / max(1, n_timed)
    alg = _alg_bytes(w)
    peak_burst, _, hbm, src = _peaks()
    gbs = alg / (k_ms * 1e-3) / 1e9
    return {"workload": w.name, "T": w.T, "d_in": w.d_in, "d_out": w.d_out, "segments": len(w.seg_ids),
            "adapter_rows": w.adapter_rows, "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 5),
            "value": round(w.useful_flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "tokens_per_s": round(w.T / (ms * 1e-3), 1), "kernel_ms": round(k_ms, 5),
            "gpu_launches": n_all - n0,
            "l2": _l2_note([(w, 0, 0)], 3),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "traffic": _profiled_traffic(w.name),
                         "peak_source": f"{src} copy bandwidth", "kernel": "lora_gemm_kernel",
                         "algorithmic_bytes_per_step": alg},
            "launch_shape": shape, "clocks": sampler.summary(t0, t1)}


# --------------------------------------------------------------------------- ranks

def aggregate_ranks(elapsed_ms, e2e_ms, flops_per_step, steps, world, dist):
    """Slowest rank's device and end-to-end times; whole-job TFLOP/s (every rank runs the
    workload: replicas, so the job's work is world x one rank's)."""
    if dist is not None:
        import torch
        t = torch.tensor([elapsed_ms, e2e_ms], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms, e2e_ms = float(t[0]), float(t[1])
    value = world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12
    e2e_value = world * flops_per_step / (e2e_ms * 1e-3) / 1e12
    return elapsed_ms, e2e_ms, value, e2e_value


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, dist):
    import torch
    from mixed_lora_projection_gb300 import LoraLinear, w4_repack, _lib as L
    from mixed_lora_projection_gb300.synth import make_inputs, make_w4_base

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    items = _workloads(args.workload)
    n_copies = 1 if args.workload in (SWEEP, SWEEP_MULTI, DECODE_SWEEP) else 3
    setups = []
    handles = {}
    for (w, layer, pi) in items:
        key = (w.d_in, w.d_out, w.rank)
        if key not in handles:
            handles[key] = LoraLinear(w.d_in, w.d_out, w.rank, w.T, max(8, len(w.seg_ids)), dev)
            if args.two_launch:
                handles[key].set_option(L.OPT_TWO_LAUNCH, 1)
            if args.k_split:
                handles[key].set_option(L.OPT_K_SPLIT, args.k_split)
            if args.pdl:
                handles[key].set_option(L.OPT_PDL, 1)
            if args.token_columns:
                handles[key].set_option(L.OPT_TOKEN_COLUMNS, args.token_columns)
            if args.wide_tiles:
                handles[key].set_option(L.OPT_WIDE_TILES, args.wide_tiles)
            if args.raster:
                mode, _, group = args.raster.partition(":")
                handles[key].set_option(L.OPT_RASTER, int(mode))
                if group:
                    handles[key].set_option(L.OPT_RASTER_GROUP, int(group))
        copies = [make_inputs(w, dev, layer=layer, proj_index=pi + 4 * c, with_x=(c == 0)) for c in range(n_copies)]
        if args.w4:
            for c, inp in enumerate(copies):
                q, sc = make_w4_base(w, dev, layer=layer, proj_index=pi + 4 * c)
                inp.w = (w4_repack(q, q), sc)   # once, at load time: plain -> kernel layout
        y = torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
        setups.append((w, handles[key], copies, y))
    stream = torch.cuda.current_stream(dev)

    def step(i, s=None):
        s = s or stream
        for (w, ll, copies, y) in setups:
            c = copies[i % len(copies)]
            if args.w4:
                ll.forward_w4(copies[0].x, w.seg_offsets, w.seg_ids, c.w[0], c.w[1], c.a, c.b, c.scales, y=y,
                              stream=s)
            else:
                ll.forward(copies[0].x, w.seg_offsets, w.seg_ids, c.w, c.a, c.b, c.scales, y=y, stream=s)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    for ll in handles.values():
        assert ll.status() == 0
        ll.set_option(L.OPT_TIMING, 1)
    launches0 = sum(ll.timing(1)[2] for ll in handles.values())

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # one event per step boundary: the total over the K steps is the reported time; the
    # per-step durations give the median / min / max beside it
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t0 = time.time()
    evs[0].record(stream)
    for i in range(args.steps):
        step(i)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist:
        dist.barrier()
    elapsed_ms = evs[0].elapsed_time(evs[-1])
    step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    launches = sum(ll.timing(1)[2] for ll in handles.values()) - launches0
    fused_ms = sum(ll.timing(1)[0] for ll in handles.values())
    fused_n = sum(ll.timing(1)[1] for ll in handles.values())
    shrink_ms = sum(ll.timing(0)[0] for ll in handles.values())
    shrink_n = sum(ll.timing(0)[1] for ll in handles.values())
    for ll in handles.values():
        ll.set_option(L.OPT_TIMING, 0)
        assert ll.status() == 0, "a kernel's bounded wait ran out"
    graph = None
    if args.graph:
        # the same steps replayed from CUDA graphs (one captured step per rotating weight copy)
        n_graphs = len(setups[0][2])
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for i in range(n_graphs):
                step(i, side)                         # the shapes once before capture
        stream.wait_stream(side)
        torch.cuda.synchronize()
        c0 = sum(ll.timing(1)[2] for ll in handles.values())
        graphs = []
        for i in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(i, torch.cuda.current_stream(dev))   # the capture stream
            graphs.append(g)
        per_step = (sum(ll.timing(1)[2] for ll in handles.values()) - c0) // n_graphs
        for i in range(args.warmup):
            graphs[i % n_graphs].replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        replay_stream = torch.cuda.current_stream(dev)
        t0 = time.time()
        g0.record(replay_stream)
        for i in range(args.steps):
            graphs[i % n_graphs].replay()
        g1.record(replay_stream)
        torch.cuda.synchronize()
        t1 = time.time()
        graph = {"ms_per_step": g0.elapsed_time(g1) / args.steps, "launches_per_step": per_step}
        for ll in handles.values():
            assert ll.status() == 0, "a kernel's bounded wait ran out"
    time.sleep(0.1)
    sampler.stop()

    # e2e: the host-buffer entry point, X in and Y out every step
    x_host = [s[2][0].x.cpu().pin_memory() for s in setups]
    y_host = [torch.empty((s[0].T, s[0].d_out), dtype=torch.bfloat16).pin_memory() for s in setups]

    def e2e_step(i):
        for j, (w, ll, copies, y) in enumerate(setups):
            c = copies[i % len(copies)]
            if args.w4:
                ll.forward_host_w4(x_host[j], w.seg_offsets, w.seg_ids, c.w[0], c.w[1], c.a, c.b, c.scales, y_host[j],
                                   stream=stream)
            else:
                ll.forward_host(x_host[j], w.seg_offsets, w.seg_ids, c.w, c.a, c.b, c.scales, y_host[j], stream=stream)

    for i in range(min(args.warmup, 3)):
        e2e_step(i)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    te0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - te0) * 1e3 / e2e_steps
    if dist:
        dist.barrier()

    flops = _flops_of(items)
    eager = None
    if graph is not None:
        # the headline numbers come from the graph replays; the eager pass stays for reference
        eager = {"ms_per_step": round(elapsed_ms / args.steps, 5),
                 "value": round(world * flops / (elapsed_ms / args.steps * 1e-3) / 1e12, 2)}
        elapsed_ms = graph["ms_per_step"] * args.steps
        launches = graph["launches_per_step"] * args.steps
    elapsed_ms, e2e_ms, value, e2e_value = aggregate_ranks(elapsed_ms, e2e_ms, flops, args.steps, world, dist)
    ms_per_step = elapsed_ms / args.steps
    peak_burst, peak_sust, hbm, src = _peaks()
    # the timed kernel: the one launch per call (shrink + base + expand), or, in two-launch
    # mode, the fused base+expand launch alone
    fused_flops = sum((_fused_flops(w) if shrink_n else w.useful_flops()) for w, _, _ in items)
    avg_fused_ms = fused_ms / args.steps if fused_n else None  # device time of the fused launches per step
    achieved = fused_flops / (avg_fused_ms * 1e-3) / 1e12 if avg_fused_ms else None
    traffic = _profiled_traffic(args.workload + ("+w4" if args.w4 else ""))
    w0 = items[0][0]
    roof, roof_other = _rooflines(items, args.w4, fused_flops, avg_fused_ms, traffic, peak_burst, hbm, src, shrink_n,
                                  peak_sust)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "step_ms": {"median": round(step_ms[len(step_ms) // 2], 5), "min": round(step_ms[0], 5),
                    "max": round(step_ms[-1], 5), "of": "eager steps, rank 0"},
        "data": "synthetic (seeded Gaussian bf16; no checkpoint)",
        "config": {"workload": args.workload + ("+w4" if args.w4 else ""),
                   **({"raster": args.raster} if args.raster else {}),
                   **({"k_split": args.k_split} if args.k_split else {}),
                   **({"pdl": True} if args.pdl else {}),
                   **({"token_columns": args.token_columns} if args.token_columns else {}),
                   **({"wide_tiles": args.wide_tiles} if args.wide_tiles else {}),
                   "base": "int4 (symmetric, group 128, bf16 scales)" if args.w4 else "bf16", "T": w0.T, "d_in": w0.d_in if len(items) == 1 else "per projection",
                   "d_out": w0.d_out if len(items) == 1 else "per projection", "rank": w0.rank,
                   "segments": len(w0.seg_ids), "adapter_rows": w0.adapter_rows, "calls_per_step": len(items),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": _l2_note(items, n_copies, args.w4)},
        "tokens_per_s": round(world * _tokens_of(items) * args.steps / (elapsed_ms * 1e-3), 1),
        "roofline": roof,
        **({"roofline_other": roof_other} if roof_other else {}),
        "kernel_ms": {"main": round(fused_ms / max(1, args.steps), 5), "separate_shrink": round(shrink_ms / max(1, args.steps), 5),
                      "main_launches": fused_n, "separate_shrink_launches": shrink_n},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(2 * w.T * w.d_in for w, _, _ in items),
                "d2h_bytes_per_step": sum(2 * w.T * w.d_out for w, _, _ in items),
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps},
        "gpu_launches": launches,
        "cuda_graph": ({"replayed": True, "launches_per_step": graph["launches_per_step"], "eager": eager}
                       if graph is not None else None),
        "launch_shape": setups[0][1].describe(w0.T, w0.seg_offsets, w0.seg_ids),
        "clocks": sampler.summary(t0, t1),
    }
    if args.workload == "prefill_16k" and not args.w4 and not args.no_decode:
        # the decode-sized batch beside the headline: the HBM roof, in the same process
        out["decode"] = decode_line(dev, args.decode_steps, max(args.warmup, 20))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(items, args.cpu_seconds, args.w4)
    for ll in handles.values():
        ll.close()
    return out


# --------------------------------------------------------------------------- oracle timing

def _oracle_block(w, layer, pi, rows, seed_rows=0, w4=False):
    """Inputs for a contiguous block of `rows` rows of workload w (starting at row 0), as
    exact fp64 values, and the segments restricted to the block. With w4 the base weight is
    the workload's seeded 4-bit base, widened to bf16 as the oracle defines it (built here,
    outside the timed call, like a weight being loaded)."""
    import numpy as np
    from mixed_lora_projection_gb300.synth import bf16_bits, make_inputs, make_w4_base
    from oracle import bf16_bits_to_f64, w4_weights_bf16_fp64
    inp = make_inputs(w, "cpu", layer=layer, proj_index=pi, x_rows=rows)
    f = lambda t: bf16_bits_to_f64(bf16_bits(t))  # noqa: E731
    if w4:
        q, sc = make_w4_base(w, "cpu", layer=layer, proj_index=pi)
        wmat = w4_weights_bf16_fp64(q.numpy(), bf16_bits(sc))
    else:
        wmat = f(inp.w)
    off, ids = [0], []
    for i, a in enumerate(w.seg_ids):
        lo, hi = min(w.seg_offsets[i], rows), min(w.seg_offsets[i + 1], rows)
        if hi > lo:
            off.append(hi)
            ids.append(a)
    return f(inp.x), off, ids, wmat, [f(a) for a in inp.a], [f(b) for b in inp.b], inp.scales


def _block_flops(w, off, ids):
    rows = off[-1]
    ta = sum(off[i + 1] - off[i] for i, a in enumerate(ids) if a)
    return 2.0 * rows * w.d_in * w.d_out + 2.0 * ta * w.rank * (w.d_in + w.d_out)


def _blas_threads():
    """Threads of the BLAS behind numpy's matmul (what the oracle runs on), or None."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    import ctypes
    import glob
    import numpy
    for path in glob.glob(os.path.join(os.path.dirname(numpy.__file__), os.pardir, "numpy.libs", "*openblas*")):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                     "openblas_get_num_threads64_", "openblas_get_num_threads"):
            f = getattr(lib, name, None)
            if f is not None:
                return int(f())
    return None


def _host_threads():
    """(threads the oracle uses, cores in this process's affinity mask)."""
    affinity = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    blas = _blas_threads()
    return (min(blas, affinity) if blas else affinity), affinity


def cpu_baseline(items, seconds, w4=False):
    """The fp64 oracle, as it stands, on a contiguous block of the workload's rows, sized
    to about `seconds` of host time."""
    from oracle import lora_linear_fp64
    w, layer, pi = items[0]
    cores, affinity = _host_threads()
    rows = min(w.T, 64)
    data = _oracle_block(w, layer, pi, rows, w4=w4)
    t = time.perf_counter()
    lora_linear_fp64(*data)
    dt = time.perf_counter() - t
    rate = _block_flops(w, data[1], data[2]) / max(dt, 1e-6)
    rows = int(min(w.T, max(64, rows * seconds / max(dt, 1e-6) * 0.8)))
    data = _oracle_block(w, layer, pi, rows, w4=w4)
    t = time.perf_counter()
    lora_linear_fp64(*data)
    dt = time.perf_counter() - t
    fl = _block_flops(w, data[1], data[2])
    return {"value": round(fl / dt / 1e12, 5), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "host_cores": affinity,
            "sample": f"rows [0,{rows}) of {w.name} ({w.T} rows), layer 0, all {w.d_out} outputs: "
                      f"{fl / 1e9:.1f} GFLOP fp64 in {dt:.1f} s (numpy/OpenBLAS, {cores} BLAS threads)"
                      + ("; base: the 4-bit weights widened to bf16" if w4 else "")}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every step is a bounded sample of the workload."""
    from oracle import lora_linear_fp64
    items = _workloads(args.workload)
    w, layer, pi = items[0]
    w4 = args.w4
    cores, affinity = _host_threads()
    budget = max(0.05, args.cpu_seconds * 4 / max(1, args.steps + args.warmup))  # ~a few minutes in all
    rows = min(w.T, 32)
    data = _oracle_block(w, layer, pi, rows, w4=w4)
    t = time.perf_counter()
    lora_linear_fp64(*data)
    dt = time.perf_counter() - t
    rows = int(min(w.T, max(8, rows * budget / max(dt, 1e-6))))
    data = _oracle_block(w, layer, pi, rows, w4=w4)
    fl = _block_flops(w, data[1], data[2])
    for _ in range(args.warmup):
        lora_linear_fp64(*data)
    t = time.perf_counter()
    for _ in range(args.steps):
        lora_linear_fp64(*data)
    dt = (time.perf_counter() - t) / args.steps
    value = fl / dt / 1e12
    sample = (f"rows [0,{rows}) of {w.name} per step ({w.T} rows in the full batch), all {w.d_out} outputs, fp64"
              + ("; base: the 4-bit weights widened to bf16" if w4 else ""))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "host": "rank 0 only, host cores",
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Gaussian bf16 values, exact in fp64)",
            "config": {"workload": args.workload + ("+w4" if w4 else ""),
                       "base": "int4 (symmetric, group 128, bf16 scales)" if w4 else "bf16",
                       "T": w.T, "d_in": w.d_in, "d_out": w.d_out, "rank": w.rank, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "host_cores": affinity, "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="prefill_16k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-sized batch timed beside the default "
                    "16k prefill")
    ap.add_argument("--decode-steps", type=int, default=4000)
    ap.add_argument("--two-launch", action="store_true", help="shrink as its own launch (for comparison)")
    ap.add_argument("--w4", action="store_true", help="4-bit base weights (int4, group 128, bf16 scales)")
    ap.add_argument("--raster", default="", help="unit order MODE[:GROUP] (the library's raster option: 0 auto, "
                    "1 row tiles first, 2 column tiles first, 3 groups of GROUP column tiles)")
    ap.add_argument("--k-split", type=int, default=0, choices=[0, 1, 2, 4], help="K parts per output block (the "
                    "library's K-split option: 0 = each handle's own choice, 1 = whole K, 2 or 4 parts)")
    ap.add_argument("--pdl", action="store_true", help="programmatic dependent launch for calls without adapter "
                    "rows (the library's PDL option): each kernel may start while the previous one ends")
    ap.add_argument("--token-columns", type=int, default=0, choices=[0, 1, 2], help="token-column units (the "
                    "library's option: 0 = when the shape model expects them sooner, 1 = never, 2 = whenever the "
                    "batch allows)")
    ap.add_argument("--wide-tiles", type=int, default=0, choices=[0, 1], help="wide row tiles (the library's "
                    "option: 0 = when the shape model expects them sooner, 1 = never)")
    ap.add_argument("--graph", action="store_true", help="time the steps as CUDA-graph replays (each call's "
                    "work list must travel in the kernel parameters, e.g. the 24-layer sweep)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as D
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            D.init_process_group("nccl")
            dist = D
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
