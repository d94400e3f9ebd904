"""Benchmark of the GGD-BAM attention hot path on GB300.

Default workload: the training step fwd+bwd at B=8, H=12, T=512, D=64,
causal, BAM+SSMax (seeded synthetic bf16 tensors shaped like the pages'
T=512 training runs).  A step is one forward and one backward through the C
ABI (distance tables, fused forward, backward preprocess, fused backward,
finalisation).  Throughput counts the algorithmic causal work: B*H*T(T+1)/2
query-key pairs at 4*D flop (forward) + 10*D flop (backward) per pair.

One JSON line on rank 0 with the device-timed value, the end-to-end value
through host buffers, the roofline of the dominant kernel (timed live with
the library's event hook), the fp64 CPU oracle as a baseline, the launch
count and the SM clocks seen during the timed region.  Extra lines of the
other workloads (long-context prefill, decode) are reported under "extra".

--impl reference times the oracle (the method's plain fp64 statement) on the
host cores on the same workload, bounded samples per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BAM attention causal fwd/bwd TFLOP/s and % of BF16 tensor peak; decode GB/s"
D = 64


def hook_events(torch, n):
    """n (before, after) CUDA event pairs for the library's profiling hook.
    torch creates the underlying event on the first record(), so record each
    once here; the library then re-records them around its launches."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        a.record()
        b.record()
    torch.cuda.synchronize()
    return evs


def pairs_causal(B, H, T):
    return B * H * T * (T + 1) // 2


def train_flops(B, H, T):
    return pairs_causal(B, H, T) * (4 * D + 10 * D)


# Nominal HBM3e bandwidth of a GB300, about 8 TB/s: decode entries report their
# fraction of it beside the fraction of the measured copy bandwidth (a
# read-only stream can beat a read+write copy, so the latter may exceed 1).
HBM_NOMINAL_GBS = 8000.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The files each profiled kernel is compiled from: its .cu, the headers it
# includes, and the build script (compiler flags).
# Cycles of the GPU spin queued ahead of the timed training steps (~2 ms at
# 2 GHz; the host enqueues a step's flush, events and graph launch in tens of
# microseconds).
STEP_SPIN_CYCLES = 4_000_000

# Cycles of the GPU spin that each timed call of `extra_workloads` is queued
# behind (~0.25 ms at 2 GHz, longer than the host needs to check a call's
# arguments and enqueue its kernels).
CALL_SPIN_CYCLES = 500_000


KERNEL_SOURCES = {
    "bam_bwd_kernel": ("bwd.cu", "table_eval.cuh", "bam_common.cuh", "bam_ptx.cuh"),
    "bam_fwd_kernel": ("fwd.cu", "bam_common.cuh", "bam_ptx.cuh"),
    "bam_fwd_single_kernel": ("fwd.cu", "bam_common.cuh", "bam_ptx.cuh"),
    "bam_decode_kernel": ("decode.cu", "bam_common.cuh", "bam_ptx.cuh"),
}


def kernel_source_hash(kernel=None):
    """16 hex digits of sha256 over the sources of `kernel` (every file under
    csrc/ when None)."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "transformer_attention_ggd_gb300")
    csrc = os.path.join(pkg, "csrc")
    names = sorted(os.listdir(csrc)) if kernel is None else KERNEL_SOURCES[kernel]
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    if kernel is not None:
        with open(os.path.join(pkg, "build.py"), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    entry = t.get(kernel)
    if not entry or entry.get("source_hash") != kernel_source_hash(kernel.split("@")[0]):
        return None
    return entry.get("dram_bytes_per_launch")


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed
    captures: the entry `kernel` or `kernel@workload` whose workload matches,
    if it was taken on the current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    for key in (kernel, f"{kernel}@{workload}"):
        entry = t.get(key)
        if entry and entry.get("workload") == workload:
            return profiled_traffic(key)
    return None


def _nvtx(torch, name):
    """Open (name given) or close an NVTX range around a bench phase, for a
    profiler's timeline; a no-op where NVTX is unavailable."""
    try:
        if name is None:
            torch.cuda.nvtx.range_pop()
        else:
            torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        # The timed region starts only once nvidia-smi has delivered a sample
        # (its driver set-up done), so that set-up does not overlap the steps.
        t0 = time.monotonic()
        while self.proc is not None and not self.lines and time.monotonic() - t0 < 5.0:
            time.sleep(0.01)
        time.sleep(0.15)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def make_train_inputs(torch, dev, seed=None):
    from transformer_attention_ggd_gb300.inputs import make_inputs
    d = make_inputs(2, seed=seed)

    def bf(b):
        return torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)

    t = {n: bf(d[n]) for n in ("q", "k", "v", "do")}
    for n in ("alpha", "beta", "mu", "s"):
        t[n] = torch.from_numpy(d[n]).to(dev)
    return d, t


def run_ours(args, rank, world, dev, torch, dist):
    from transformer_attention_ggd_gb300 import bam_attn as ba
    from transformer_attention_ggd_gb300.dist_utils import max_over_ranks

    ba.load_library()
    peaks = load_peaks()
    B, H, T = 8, 12, 512
    d, t = make_train_inputs(torch, dev, seed=args.seed + rank)
    prm = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    o = torch.empty((B, H, T, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    g = [torch.empty(H, dtype=torch.float32, device=dev) for _ in range(4)]
    ws_f = ba.workspace(ba.BAM_OP_FWD, B, H, T, dev)
    ws_b = ba.workspace(ba.BAM_OP_BWD, B, H, T, dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2

    def step(q, k, v, do):
        # current stream at call time (the capture stream while capturing)
        ba.bam_attn_fwd(q, k, v, o, lse, prm, ws_f)
        ba.bam_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, g[0], g[1], g[2], g[3], prm, ws_b)

    for _ in range(args.warmup):
        step(t["q"], t["k"], t["v"], t["do"])
    torch.cuda.synchronize()
    if ba.bam_attn_check_status(ws_b) != ba.BAM_OK or ba.bam_attn_check_status(ws_f) != ba.BAM_OK:
        raise RuntimeError("device status not clean after warm-up")

    # The step's launches (two C-ABI calls, five kernels) are captured once
    # into a CUDA graph and replayed, so that host launch latency does not
    # leave the GPU idle between kernels.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def capture(fn):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()  # one eager call on the capture stream first
        torch.cuda.synchronize()
        with torch.cuda.graph(g_, stream=side):
            fn()
        torch.cuda.synchronize()
        return g_

    launches0 = ba.bam_attn_launch_count()
    graph = capture(lambda: step(t["q"], t["k"], t["v"], t["do"]))
    launches_per_step = (ba.bam_attn_launch_count() - launches0) // 2
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # Device-timed steps; L2 flushed between steps (outside the events).
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    _nvtx(torch, "timed training steps")
    with ClockSampler(torch.cuda.current_device()) as clk:
        # A GPU spin ahead of the steps (outside their events) lets the host
        # enqueue all K of them before the first runs, so that a pause on the
        # host cannot leave the GPU idle inside a step's interval.
        torch.cuda._sleep(STEP_SPIN_CYCLES)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record()
            graph.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
    _nvtx(torch, None)
    if world > 1:
        dist.barrier()
    launches = launches_per_step * args.steps
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dist, dev)
    flops_step = train_flops(B, H, T)
    value = flops_step * args.steps * world / (total_ms * 1e-3) / 1e12

    # Per-kernel durations: a second graph of the same step whose kernels are
    # bracketed by the library's event hook (event-record nodes in the graph).
    kinds = (ba.BAM_KERNEL_TABLE, ba.BAM_KERNEL_FWD, ba.BAM_KERNEL_BWD_PREP, ba.BAM_KERNEL_BWD,
             ba.BAM_KERNEL_BWD_FINAL)
    kev = {k: hook_events(torch, 1)[0] for k in kinds}
    for k, (b0, b1) in kev.items():
        ba.bam_attn_profile_events(k, b0, b1)
    kgraph = capture(lambda: step(t["q"], t["k"], t["v"], t["do"]))
    for k in kinds:
        ba.bam_attn_profile_events(k, None, None)
    kms = {k: [] for k in kinds}
    gaps = []
    for i in range(args.steps):
        flush.zero_()
        kgraph.replay()
        torch.cuda.synchronize()
        for k, (b0, b1) in kev.items():
            kms[k].append(b0.elapsed_time(b1))
        # Between one kernel's closing record and the next kernel's opening
        # record nothing runs: that interval is the cost of an empty bracket
        # (two event-record nodes), which every bracketed time also carries.
        for k0, k1 in zip(kinds[:-1], kinds[1:]):
            gaps.append(kev[k0][1].elapsed_time(kev[k1][0]))
    kern_ms_raw = {k: statistics.mean(v) for k, v in kms.items()}
    bracket_ms = statistics.median(gaps)
    kern_ms = {k: max(v - bracket_ms, 1e-6) for k, v in kern_ms_raw.items()}

    # End to end through the C ABI with host buffers, as a training loop
    # streams them: every step copies its inputs from pinned host memory
    # (H2D) and reads its gradients back (D2H), and the copies of the steps
    # before and after overlap the current step's kernels (double-buffered
    # device inputs and gradients, one stream each for H2D, compute and
    # D2H).  Timed from the first H2D to the last D2H over all K steps.
    # A step's inputs (q, k, v, dO) sit in one pinned block and its outputs
    # (dq, dk, dv and the [4, H] scalar gradients) in another, each with a
    # contiguous device twin: one copy per direction per step.  On the box
    # one 25 MB copy runs at ~205 GB/s host to device and one 19 MB copy at
    # ~187 GB/s back, ~310 GB/s together; four copies per direction per step
    # left ~15% of that unused (gaps between copies).
    names = ("q", "k", "v", "do")
    tin = t["q"].numel() * t["q"].element_size()  # bytes of one bf16 [B, H, T, D] tensor

    def carve(buf):
        """Views of one byte block as q, k, v, dO (bf16, shaped like t[...])."""
        return {n: buf[j * tin:(j + 1) * tin].view(torch.bfloat16).view(t[n].shape)
                for j, n in enumerate(names)}

    def carve_out(buf):
        """Views of one byte block as dq, dk, dv (bf16) and the [4, H] scalars."""
        g3 = [buf[j * tin:(j + 1) * tin].view(torch.bfloat16).view(dq.shape) for j in range(3)]
        return g3, buf[3 * tin:3 * tin + 16 * H].view(torch.float32).view(4, H)

    host_in_buf = torch.empty(4 * tin, dtype=torch.uint8).pin_memory()
    host_in = carve(host_in_buf)
    for n in names:
        host_in[n].copy_(t[n].cpu())
    nb = 2
    dev_in_buf = [torch.empty(4 * tin, dtype=torch.uint8, device=dev) for _ in range(nb)]
    dev_in = [carve(x) for x in dev_in_buf]
    out_bytes = 3 * tin + 16 * H
    dev_out_buf = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(nb)]
    dev_out = [carve_out(x) for x in dev_out_buf]
    host_out_buf = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    h2d = host_in_buf.numel()
    d2h = out_bytes
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(K, check):
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_cmp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for st in (s_h2d, s_cmp, s_d2h):
            st.wait_stream(torch.cuda.current_stream())
        t0.record(s_h2d)
        for i in range(K + 2):
            if i < K:  # H2D of step i (its buffer's previous step is computed)
                b = i % nb
                with torch.cuda.stream(s_h2d):
                    if i >= nb:
                        s_h2d.wait_event(ev_cmp[b])
                    dev_in_buf[b].copy_(host_in_buf, non_blocking=True)
                    ev_in[b].record(s_h2d)
            if 1 <= i <= K:  # kernels of step i-1
                b = (i - 1) % nb
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in[b])
                    if i - 1 >= nb:
                        s_cmp.wait_event(ev_out[b])
                    (gq, gk, gv), gs = dev_out[b]
                    x = dev_in[b]
                    ba.bam_attn_fwd(x["q"], x["k"], x["v"], o, lse, prm, ws_f, check=check)
                    ba.bam_attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], gq, gk, gv,
                                    gs[0], gs[1], gs[2], gs[3], prm, ws_b, check=check)
                    ev_cmp[b].record(s_cmp)
            if 2 <= i <= K + 1:  # D2H of step i-2
                b = (i - 2) % nb
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(ev_cmp[b])
                    host_out_buf[b].copy_(dev_out_buf[b], non_blocking=True)
                    ev_out[b].record(s_d2h)
        t1.record(s_d2h)
        t1.synchronize()
        return t0.elapsed_time(t1)

    # The warm-up pass checks every buffer (and fails loudly on a bad one);
    # the timed pass reuses the same preallocated buffers with check=False.
    e2e_run(max(3, args.warmup), check=True)
    torch.cuda.synchronize()
    flush.zero_()
    torch.cuda.synchronize()
    _nvtx(torch, "end-to-end steps")
    e_ms = e2e_run(args.steps, check=False)
    _nvtx(torch, None)
    if world > 1:
        e_ms = max_over_ranks(e_ms, dist, dev)
    e2e_value = flops_step * args.steps * world / (e_ms * 1e-3) / 1e12

    # Roofline of the dominant kernel (the fused backward): algorithmic
    # flops of one launch (10 D per causal pair) over its mean duration.
    bwd_flops = pairs_causal(B, H, T) * 10 * D
    fwd_flops = pairs_causal(B, H, T) * 4 * D
    dom = ba.BAM_KERNEL_BWD if kern_ms[ba.BAM_KERNEL_BWD] >= kern_ms[ba.BAM_KERNEL_FWD] \
        else ba.BAM_KERNEL_FWD
    dom_flops = bwd_flops if dom == ba.BAM_KERNEL_BWD else fwd_flops
    achieved = dom_flops / (kern_ms[dom] * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    # The forward of this workload runs the persistent single-tile kernel
    # (fewer than two waves of 256-row CTAs at B=8 H=12 T=512).
    dom_name = "bam_bwd_kernel" if dom == ba.BAM_KERNEL_BWD else "bam_fwd_single_kernel"
    roof = {"kernel": dom_name,
            "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": traffic_for(dom_name, f"train_B{B}_H{H}_T{T}"),
            "peak_source": f"{peaks['source']} bf16 burst (cuBLAS)",
            "kernel_ms": {"table": round(kern_ms[ba.BAM_KERNEL_TABLE], 4),
                          "fwd": round(kern_ms[ba.BAM_KERNEL_FWD], 4),
                          "bwd_prep": round(kern_ms[ba.BAM_KERNEL_BWD_PREP], 4),
                          "bwd": round(kern_ms[ba.BAM_KERNEL_BWD], 4),
                          "bwd_final": round(kern_ms[ba.BAM_KERNEL_BWD_FINAL], 4)},
            "kernel_ms_method": "event-bracketed kernel in a second graph of the step, minus "
                                "the empty-bracket time measured between consecutive "
                                "brackets of the same replay",
            "bracket_ms": round(bracket_ms, 4),
            "kernel_ms_raw": {"fwd": round(kern_ms_raw[ba.BAM_KERNEL_FWD], 4),
                              "bwd": round(kern_ms_raw[ba.BAM_KERNEL_BWD], 4)},
            "fwd_frac": round(fwd_flops / (kern_ms[ba.BAM_KERNEL_FWD] * 1e-3) / 1e12 / peak, 4)}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "step_ms_spread": {"min": round(min(step_ms), 5),
                           "median": round(statistics.median(step_ms), 5),
                           "max": round(max(step_ms), 5)},
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 tensors and per-head parameters)",
        "config": {"workload": "train_B8_H12_T512", "B": B, "H": H, "T": T, "D": D,
                   "causal": True, "ssmax": True, "step": "fwd+bwd",
                   "l2": "flushed (256 MB write) between timed steps",
                   "launch": "CUDA graph of the two C-ABI calls, replayed per step",
                   "seed": f"{args.seed} + rank",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms / args.steps, 5),
                "mode": "streamed: each step's pinned-host H2D of q, k, v, dO (one 25 MB "
                        "block, one copy) and D2H of dq, dk, dv and the scalar gradients "
                        "(one block, one copy), overlapping the neighbouring steps' "
                        "kernels (double-buffered, one copy stream per direction, eager "
                        "C-ABI calls; tensor checks on the warm-up pass, check=False on the "
                        "timed pass over the same preallocated buffers)"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    return line, t


def gpu_call_ms(torch, call, a, b):
    """GPU time of one library call: the call is enqueued behind a short spin
    kernel, so the start event fires with the call's kernels already queued and
    the host's argument checks and launches stay out of the interval (as in a
    serving loop that keeps the stream full).  The interval still holds the
    call's kernels and the gaps between them."""
    torch.cuda._sleep(CALL_SPIN_CYCLES)
    a.record()
    call()
    b.record()
    b.synchronize()
    return a.elapsed_time(b)


def extra_workloads(torch, dev, steps, peaks, cpu=True):
    """The other workloads of the method, timed briefly: the small forward
    (workload 1), the long-context prefills (causal, and the 32k one
    non-causal too) and decode.  With `cpu`, each entry also carries the fp64
    oracle's rate on the same inputs (in full, or on a stated sample)."""
    from transformer_attention_ggd_gb300 import bam_attn as ba
    from transformer_attention_ggd_gb300.inputs import make_inputs

    out = {}

    def bf(b):
        return torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)

    for cfg, reps, causal in ((1, max(5, steps), True), (3, max(3, steps // 4), True),
                              (4, 3, True), (3, max(3, steps // 4), False)):
        d = make_inputs(cfg)
        q, k, v = bf(d["q"]), bf(d["k"]), bf(d["v"])
        p = {n: torch.from_numpy(d[n]).to(dev) for n in ("alpha", "beta", "mu", "s")}
        B, H, T = d["B"], d["H"], d["T"]
        ssmax = bool(d["ssmax"])
        prm = ba.make_params(p["alpha"], p["beta"], p["mu"], p["s"], 1e-5, causal, ssmax)
        o = torch.empty((B, H, T, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        ws = ba.workspace(ba.BAM_OP_FWD, B, H, T, dev)
        ba.bam_attn_fwd(q, k, v, o, lse, prm, ws)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        (ka, kb_), = hook_events(torch, 1)
        ms, kms = [], []
        for _ in range(reps):
            ba.bam_attn_profile_events(ba.BAM_KERNEL_FWD, ka, kb_)
            ms.append(gpu_call_ms(torch, lambda: ba.bam_attn_fwd(q, k, v, o, lse, prm, ws),
                                  a, b))
            kms.append(ka.elapsed_time(kb_))
        ba.bam_attn_profile_events(ba.BAM_KERNEL_FWD, None, None)
        fl = (pairs_causal(B, H, T) if causal else B * H * T * T) * 4 * D
        tf = fl / (statistics.median(ms) * 1e-3) / 1e12
        ktf = fl / (statistics.median(kms) * 1e-3) / 1e12
        kind = "fwd" if cfg == 1 else "prefill"
        name = f"{kind}_{'' if causal else 'noncausal_'}B{B}_H{H}_T{T}"
        out[name] = {
            "ms": round(statistics.median(ms), 4), "TFLOP/s": round(tf, 2),
            "fwd_kernel_TFLOP/s": round(ktf, 2),
            "frac_of_bf16_peak": round(ktf / peaks["bf16_tflops"], 4),
            "traffic": traffic_for("bam_fwd_kernel", name)}
        del q, k, v, o, ws
        torch.cuda.empty_cache()
        if cpu:
            out[name]["cpu_baseline"] = (oracle_fwd_full(d, causal) if cfg == 1
                                         else oracle_fwd_sampled(d, causal))

    d = make_inputs(5)
    q, kc, vc = bf(d["q"]), bf(d["k"]), bf(d["v"])
    p = {n: torch.from_numpy(d[n]).to(dev) for n in ("alpha", "beta", "mu", "s")}
    B, H, Tkv = d["B"], d["H"], d["T"]
    prm = ba.make_params(p["alpha"], p["beta"], p["mu"], p["s"], 1e-5, True, True)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tkv, dev)
    ba.bam_attn_decode(q, kc, vc, o, lse, prm, ws)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    (ka, kb_), = hook_events(torch, 1)
    ms, kms = [], []
    for _ in range(max(5, steps // 2)):
        ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, ka, kb_)
        ms.append(gpu_call_ms(torch, lambda: ba.bam_attn_decode(q, kc, vc, o, lse, prm, ws),
                              a, b))
        kms.append(ka.elapsed_time(kb_))
    ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, None, None)
    kv_bytes = 2 * B * H * Tkv * D * 2
    gbs = kv_bytes / (statistics.median(ms) * 1e-3) / 1e9
    kgbs = kv_bytes / (statistics.median(kms) * 1e-3) / 1e9
    name = f"decode_B{B}_H{H}_Tkv{Tkv}"
    out[name] = {
        "ms": round(statistics.median(ms), 4), "GB/s": round(gbs, 1),
        "decode_kernel_GB/s": round(kgbs, 1), "frac_of_hbm": round(kgbs / peaks["hbm_gbs"], 4),
        "frac_of_nominal_hbm": round(kgbs / HBM_NOMINAL_GBS, 4),
        "traffic": traffic_for("bam_decode_kernel", name)}
    if cpu:
        out[name]["cpu_baseline"] = oracle_decode_full(d)

    # Ragged decode on the same cache: seeded lengths U[1, Tkv] per sequence;
    # the bytes are those of the keys each sequence actually holds.
    lens = np.random.default_rng(5005).integers(1, Tkv + 1, B)
    lens[:3] = [1, Tkv, 64]
    lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
    ba.bam_attn_decode_varlen(q, kc, vc, lens_d, o, lse, prm, ws)
    torch.cuda.synchronize()
    ms, kms = [], []
    for _ in range(max(5, steps // 2)):
        ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, ka, kb_)
        ms.append(gpu_call_ms(
            torch, lambda: ba.bam_attn_decode_varlen(q, kc, vc, lens_d, o, lse, prm, ws), a, b))
        kms.append(ka.elapsed_time(kb_))
    ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, None, None)
    if ba.bam_attn_check_status(ws) != ba.BAM_OK:
        raise RuntimeError("ragged decode status not clean")
    kv_bytes = 2 * int(lens.sum()) * H * D * 2
    gbs = kv_bytes / (statistics.median(ms) * 1e-3) / 1e9
    kgbs = kv_bytes / (statistics.median(kms) * 1e-3) / 1e9
    name = f"decode_varlen_B{B}_H{H}_Tmax{Tkv}"
    out[name] = {
        "ms": round(statistics.median(ms), 4), "mean_len": round(float(lens.mean()), 1),
        "GB/s": round(gbs, 1), "decode_kernel_GB/s": round(kgbs, 1),
        "frac_of_hbm": round(kgbs / peaks["hbm_gbs"], 4),
        "frac_of_nominal_hbm": round(kgbs / HBM_NOMINAL_GBS, 4),
        "traffic": traffic_for("bam_decode_kernel", name)}

    # Paged decode: the same ragged cache in 256-key pages, randomly permuted
    # (page p of the [B * Tkv/256] blocks stored at slot perm[p]).
    page = 256
    mb = Tkv // page
    perm = torch.randperm(B * mb, generator=torch.Generator().manual_seed(6)).to(dev)
    table = perm.view(B, mb).to(torch.int32)
    pools = []
    for c in (kc, vc):
        blocks = c.view(B, H, mb, page, D).permute(0, 2, 1, 3, 4).reshape(B * mb, H, page, D)
        pool = torch.empty_like(blocks)
        pool[perm] = blocks
        pools.append(pool)
        del blocks
    ba.bam_attn_decode_paged(q, pools[0], pools[1], table, lens_d, o, lse, prm, ws)
    torch.cuda.synchronize()
    ms, kms = [], []
    for _ in range(max(5, steps // 2)):
        ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, ka, kb_)
        ms.append(gpu_call_ms(
            torch,
            lambda: ba.bam_attn_decode_paged(q, pools[0], pools[1], table, lens_d, o, lse, prm,
                                             ws), a, b))
        kms.append(ka.elapsed_time(kb_))
    ba.bam_attn_profile_events(ba.BAM_KERNEL_DECODE, None, None)
    if ba.bam_attn_check_status(ws) != ba.BAM_OK:
        raise RuntimeError("paged decode status not clean")
    gbs = kv_bytes / (statistics.median(ms) * 1e-3) / 1e9
    kgbs = kv_bytes / (statistics.median(kms) * 1e-3) / 1e9
    name = f"decode_paged{page}_B{B}_H{H}_Tmax{Tkv}"
    out[name] = {
        "ms": round(statistics.median(ms), 4), "mean_len": round(float(lens.mean()), 1),
        "GB/s": round(gbs, 1), "decode_kernel_GB/s": round(kgbs, 1),
        "frac_of_hbm": round(kgbs / peaks["hbm_gbs"], 4),
        "frac_of_nominal_hbm": round(kgbs / HBM_NOMINAL_GBS, 4),
        "traffic": traffic_for("bam_decode_kernel", name)}
    del pools
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- oracle arm

def _oracle_entry(value, unit, seconds, sample, extra=None):
    e = {"value": round(value, 6), "unit": unit, "cores": os.cpu_count() or 1, "kind": "oracle",
         "seconds": round(seconds, 3), "sample": sample}
    if extra:
        e.update(extra)
    return e


def oracle_fwd_full(d, causal):
    """The fp64 oracle's forward over a whole (small) workload."""
    import oracle
    from transformer_attention_ggd_gb300.inputs import bf16_to_f64
    oracle.build()
    B, H, T = d["B"], d["H"], d["T"]
    x = {n: bf16_to_f64(d[n]) for n in ("q", "k", "v")}
    t0 = time.perf_counter()
    oracle.fwd(x["q"], x["k"], x["v"], d["alpha"], d["beta"], d["mu"], d["s"], causal=causal,
               ssmax=bool(d["ssmax"]), nthreads=os.cpu_count() or 1)
    dt = time.perf_counter() - t0
    fl = (pairs_causal(B, H, T) if causal else B * H * T * T) * 4 * D
    return _oracle_entry(fl / dt / 1e12, "TFLOP/s", dt,
                         f"fp64 oracle forward of the whole workload (B={B} H={H} T={T})")


def oracle_sample_rows(T, nrows, seed):
    """Stratified query rows of a length-T sequence: one row drawn from each
    of nrows equal strata, with rows 0 and T-1 always included."""
    rng = np.random.default_rng(seed)
    edges = np.linspace(0, T, nrows + 1).astype(np.int64)
    rows = np.array([rng.integers(a, max(a + 1, b)) for a, b in zip(edges[:-1], edges[1:])])
    rows[0], rows[-1] = 0, T - 1
    return np.unique(rows)


def oracle_fwd_sampled(d, causal, nrows=256, seed=7):
    """The fp64 oracle's forward on a stratified sample of query rows of a
    long-context prefill, dealt round-robin over the heads of batch row 0;
    the rate is the sample's algorithmic flops (4 D per visible key) over the
    oracle's time, and the full workload's time is extrapolated by the same
    per-key cost (a causal row i costs i+1 keys)."""
    import oracle
    from transformer_attention_ggd_gb300.inputs import bf16_to_f64
    oracle.build()
    B, H, T = d["B"], d["H"], d["T"]
    rows = oracle_sample_rows(T, nrows, seed)
    dt, keys = 0.0, 0
    for h in range(H):
        mine = rows[h::H]
        if mine.size == 0:
            continue
        x = {n: bf16_to_f64(d[n][0:1, h:h + 1]) for n in ("q", "k", "v")}
        sel = {n: d[n][h:h + 1] for n in ("alpha", "beta", "mu", "s")}
        t0 = time.perf_counter()
        oracle.fwd_rows(x["q"], x["k"], x["v"], mine, sel["alpha"], sel["beta"], sel["mu"],
                        sel["s"], causal=causal, ssmax=bool(d["ssmax"]),
                        nthreads=os.cpu_count() or 1)
        dt += time.perf_counter() - t0
        keys += int((mine + 1).sum()) if causal else mine.size * T
        del x
    fl = keys * 4 * D
    full_keys = (pairs_causal(B, H, T) if causal else B * H * T * T)
    return _oracle_entry(fl / dt / 1e12, "TFLOP/s", dt,
                         f"fp64 oracle forward of {rows.size} stratified query rows (rows 0 and "
                         f"T-1 included) dealt over the {H} heads of batch row 0, "
                         f"extrapolated by keys seen per row",
                         {"extrapolated_full_s": round(full_keys / keys * dt, 1)})


def oracle_decode_full(d):
    """The fp64 oracle's decode over the whole cache, one batch row per call
    (only the oracle calls are timed); the rate is in GB/s of the bf16 K and
    V cache, as the kernel's."""
    import oracle
    from transformer_attention_ggd_gb300.inputs import bf16_to_f64
    oracle.build()
    B, H, Tkv = d["B"], d["H"], d["T"]
    dt = 0.0
    for b in range(B):
        x = {n: bf16_to_f64(d[n][b:b + 1]) for n in ("q", "k", "v")}
        t0 = time.perf_counter()
        oracle.decode(x["q"], x["k"], x["v"], d["alpha"], d["beta"], d["mu"], d["s"],
                      ssmax=bool(d["ssmax"]), nthreads=os.cpu_count() or 1)
        dt += time.perf_counter() - t0
        del x
    kv_bytes = 2 * B * H * Tkv * D * 2
    return _oracle_entry(kv_bytes / dt / 1e9, "GB/s", dt,
                         f"fp64 oracle decode of all {B * H} (b,h) caches (B={B} H={H} "
                         f"Tkv={Tkv}), one batch row per call")


def oracle_sample_step(d, nbh, nthreads):
    """fwd + bwd of the fp64 oracle on the first `nbh` (b, h) pairs of the
    training workload; returns (seconds, flops)."""
    import oracle
    from transformer_attention_ggd_gb300.inputs import bf16_to_f64
    B, H, T = d["B"], d["H"], d["T"]
    bsel = max(1, nbh // H)
    hsel = min(H, nbh)
    sl = (slice(0, bsel), slice(0, hsel))
    x = {n: bf16_to_f64(d[n][sl]) for n in ("q", "k", "v", "do")}
    prm = {n: d[n][:hsel] for n in ("alpha", "beta", "mu", "s")}
    t0 = time.perf_counter()
    oracle.fwd(x["q"], x["k"], x["v"], prm["alpha"], prm["beta"], prm["mu"], prm["s"],
               causal=True, ssmax=True, nthreads=nthreads)
    oracle.bwd(x["q"], x["k"], x["v"], x["do"], prm["alpha"], prm["beta"], prm["mu"], prm["s"],
               causal=True, ssmax=True, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, train_flops(bsel, hsel, T)


def cpu_baseline(nbh=96, seed=1002):
    from transformer_attention_ggd_gb300.inputs import make_inputs
    import oracle
    oracle.build()
    d = make_inputs(2, seed=seed)
    cores = os.cpu_count() or 1
    dt, fl = oracle_sample_step(d, nbh, cores)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of {nbh} of the 96 (b,h) pairs of the B=8 H=12 "
                      f"T=512 training step ({dt:.2f} s), scaled by algorithmic flops"}


def run_reference(args):
    from transformer_attention_ggd_gb300.inputs import make_inputs
    import oracle
    oracle.build()
    d = make_inputs(2, seed=args.seed)
    cores = os.cpu_count() or 1
    nbh = 96
    for _ in range(args.warmup):
        oracle_sample_step(d, nbh, cores)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        dt, fl = oracle_sample_step(d, nbh, cores)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "train_B8_H12_T512", "B": 8, "H": 12, "T": 512, "D": D,
                   "causal": True, "ssmax": True, "step": "fwd+bwd"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: fp64 oracle fwd+bwd of {nbh} of the 96 (b,h) "
                                   "pairs, scaled by algorithmic flops"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


PROFILE_CASES = ("train", "prefill32k", "prefill262k", "decode", "decode_varlen",
                 "decode_paged", "prefill32k_noncausal", "decode_all", "decode_b8")


def profile_case(name, warmup):
    """A few untimed calls of one workload, for capturing its kernels with a
    profiler (no JSON line).  "decode_all" runs the decode, decode_varlen and
    decode_paged cases in that order on one set of inputs (warmup + 1 calls
    each)."""
    import torch
    import __graft_entry__
    from transformer_attention_ggd_gb300 import bam_attn as ba
    from transformer_attention_ggd_gb300.inputs import make_inputs

    __graft_entry__.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    cases = ("decode", "decode_varlen", "decode_paged") if name == "decode_all" else (name,)
    cfg = {"train": 2, "prefill32k": 3, "prefill262k": 4, "decode": 5, "decode_varlen": 5,
           "decode_paged": 5, "prefill32k_noncausal": 3, "decode_b8": 5}[cases[0]]
    causal = name != "prefill32k_noncausal"
    # decode_b8: the decode workload's cache shape for 8 of its 64 sequences
    # (0.8 GB of K and V, still far above L2), for captures of many metrics.
    d = make_inputs(cfg, B=8) if name == "decode_b8" else make_inputs(cfg)

    def bf(b):
        return torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)

    p = {n: torch.from_numpy(d[n]).to(dev) for n in ("alpha", "beta", "mu", "s")}
    prm = ba.make_params(p["alpha"], p["beta"], p["mu"], p["s"], 1e-5, causal, True)
    B, H, T = d["B"], d["H"], d["T"]
    q, k, v = bf(d["q"]), bf(d["k"]), bf(d["v"])
    for name, _ in ((c, i) for c in cases for i in range(warmup + 1)):
        if name in ("decode_varlen", "decode_paged"):
            lens = np.random.default_rng(5005).integers(1, T + 1, B)
            lens[:3] = [1, T, 64]
            lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
            o = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((B, H), dtype=torch.float32, device=dev)
            ws = ba.workspace(ba.BAM_OP_DECODE, B, H, T, dev)
            if name == "decode_varlen":
                ba.bam_attn_decode_varlen(q, k, v, lens_d, o, lse, prm, ws)
            else:
                # the bench's layout: 256-key pages of every block, permuted
                page, mb = 256, T // 256
                perm = torch.randperm(B * mb, generator=torch.Generator().manual_seed(6)).to(dev)
                pools = []
                for c in (k, v):
                    blk = c.view(B, H, mb, page, D).permute(0, 2, 1, 3, 4).reshape(B * mb, H,
                                                                                  page, D)
                    pool = torch.empty_like(blk)
                    pool[perm] = blk
                    pools.append(pool)
                ba.bam_attn_decode_paged(q, pools[0], pools[1], perm.view(B, mb).to(torch.int32),
                                         lens_d, o, lse, prm, ws)
        elif name in ("decode", "decode_b8"):
            o = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((B, H), dtype=torch.float32, device=dev)
            ws = ba.workspace(ba.BAM_OP_DECODE, B, H, T, dev)
            ba.bam_attn_decode(q, k, v, o, lse, prm, ws)
        elif name == "train":
            o = torch.empty((B, H, T, D), dtype=torch.float32, device=dev)
            lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
            wf = ba.workspace(ba.BAM_OP_FWD, B, H, T, dev)
            wb = ba.workspace(ba.BAM_OP_BWD, B, H, T, dev)
            do = bf(d["do"])
            dq, dk, dv = (torch.empty_like(q) for _ in range(3))
            g = [torch.empty(H, dtype=torch.float32, device=dev) for _ in range(4)]
            ba.bam_attn_fwd(q, k, v, o, lse, prm, wf)
            ba.bam_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, *g, prm, wb)
        else:
            o = torch.empty((B, H, T, D), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
            ws = ba.workspace(ba.BAM_OP_FWD, B, H, T, dev)
            ba.bam_attn_fwd(q, k, v, o, lse, prm, ws)
    torch.cuda.synchronize()
    print(f"profile case {'+'.join(cases)}: {warmup + 1} calls each, "
          f"{ba.bam_attn_launch_count()} launches")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip prefill/decode extras")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--seed", type=int, default=1002,
                    help="seed of the training-step inputs (rank r draws with seed + r)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="only run a few untimed calls of one workload (for profilers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_case:
        profile_case(args.profile_case, args.warmup)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    line, _ = run_ours(args, rank, world, dev, torch, dist)
    if rank == 0:
        peaks = load_peaks()
        if not args.no_extra:
            _nvtx(torch, "prefill and decode extras")
            line["extra"] = extra_workloads(torch, dev, args.steps, peaks, cpu=not args.no_cpu)
            _nvtx(torch, None)
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(seed=args.seed)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
