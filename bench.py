#!/usr/bin/env python
"""RG-LRU layer benchmark: fused forward + backward tokens/s at B4 T2048 W2048, bf16 I/O with
a float32 carry, restricted protocol (zero initial state, no resets), 16 gate blocks of 128.

One step = rglru_fused_forward + rglru_fused_backward over one batch of seeded synthetic
input already resident in HBM: the gate projections, gates, decay, multiplier, write and
scan, then the reverse scan, pointwise gradients, the on-device Lambda reduction and the
projection gradients (dx, dWa, dWx, dba, dbx).  The two calls are captured once in a CUDA
graph and the graph is replayed once a step, as a training loop on one GPU runs them.  L2 is
flushed (a 256 MiB write) before every timed step; two CUDA events bracket each step on the
launching stream, with nothing else recorded between them.  A second pass times the same
step with the calls issued directly (`eager`), a third records the forward / backward split
and the backward kernel's own duration (for the roofline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own batch on its own GPU (weak scaling, no
collective on the data path); rank 0 prints one JSON line with the max-over-ranks time.
`--impl reference` times the float64 CPU oracle (the reference arm of this build) on the
host cores instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RG-LRU fwd+bwd tokens/s (B4 T2048 W2048 bf16); % of HBM roofline"
UNIT = "tokens/s"


# ------------------------------------------------------------------ process group helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(value: float, world: int, device="cpu") -> float:
    """Max of a float over ranks (measurement only; nothing on the data path)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks during timing
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ workload
def workload():
    from linear_recurrent_rnn_gb300.inputs import WORKLOADS
    return WORKLOADS[2]


def algorithmic_bytes(wl, grad=None):
    """Compulsory HBM bytes of one fused forward and one fused backward: every input read
    once, every output written once.  s = bytes of an activation element (the I/O dtype),
    g = bytes of a dx element (the gradient dtype; the I/O dtype unless given).
    fwd: x read and y written (2sN), Wa/Wx, biases, Lambda read, hT written; canonical inputs
         also read h0 and the reset markers (uint8 mask or int32 segment positions).
    bwd: x, dy read (2sN), dx written (gN), Wa/Wx, biases, Lambda read, dWa/dWx (float32),
         dba, dbx, dLambda written; canonical inputs also read dhT and the markers and write
         dh0.  Saved chunk states and look-back slots are overhead, not counted."""
    N = wl.B * wl.T * wl.W
    s = 2 if wl.io == "bf16" else 4
    g = s if grad is None else (2 if grad == "bf16" else 4)
    wbytes = 2 * wl.nblk * wl.k * wl.k * s
    vec = wl.W * 4
    state = wl.B * wl.W * 4
    marks = 0
    if wl.mode == "canonical":
        marks = wl.B * wl.T * (4 if wl.seg_len is not None else 1) if (
            wl.seg_len is not None or wl.reset_p > 0 or wl.reset_t0) else 0
    h0 = state if (wl.mode == "canonical" and wl.h0_std > 0) else 0
    fwd = 2 * s * N + wbytes + 3 * vec + state + h0 + marks
    bwd = (2 * s + g) * N + wbytes + 3 * vec + 2 * wl.nblk * wl.k * wl.k * 4 + 3 * vec + marks
    if wl.mode == "canonical":
        bwd += 2 * state   # dhT read, dh0 written
    return fwd, bwd


def tensor_flops(wl):
    """Tensor-core FLOPs of one fused backward.  Algorithmic (the method's contractions): the
    logits recompute (2 x 2Nk), dx += dl W^T (2 x 2Nk) and dW = x^T dl (2 x 2Nk), 12 N k.
    Executed: the dx and dW products also take the bf16 low halves of dl, 20 N k."""
    N = wl.B * wl.T * wl.W
    return 12 * N * wl.k, 20 * N * wl.k


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


# DRAM traffic of one k_fused_bwd launch at B4 T2048 W2048 (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture; writes still resident in L2 when the kernel
# ends are not counted).  It holds for the kernel sources whose hash is recorded beside it;
# when they have changed since, the line reports null until the counters are taken again.
TRAFFIC = {"bytes": 70497792 + 12541952, "sources_sha16": "99e6a620ffd40735"}
KERNEL_SOURCES = ("fused_bwd.cu", "tc.cuh", "common.cuh", "lookback.cuh", "internal.h")


def kernel_sources_sha16():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "linear_recurrent_rnn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_field():
    sha = kernel_sources_sha16()
    ok = TRAFFIC["bytes"] is not None and TRAFFIC["sources_sha16"] == sha
    return (TRAFFIC["bytes"] if ok else None,
            {"source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch",
             "kernel_sources_sha16": sha, "captured_on_sha16": TRAFFIC["sources_sha16"],
             "note": "null when the kernel changed after the capture; L2-resident writes at "
                     "the kernel's end are not counted"})


def run_ours(args, rank, world, local):
    import torch
    from linear_recurrent_rnn_gb300 import build as B_
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import generate

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    B_.build()
    R.lib()
    wl = workload()
    inp = generate(wl, 2 + rank)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sh = R.make_shape(wl.B, wl.T, wl.W, wl.nblk, R.BF16, R.BF16, R.RESTRICTED)
    x, Wa, Wx, ba, bx, L, dy = (dev[k] for k in ("x", "Wa", "Wx", "ba", "bx", "Lambda", "dy"))
    y = torch.empty_like(x)
    hT = torch.empty(wl.B, wl.W, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    dx = torch.empty_like(x)
    dWa = torch.empty(wl.nblk, wl.k, wl.k, device="cuda")
    dWx = torch.empty_like(dWa)
    dba, dbx, dL = (torch.empty(wl.W, device="cuda") for _ in range(3))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def fwd():
        R.rglru_fused_forward(sh, x, Wa, ba, Wx, bx, L, None, None, None, y, hT, saved, stream)

    def bwd():
        R.rglru_fused_backward(sh, dy, None, x, Wa, ba, Wx, bx, L, None, None, None, saved, dx,
                               dWa, dba, dWx, dbx, dL, None, ws, stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout during warm-up")

    # The step as a training loop on this GPU runs it: the forward and backward calls captured
    # once in a CUDA graph (the library's calls enqueue only stream-ordered work: the slot
    # clears and the two kernels), replayed once a step.  Each step is timed between two
    # events on the launching stream (nothing else recorded inside), the L2 flushed before
    # each.  Our kernels per step: counted while capturing.
    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    nc0 = R.rglru_kernel_launches()
    with torch.cuda.graph(g, stream=gs):
        R.rglru_fused_forward(sh, x, Wa, ba, Wx, bx, L, None, None, None, y, hT, saved, gs)
        R.rglru_fused_backward(sh, dy, None, x, Wa, ba, Wx, bx, L, None, None, None, saved,
                               dx, dWa, dba, dWx, dbx, dL, None, ws, gs)
    per_step_launches = R.rglru_kernel_launches() - nc0
    stream.wait_stream(gs)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    dist_barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        g.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    launches = per_step_launches * args.steps
    clk = clocks.stop()
    dist_barrier(world)
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout during the timed region")
    step_list = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = dist_max(sum(step_list), world, device="cuda")
    tokens = wl.B * wl.T
    value = tokens * world * args.steps / (total_ms / 1e3)
    del g

    # The same step with the two calls issued directly each time (no graph).
    dev_ = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        dev_[k][0].record(stream)
        fwd()
        bwd()
        dev_[k][1].record(stream)
    torch.cuda.synchronize()
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout in the direct calls")
    d_ms = dist_max(sum(e[0].elapsed_time(e[1]) for e in dev_), world, device="cuda")
    eager = {"ms_per_step": d_ms / args.steps,
             "value": tokens * world * args.steps / (d_ms / 1e3), "unit": UNIT,
             "how": "the forward and backward calls issued directly every step (no graph); "
                    "L2 flushed before every step"}

    # A second pass for the split: the forward call, and the backward's tensor-core kernel
    # alone between events the library records around its launch (the call also runs the
    # look-back slot clear).
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for e in kev:
        for x_ in e:
            x_.record(stream)  # creates the event
    for k in range(args.steps):
        flush.zero_()
        sev[k][0].record(stream)
        fwd()
        sev[k][1].record(stream)
        R.rglru_debug_kernel_events(kev[k][0], kev[k][1])
        bwd()
        sev[k][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in sev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in sev]

    # end to end through the C ABI with host buffers: H2D of x and dy from pinned memory, the
    # step, D2H of every result (y, dx and the parameter gradients), all inside the events.
    # The copies overlap the calls as a training loop would overlap them: dy comes in on a
    # second stream while the forward runs, y goes out on a third while the backward runs.
    hx = inp["x"].pin_memory()
    hdy = inp["dy"].pin_memory()
    results = (y, dx, dWa, dWx, dba, dbx, dL)
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in results]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.warmup + args.steps):
        if k >= args.warmup:
            flush.zero_()
            e2e_ev[k - args.warmup][0].record(stream)
        x.copy_(hx, non_blocking=True)
        s_in.wait_stream(stream)  # dy after x, beside the forward
        with torch.cuda.stream(s_in):
            dy.copy_(hdy, non_blocking=True)
        fwd()
        s_out.wait_stream(stream)  # y out beside the backward
        with torch.cuda.stream(s_out):
            hout[0].copy_(y, non_blocking=True)
        stream.wait_stream(s_in)
        bwd()
        for h, d in zip(hout[1:], results[1:]):
            h.copy_(d, non_blocking=True)
        stream.wait_stream(s_out)
        if k >= args.warmup:
            e2e_ev[k - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist_max(sum(e[0].elapsed_time(e[1]) for e in e2e_ev), world, device="cuda")
    h2d = hx.numel() * hx.element_size() + hdy.numel() * hdy.element_size()
    d2h = sum(h.numel() * h.element_size() for h in hout)

    fwd_b, bwd_b = algorithmic_bytes(wl)
    traffic_bytes, traffic_src = traffic_field()
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    kern_ms = [e[0].elapsed_time(e[1]) for e in kev]
    kern_mean = statistics.fmean(kern_ms)
    achieved = bwd_b / (kern_mean / 1e3) / 1e9
    flop_alg, flop_exec = tensor_flops(wl)
    tpeak = peaks.get("bf16_tflops")
    t_hbm_us = bwd_b / (peak * 1e9) * 1e6 if peak else None
    t_tc_us = flop_alg / (tpeak * 1e12) * 1e6 if tpeak else None
    combined_us = max(t_hbm_us, t_tc_us) if (t_hbm_us and t_tc_us) else None
    step_ms = total_ms / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + " fused fwd+bwd", "B": wl.B, "T": wl.T, "W": wl.W,
                   "k": wl.k, "nblk": wl.nblk, "mode": wl.mode, "grad": "bf16",
                   "carry": "f32", "seed": "2 + rank",
                   "l2": "flushed by a 256 MiB write before every timed step",
                   "launch": "the fwd + bwd calls captured once in a CUDA graph, replayed once "
                             "a step (key eager: the calls issued directly)",
                   "parallelism": f"dp{world} (independent batches, no collective)"},
        "fwd_ms": {"median": statistics.median(fwd_ms), "min": min(fwd_ms), "max": max(fwd_ms),
                   "mean": statistics.fmean(fwd_ms)},
        "bwd_ms": {"median": statistics.median(bwd_ms), "min": min(bwd_ms), "max": max(bwd_ms),
                   "mean": statistics.fmean(bwd_ms)},
        "fwd_bwd_ms": {"median": statistics.median(step_list), "min": min(step_list),
                       "max": max(step_list), "mean": statistics.fmean(step_list)},
        "hbm_fraction_of_8TBps": (fwd_b + bwd_b) / (step_ms / 1e3) / 8e12,
        "roofline": {"bound": "hbm", "unit": "GB/s", "kernel": "k_fused_bwd",
                     "achieved": achieved, "peak": peak,
                     "frac": (achieved / peak) if peak else None,
                     "peak_source": "measured (hbm_gbs)",
                     "algorithmic_bytes": bwd_b, "traffic": traffic_bytes,
                     "traffic_source": traffic_src,
                     "kernel_ms_mean": kern_mean,
                     # context bound: the same kernel against the tensor pipe, and the larger
                     # of the two bounds (bytes / measured copy bandwidth, flops / measured
                     # bf16 burst) against its duration
                     "tensor": {"algorithmic_flop": flop_alg, "executed_flop": flop_exec,
                                "achieved_tflops": flop_alg / (kern_mean / 1e3) / 1e12,
                                "peak_tflops": tpeak,
                                "frac": (flop_alg / (kern_mean / 1e3) / 1e12 / tpeak)
                                if tpeak else None,
                                "peak_source": "measured (bf16_tflops, burst)"},
                     "combined_bound_us": combined_us,
                     "frac_of_combined": (combined_us / (kern_mean * 1e3))
                     if combined_us else None},
        "e2e": {"value": tokens * world * args.steps / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "x, dy from pinned host memory and every result back to it inside each "
                       "step's events; dy's copy beside the forward and y's beside the "
                       "backward on two side streams"},
        "gpu_launches": launches,
        "clocks": clk,
        "eager": eager,
        "memory": memory_footprint(sh, wl),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, T=args.cpu_sample_T)
    if rank == 0 and world == 1 and not args.no_decode:
        line["decode"] = decode_step(flush, peak)
    if rank == 0 and world == 1 and not args.no_varlen:
        line["varlen"] = varlen_measure(flush, peak)
    if rank == 0 and world == 1 and not args.no_unfused:
        line["unfused"] = unfused_measure(flush, peak)
        line["protocol"] = protocol_measure(flush)
    if rank == 0 and world == 1 and not args.no_configs:
        line["configs"] = configs_measure(flush, peak)
    if rank == 0 and world == 1 and not args.no_delta:
        line["delta_rule"] = delta_rule_measure(flush, peak)
    if rank == 0:
        print(json.dumps(line), flush=True)


def memory_footprint(sh, wl):
    """What the layer keeps between its forward and backward, against the float32 states of
    every token that a backward without recomputation would keep; and the scratch the backward
    takes.  The library allocates nothing itself: these buffers are the caller's."""
    from linear_recurrent_rnn_gb300 import librglru as R
    saved = R.saved_bytes(sh)
    all_states = wl.B * wl.T * wl.W * 4
    return {"saved_bytes": saved, "saved_bytes_per_token": saved / (wl.B * wl.T),
            "all_states_bytes": all_states, "saved_fraction_of_all_states": saved / all_states,
            "workspace_bytes": R.workspace_bytes(sh), "library_allocations": 0}


def decode_step(flush, peak, W=2048, k=128, reps=20):
    """The decode step (rglru_step) on the same layer width and gate blocks, bf16, canonical,
    states carried in place: microseconds per step at batch 1 and 256 (L2 flushed before each
    timed step), tokens/s at 256, and its bytes (weights once, x, h in and out, y) against the
    measured copy bandwidth."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import Workload, generate
    out = {"workload": f"decode step, W{W} k{k} bf16 canonical, states carried in place"}
    for B in (1, 256):
        inp = generate(Workload("decode", B, 1, W, k, "bf16", "canonical", h0_std=1.0), 1)
        d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
        sh = R.make_shape(B, 1, W, W // k, R.BF16, R.BF16, R.CANONICAL)
        x = d["x"].reshape(B, W).contiguous()
        h = d["h0"].clone()
        y = torch.empty_like(x)
        step = lambda: R.rglru_step(sh, x, d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"],
                                    None, h, y, h)
        for _ in range(5):
            step()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        us = statistics.median(ts) * 1e3
        nbytes = 2 * (W // k) * k * k * 2 + B * W * (2 + 4 + 4 + 2)
        out[f"us_per_step_B{B}"] = us
        if B == 256:
            out["tokens_per_s_B256"] = B / (us / 1e6)
            gbs = nbytes / (us / 1e6) / 1e9
            out["roofline_B256"] = {"bound": "hbm", "unit": "GB/s", "achieved": gbs, "peak": peak,
                                    "frac": (gbs / peak) if peak else None,
                                    "algorithmic_bytes": nbytes}
    out["stack_B256"] = decode_stack(flush, peak, W, k)
    out["stack_B1"] = decode_stack(flush, peak, W, k, B=1, L=160)
    return out


def decode_stack(flush, peak, W=2048, k=128, B=256, L=48, reps=10):
    """One decode token through a stack of L layers at batch B: each layer has its own weights,
    constants and carried states, and layer l's y is layer l + 1's x.  The L steps are captured
    once in a CUDA graph and replayed, the L2 flushed before each replay, so the steps follow
    one another on the GPU as in a graph-captured serving loop.  Weights and states of all
    layers exceed the L2 (48 x 4 MB at batch 256, 160 x 1 MB at batch 1), so each step reads
    its operands from HBM.  Reports microseconds per layer step and its bytes against the
    measured copy bandwidth."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import Workload, generate
    sh = R.make_shape(B, 1, W, W // k, R.BF16, R.BF16, R.CANONICAL)
    layers, xs = [], []
    for l in range(L):
        inp = generate(Workload("decode", B, 1, W, k, "bf16", "canonical", h0_std=1.0), 100 + l)
        d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
        layers.append((d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], d["h0"].clone()))
        if l == 0:
            xs.append(d["x"].reshape(B, W).contiguous())
        xs.append(torch.empty(B, W, dtype=xs[0].dtype, device="cuda"))

    def run(s):
        for l, (Wa, ba, Wx, bx, Lam, h) in enumerate(layers):
            R.rglru_step(sh, xs[l], Wa, ba, Wx, bx, Lam, None, h, xs[l + 1], h, s)

    stream = torch.cuda.current_stream()
    run(stream)
    torch.cuda.synchronize()
    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    nc0 = R.rglru_kernel_launches()
    with torch.cuda.graph(g, stream=gs):
        run(gs)
    launches = R.rglru_kernel_launches() - nc0
    stream.wait_stream(gs)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    del g
    us = statistics.median(ts) * 1e3 / L
    nbytes = 2 * (W // k) * k * k * 2 + B * W * (2 + 4 + 4 + 2)
    gbs = nbytes / (us / 1e6) / 1e9
    return {"layers": L, "launches_per_token": launches, "us_per_layer_step": us,
            "tokens_per_s_per_layer": B / (us / 1e6),
            "roofline": {"bound": "hbm", "unit": "GB/s", "achieved": gbs, "peak": peak,
                         "frac": (gbs / peak) if peak else None, "algorithmic_bytes": nbytes},
            "how": "L layer steps captured once in a CUDA graph, replayed; L2 flushed before "
                   "each replay; weights and states of all layers exceed the L2"}


def varlen_measure(flush, peak, reps=10, W=2048, k=128, T=8192, seed=5):
    """Packed variable-length sequences (rglru_fused_forward_varlen / _backward_varlen): the
    headline's 8192 tokens in one row, sequence lengths drawn U[1, 2048] until the row is full
    (the last one truncated), each sequence with its own float32 initial state N(0, 0.5^2) and
    final-state gradient; bf16, canonical.  Milliseconds per call (L2 flushed before each),
    tokens/s of the pair, and the backward kernel's algorithmic bytes (the headline's, plus
    h0, dhT read and dh0 written per sequence) against the measured copy bandwidth."""
    import numpy as np
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import Workload, generate, packed_lengths
    lengths = packed_lengths(seed, T, 1, 2048)
    S = len(lengths)
    rng = np.random.default_rng(seed + 1)
    wl = Workload("varlen", 1, T, W, k, "bf16", "canonical", (0.9, 0.999))
    inp = generate(wl, seed)
    d = {n: v.cuda() for n, v in inp.items() if isinstance(v, torch.Tensor)}
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32).cuda()
    h0 = (torch.from_numpy(rng.standard_normal((S, W))).float() * 0.5).cuda()
    dhT = torch.from_numpy(rng.standard_normal((S, W))).float().cuda()
    sh = R.make_shape(1, T, W, W // k, R.BF16, R.BF16, R.CANONICAL)
    y = torch.empty_like(d["x"])
    hT = torch.empty(S, W, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    dx = torch.empty_like(d["x"])
    dWa = torch.empty(W // k, k, k, device="cuda")
    dWx = torch.empty_like(dWa)
    dba, dbx, dL = (torch.empty(W, device="cuda") for _ in range(3))
    dh0 = torch.empty(S, W, device="cuda")
    ba, bx = d["ba"], d["bx"]
    fwd = lambda: R.rglru_fused_forward_varlen(sh, d["x"], d["Wa"], ba, d["Wx"], bx, d["Lambda"],
                                               cu, S, h0, y, hT, saved)
    bwd = lambda: R.rglru_fused_backward_varlen(sh, d["dy"], dhT, d["x"], d["Wa"], ba, d["Wx"],
                                                bx, d["Lambda"], cu, S, h0, saved, dx, dWa, dba,
                                                dWx, dbx, dL, dh0, ws)
    for _ in range(3):
        fwd()
        bwd()
    tf, tb, tk = [], [], []
    for _ in range(reps):
        for fn, acc in ((fwd, tf), (bwd, tb)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if fn is bwd:
                ka.record()  # creates the events
                kb.record()
                R.rglru_debug_kernel_events(ka, kb)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            acc.append(a.elapsed_time(b))
            if fn is bwd:
                tk.append(ka.elapsed_time(kb))
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout in the packed-sequence measurement")
    fms, bms, kms = statistics.median(tf), statistics.median(tb), statistics.median(tk)
    _, bwd_b = algorithmic_bytes(wl.scaled(mode="restricted"))
    bwd_b += 3 * S * W * 4   # per-sequence h0, dhT read, dh0 written
    gbs = bwd_b / (kms / 1e3) / 1e9
    return {"workload": f"packed B1 T{T} W{W} k{k} bf16 canonical, {S} sequences of U[1, 2048] "
                        "tokens, per-sequence h0 and dhT",
            "sequences": S, "fwd_ms": fms, "bwd_ms": bms,
            "tokens_per_s": T / ((fms + bms) / 1e3),
            "roofline_bwd": {"bound": "hbm", "unit": "GB/s", "kernel": "k_fused_bwd (varlen)",
                             "achieved": gbs, "peak": peak,
                             "frac": (gbs / peak) if peak else None,
                             "algorithmic_bytes": bwd_b, "kernel_ms": kms}}


def stats(v):
    return {"median": statistics.median(v), "min": min(v), "max": max(v),
            "mean": statistics.fmean(v)}


def configs_measure(flush, peak, reps=10, cfgs=(1, 3, 4, 5)):
    """The other synthetic workloads of the layer's specification through the fused calls
    (rglru_fused_forward + rglru_fused_backward), each with its own seeded inputs: forward and
    forward + backward milliseconds (L2 flushed before each sample; the two calls back to back
    inside the pair), tokens/s of the pair, and the pair's compulsory bytes against the
    measured copy bandwidth and against 8 TB/s.  Gradients are stored in the I/O dtype, as in
    the headline.  `path` names the kernels the shape takes."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import WORKLOADS, generate
    out = {}
    for cfg in cfgs:
        wl = WORKLOADS[cfg]
        inp = generate(wl, cfg)
        d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
        del inp
        io = R.BF16 if wl.io == "bf16" else R.F32
        mode = R.CANONICAL if wl.mode == "canonical" else R.RESTRICTED
        sh = R.make_shape(wl.B, wl.T, wl.W, wl.nblk, io, io, mode)
        x = d["x"]
        y = torch.empty_like(x)
        hT = torch.empty(wl.B, wl.W, device="cuda")
        saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
        dx = torch.empty_like(x)
        dWa = torch.empty(wl.nblk, wl.k, wl.k, device="cuda")
        dWx = torch.empty_like(dWa)
        dba, dbx, dL = (torch.empty(wl.W, device="cuda") for _ in range(3))
        dh0 = torch.empty(wl.B, wl.W, device="cuda") if wl.mode == "canonical" else None
        args_f = (sh, x, d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], d["reset_mask"],
                  d["segment_pos"], d["h0"], y, hT, saved)
        fwd = lambda: R.rglru_fused_forward(*args_f)
        bwd = lambda: R.rglru_fused_backward(sh, d["dy"], d["dhT"], x, d["Wa"], d["ba"], d["Wx"],
                                             d["bx"], d["Lambda"], d["reset_mask"],
                                             d["segment_pos"], d["h0"], saved, dx, dWa, dba,
                                             dWx, dbx, dL, dh0, ws)
        for _ in range(3):
            fwd()
            bwd()
        torch.cuda.synchronize()
        n0 = R.rglru_kernel_launches()
        fwd()
        n1 = R.rglru_kernel_launches()
        bwd()
        n2 = R.rglru_kernel_launches()
        tf, tp = [], []
        for _ in range(reps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            fwd()
            e[1].record()
            bwd()
            e[2].record()
            torch.cuda.synchronize()
            tf.append(e[0].elapsed_time(e[1]))
            tp.append(e[0].elapsed_time(e[2]))
        if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
            raise RuntimeError(f"look-back timeout in configuration {cfg}")
        fb, bb = algorithmic_bytes(wl)
        pm = statistics.median(tp)
        gbs = (fb + bb) / (pm / 1e3) / 1e9
        out[str(cfg)] = {
            "workload": wl.name, "B": wl.B, "T": wl.T, "W": wl.W, "k": wl.k, "io": wl.io,
            "mode": wl.mode, "path": R.fused_path(sh),
            "kernels": {"fwd": n1 - n0, "bwd": n2 - n1},
            "fwd_ms": stats(tf), "fwd_bwd_ms": stats(tp),
            "tokens_per_s": wl.B * wl.T / (pm / 1e3),
            "algorithmic_bytes": fb + bb, "achieved_gbs": gbs,
            "hbm_frac_measured": (gbs / peak) if peak else None,
            "hbm_frac_of_8TBps": gbs / 8e3}
        del d, x, y, dx, saved, ws
        torch.cuda.empty_cache()
    return out


def protocol_measure(flush, reps=5):
    """The pages' timing protocol at the headline shape: two rounds, the fused and the unfused
    variant in A-B order in the first and B-A in the second, `reps` samples of each per round
    (10 per variant), every sample the forward and then the backward with events around each
    and the L2 flushed before it; median / min / max / mean of forward and forward + backward.
    Unfused = rglru_gate_proj + rglru_forward, then rglru_backward + rglru_gate_proj_backward."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import WORKLOADS, generate
    wl = WORKLOADS[2]
    inp = generate(wl, 2)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sh = R.make_shape(wl.B, wl.T, wl.W, wl.nblk, R.BF16, R.BF16, R.RESTRICTED)
    x = d["x"]
    lr, li, y, dx, dlr, dli = (torch.empty_like(x) for _ in range(6))
    hT = torch.empty(wl.B, wl.W, device="cuda")
    dL, dba, dbx = (torch.empty(wl.W, device="cuda") for _ in range(3))
    dWa = torch.empty(wl.nblk, wl.k, wl.k, device="cuda")
    dWx = torch.empty_like(dWa)
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    Wa, Wx, ba, bx, L, dy = d["Wa"], d["Wx"], d["ba"], d["bx"], d["Lambda"], d["dy"]

    def fused_f():
        R.rglru_fused_forward(sh, x, Wa, ba, Wx, bx, L, None, None, None, y, hT, saved)

    def fused_b():
        R.rglru_fused_backward(sh, dy, None, x, Wa, ba, Wx, bx, L, None, None, None, saved, dx,
                               dWa, dba, dWx, dbx, dL, None, ws)

    def unf_f():
        R.rglru_gate_proj(sh, x, Wa, ba, Wx, bx, lr, li)
        R.rglru_forward(sh, x, lr, li, L, None, None, None, y, hT, saved)

    def unf_b():
        R.rglru_backward(sh, dy, None, x, lr, li, L, None, None, None, saved, dx, dlr, dli, dL,
                         None, ws)
        R.rglru_gate_proj_backward(sh, dlr, dli, x, Wa, Wx, dx, dWa, dba, dWx, dbx, ws)

    variants = {"fused": (fused_f, fused_b), "unfused": (unf_f, unf_b)}
    for f, b in variants.values():
        for _ in range(3):
            f()
            b()
    torch.cuda.synchronize()
    res = {n: {"fwd": [], "fwd_bwd": []} for n in variants}
    for order in (("fused", "unfused"), ("unfused", "fused")):
        for n in order:
            f, b = variants[n]
            for _ in range(reps):
                flush.zero_()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record()
                f()
                e[1].record()
                b()
                e[2].record()
                torch.cuda.synchronize()
                res[n]["fwd"].append(e[0].elapsed_time(e[1]))
                res[n]["fwd_bwd"].append(e[0].elapsed_time(e[2]))
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout in the protocol measurement")
    out = {"workload": wl.name, "rounds": "2 x 5 samples per variant, AB then BA",
           "unit": "ms"}
    for n, r in res.items():
        out[n] = {"fwd_ms": stats(r["fwd"]), "fwd_bwd_ms": stats(r["fwd_bwd"])}
    return out


def unfused_measure(flush, peak, reps=10):
    """The unfused API at the headline shape (B4 T2048 W2048, 16 blocks of 128, bf16, restricted):
    rglru_gate_proj (logits to HBM), rglru_forward and rglru_backward (the scan kernels over
    stored logits), rglru_gate_proj_backward.  Milliseconds per call (L2 flushed before each),
    tokens/s of the four, and the two scan calls against the measured copy bandwidth with
    their compulsory bytes: forward x, lr, li read and y written (8 bytes per element, plus
    Lambda and hT); backward x, lr, li, dy read and dx, dlr, dli written (14 bytes per element,
    plus Lambda and dLambda).  Each scan call also clears its look-back slots; the backward
    call also reduces the Lambda partials (a second, small kernel)."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.inputs import WORKLOADS, generate
    wl = WORKLOADS[2]
    inp = generate(wl, 2)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sh = R.make_shape(wl.B, wl.T, wl.W, wl.nblk, R.BF16, R.BF16, R.RESTRICTED)
    x = d["x"]
    lr, li, y, dx, dlr, dli = (torch.empty_like(x) for _ in range(6))
    hT = torch.empty(wl.B, wl.W, device="cuda")
    dL, dba, dbx = (torch.empty(wl.W, device="cuda") for _ in range(3))
    dWa = torch.empty(wl.nblk, wl.k, wl.k, device="cuda")
    dWx = torch.empty_like(dWa)
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    calls = {
        "gate_proj": lambda: R.rglru_gate_proj(sh, x, d["Wa"], d["ba"], d["Wx"], d["bx"], lr, li),
        "forward": lambda: R.rglru_forward(sh, x, lr, li, d["Lambda"], None, None, None, y, hT,
                                           saved),
        "backward": lambda: R.rglru_backward(sh, d["dy"], None, x, lr, li, d["Lambda"], None,
                                             None, None, saved, dx, dlr, dli, dL, None, ws),
        "gate_proj_backward": lambda: R.rglru_gate_proj_backward(sh, dlr, dli, x, d["Wa"],
                                                                 d["Wx"], dx, dWa, dba, dWx,
                                                                 dbx, ws),
    }
    for _ in range(3):
        for fn in calls.values():
            fn()
    torch.cuda.synchronize()
    times = {n: [] for n in calls}
    for _ in range(reps):
        for n, fn in calls.items():
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            times[n].append(a.elapsed_time(b))
    if R.rglru_sync_status(saved) != R.OK or R.rglru_sync_status(ws) != R.OK:
        raise RuntimeError("look-back timeout in the unfused measurement")
    ms = {n: statistics.median(t) for n, t in times.items()}
    N = wl.B * wl.T * wl.W
    out = {"workload": f"{wl.name} unfused API (logits through HBM)",
           "ms": ms, "tokens_per_s": wl.B * wl.T / (sum(ms.values()) / 1e3)}
    for n, nbytes in (("forward", 8 * N + 4 * wl.W + 4 * wl.B * wl.W),
                      ("backward", 14 * N + 8 * wl.W)):
        gbs = nbytes / (ms[n] / 1e3) / 1e9
        out[f"roofline_{n}"] = {"bound": "hbm", "unit": "GB/s", "achieved": gbs, "peak": peak,
                                "frac": (gbs / peak) if peak else None,
                                "algorithmic_bytes": nbytes, "timed": "the whole call"}
    return out


# FP32 CUDA-core peak of the GB300 for the delta-rule kernels (no tensor cores): 152 SMs x 128
# FP32 lanes x 2 FLOP per FMA x 2070 MHz (the maximum SM clock).
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2070e6 / 1e12


def delta_rule_measure(flush, peak, reps=10):
    """The gated delta rule (delta_rule_forward / _backward, GDN) at B4 T2048 with 16 heads of
    128 x 128, bf16: milliseconds per call (L2 flushed before each), tokens/s of the pair, and
    each kernel against the FP32 CUDA-core peak.  Algorithmic FLOPs per state element and
    token: forward 7 (decay, S'^T k, the rank-1 write, S^T q); backward 22 (the forward again,
    since the per-token states are not stored, and 15 for the reverse recurrence)."""
    import torch
    from linear_recurrent_rnn_gb300 import librglru as R
    from linear_recurrent_rnn_gb300.delta_inputs import DELTA_WORKLOADS, generate
    wl = DELTA_WORKLOADS["headline"]
    inp = generate(wl, 7)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    sh = R.make_delta_shape(wl.B, wl.T, wl.Hk, wl.Hv, wl.Dk, wl.Dv, R.BF16)
    scale = wl.Dk ** -0.5
    N = wl.B
    o = torch.empty_like(d["v"])
    hT = torch.empty(N, wl.Hv, wl.Dk, wl.Dv, device="cuda")
    saved = torch.empty(R.delta_rule_saved_bytes(sh, N), dtype=torch.uint8, device="cuda")
    grads = {n: torch.empty(d[m].shape, device="cuda") for n, m in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    dh0 = torch.empty_like(hT)
    ws = torch.empty(max(1, R.delta_rule_workspace_bytes(sh)), dtype=torch.uint8, device="cuda")
    fwd = lambda: R.delta_rule_forward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale, None,
                                       N, None, o, hT, saved)
    bwd = lambda: R.delta_rule_backward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale,
                                        None, N, None, saved, d["do"], None, grads["dq"],
                                        grads["dk"], grads["dv"], grads["dg"], grads["dbeta"],
                                        dh0, ws)
    for _ in range(3):
        fwd()
        bwd()
    tf, tb = [], []
    for _ in range(reps):
        for fn, acc in ((fwd, tf), (bwd, tb)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            acc.append(a.elapsed_time(b))
    fms, bms = statistics.median(tf), statistics.median(tb)
    # the E4M3 state quantize-dequantize (64-column tiles), in place on the saved block states
    # seen as float32 [n, 128, 128] states: read and written once, against HBM
    st = saved.view(torch.float32).view(-1, wl.Dk, wl.Dv)
    tq = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        R.delta_rule_state_fp8_qdq(st, st, 64)
        b.record()
        torch.cuda.synchronize()
        tq.append(a.elapsed_time(b))
    qms = statistics.median(tq)
    qbytes = 2 * st.numel() * 4
    # decode: one token per sequence from states carried in place (T = 1), batch 1 and 64
    dec = {}
    for Bd in (1, 64):
        dsh = R.make_delta_shape(Bd, 1, wl.Hk, wl.Hv, wl.Dk, wl.Dv, R.BF16)
        tok = {n: d[n][:1, :1].expand(Bd, 1, *d[n].shape[2:]).contiguous()
               for n in ("q", "k", "v", "g", "beta")}
        hs = torch.zeros(Bd, wl.Hv, wl.Dk, wl.Dv, device="cuda")
        od = torch.empty_like(tok["v"])
        step = lambda: R.delta_rule_forward(dsh, tok["q"], tok["k"], tok["v"], tok["g"],
                                            tok["beta"], scale, None, Bd, hs, od, hs, None)
        for _ in range(3):
            step()
        td = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            torch.cuda.synchronize()
            td.append(a.elapsed_time(b))
        dec[f"us_per_step_B{Bd}"] = statistics.median(td) * 1e3
    elems = wl.B * wl.T * wl.Hv * wl.Dk * wl.Dv
    out = {"workload": f"{wl.name} GDN bf16 (q, k unit length, exp(g) U[0.8, 1), beta U(0, 1))",
           "fwd_ms": fms, "bwd_ms": bms, "tokens_per_s": wl.B * wl.T / ((fms + bms) / 1e3),
           "saved_bytes": saved.numel(), "decode": dec,
           "state_fp8_qdq": {"states": st.shape[0], "ms": qms, "bound": "hbm", "unit": "GB/s",
                             "achieved": qbytes / (qms / 1e3) / 1e9, "peak": peak,
                             "frac": (qbytes / (qms / 1e3) / 1e9 / peak) if peak else None,
                             "algorithmic_bytes": qbytes}}
    for name, flop, ms in (("fwd", 7 * elems, fms), ("bwd", 22 * elems, bms)):
        tf_s = flop / (ms / 1e3) / 1e12
        out[f"roofline_{name}"] = {"bound": "alu", "unit": "TFLOP/s", "achieved": tf_s,
                                   "peak": ALU_FP32_TFLOPS, "frac": tf_s / ALU_FP32_TFLOPS,
                                   "algorithmic_flop": flop,
                                   "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2070 MHz"}
    return out


def oracle_step(wl_sample, inp):
    import oracle
    from linear_recurrent_rnn_gb300.inputs import as_f64
    o = {k: as_f64(v) if v is not None and not isinstance(v, str) else v for k, v in inp.items()}
    mode = oracle.RESTRICTED if wl_sample.mode == "restricted" else oracle.CANONICAL
    oracle.fused_forward(mode, o["x"], o["Wa"], o["ba"], o["Wx"], o["bx"], o["Lambda"])
    oracle.fused_backward(mode, o["x"], o["Wa"], o["ba"], o["Wx"], o["bx"], o["Lambda"], o["dy"])


def cpu_cores():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline(wl, T=2048, min_seconds=10.0):
    """The float64 oracle as it stands, on the host cores, on a bounded sample of the
    workload: batch row 0, the first T tokens, all W channels (every gate block), repeated
    until at least `min_seconds` of CPU work have been timed."""
    from linear_recurrent_rnn_gb300.inputs import generate
    ws = wl.scaled(B=1, T=T)
    inp = generate(ws, 2)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(ws, inp)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    out = {"value": reps * ws.B * ws.T / dt, "unit": UNIT, "cores": cpu_cores(),
           "kind": "oracle",
           "sample": f"B1 T{T} W{wl.W} (all {wl.nblk} blocks) fused fwd+bwd, float64, "
                     f"{reps} repetitions in {dt:.1f} s",
           "cpu_model": cpu_model()}
    out["single_thread"] = cpu_baseline_single_thread(wl)
    return out


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_single_thread(wl, T=512):
    """The same oracle on one thread (a subprocess with OMP_NUM_THREADS=1), on a smaller
    sample (T tokens of batch row 0, all channels), timed once after a warm-up call."""
    code = (
        "import sys, time, json; sys.path.insert(0, %r)\n"
        "import bench\n"
        "from linear_recurrent_rnn_gb300.inputs import generate\n"
        "wl = bench.workload().scaled(B=1, T=%d)\n"
        "inp = generate(wl, 2)\n"
        "bench.oracle_step(wl, inp)\n"
        "t0 = time.perf_counter(); bench.oracle_step(wl, inp); dt = time.perf_counter() - t0\n"
        "print(json.dumps({'value': wl.T / dt, 'seconds': dt}))\n" % (ROOT, T))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=300)
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the multi-core figure is the baseline
        return {"error": str(e)[:200]}
    return {"value": res["value"], "unit": UNIT, "cores": 1,
            "sample": f"B1 T{T} W{wl.W} (all {wl.nblk} blocks) fused fwd+bwd, float64, "
                      f"one call in {res['seconds']:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the oracle on the host cores, each step a bounded sample."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    from linear_recurrent_rnn_gb300.inputs import generate
    wl = workload()
    T = args.ref_sample_T
    ws = wl.scaled(B=1, T=T)
    inp = generate(ws, 2)
    for _ in range(args.warmup):
        oracle_step(ws, inp)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(ws, inp)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = ws.B * ws.T * args.steps / total
    sample = f"B1 T{T} W{wl.W} (all {wl.nblk} blocks) fused fwd+bwd per step, float64"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name + " fused fwd+bwd", "B": wl.B, "T": wl.T,
                       "W": wl.W, "k": wl.k, "mode": wl.mode},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    p.add_argument("--no-delta", action="store_true", help="skip the delta-rule measurement")
    p.add_argument("--no-varlen", action="store_true",
                   help="skip the packed-sequence (varlen) measurement")
    p.add_argument("--no-unfused", action="store_true",
                   help="skip the unfused-API (scan kernels over stored logits) measurement")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other synthetic workloads (configurations 1, 3, 4, 5)")
    p.add_argument("--cpu-sample-T", type=int, default=2048)
    p.add_argument("--ref-sample-T", type=int, default=256)
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
