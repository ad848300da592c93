#!/usr/bin/env python3
"""Benchmark of the SGMV multi-LoRA hot path on GB300.

One step = one pass of the whole path over one batch through the C ABI:
sgmv_apply_rows groups the batch's rows by adapter, gathers x, shrinks,
expands and scatters into y (one kernel for decode batches; grouping kernel +
CUDA-core + tensor-core kernels for prefill).  The default workload,
llama7b-stack, is one decode step of a Llama-2-7B LoRA stack: all 224
projections (32 layers x q, k, v, o, gate, up, down), 128 rows on 128
distinct adapters, ~11.2 GB of algorithmic traffic per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the fp64 oracle on the host cores

Prints one JSON line (rank 0).  `value` is rows/s with inputs resident in HBM:
inputs are rotated over enough copies that one pass touches more than twice
the L2 cache, the K timed steps run as CUDA-graph replays, and the K-step
region is timed `--repeats` times (each bracketed by a barrier and a device
synchronisation); `value` comes from the median region.  `roofline` gives the
update call's time back to back (the figure `frac` uses) and alone after an
L2 flush.  `workloads` times the other named workloads the same way, with
each decode workload's read-only floor.  `e2e` is the same metric through
the public API with each step's inputs copied from pinned host memory and its
result read back, called eagerly (and, for comparison, as graph replays).
With N > 1 (torchrun) every rank runs an independent replica: the path has no
exchange step.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SGMV shrink+expand rows/s and achieved HBM GB/s (% of GB300 roofline)"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ["tiny", "decode-distinct", "decode-shared", "decode-zipf", "prefill", "llama7b-q",
             "llama7b-stack"]
# the other workloads timed beside the headline one (the small case the oracle
# finishes in seconds, the two decode batches and their shared-adapter twin,
# and prefill)
SIDE_WORKLOADS = ["tiny", "decode-distinct", "decode-shared", "decode-zipf", "prefill"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--repeats", type=int, default=5,
                   help="timed regions of --steps steps each; value from the median one")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama7b-stack", choices=WORKLOADS)
    p.add_argument("--stack-calls", default="grouped", choices=["grouped", "single"],
                   help="llama7b-stack: a layer's q/k/v and gate/up as one launch each "
                        "(sgmv_apply_multi; 128 update launches per step), or 224 single calls")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=6.0,
                   help="host-core budget of each oracle baseline sample (one thread, all cores)")
    p.add_argument("--soak-seconds", type=float, default=1.0,
                   help="load before the timed region while clocks are sampled")
    p.add_argument("--latency-iters", type=int, default=30,
                   help="L2-flushed single calls per isolated timing (median)")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the side workloads, e2e and the cpu baseline (profiling runs)")
    p.add_argument("--load", action="store_true",
                   help="on-demand adapter loading instead: one Llama-2-7B adapter (224 "
                        "projections) from pinned host memory, alone and during the stack's SGMV")
    p.add_argument("--fused", action="store_true",
                   help="the fused LoRA layer instead: y = x W + LoRA delta in one pass "
                        "(sgmv_fused_linear_lora) against cuBLAS x W alone and x W + SGMV, "
                        "over batch sizes and the Llama-2-7B projection shapes")
    p.add_argument("--fused-point", default=None, metavar="H1,H2,T",
                   help="with --fused: that one point only (for profiling)")
    p.add_argument("--figure", action="store_true",
                   help="the pages' micro-benchmark instead: latency of the base layer alone, "
                        "with a per-adapter loop and with SGMV, over batch sizes and adapter counts")
    return p.parse_args(argv)


# ---------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# Kernel sources behind each workload's launches: a profile's counters stand
# only for the code that hashes to the value recorded beside them.  Host-side
# argument checks and dispatch (sgmv_api.cu, sgmv_noalloc.cu) hold no kernel.
_COMMON_SOURCES = ("sgmv_device.cuh", "sgmv_internal.h", "sgmv_builder.cu")
KERNEL_SOURCES = {
    "stream": _COMMON_SOURCES + ("sgmv_stream.cuh", "sgmv_stream_f16.cu", "sgmv_stream_bf16.cu"),
    "tc": _COMMON_SOURCES + ("sgmv_tc.cu", "sgmv_tcgen05.cuh", "sgmv_tiles.cuh", "sgmv_cc.cuh",
                             "sgmv_cc_f16.cu", "sgmv_cc_bf16.cu"),
    "fused": _COMMON_SOURCES + ("sgmv_fused.cu", "sgmv_fused.h", "sgmv_tcgen05.cuh",
                                "sgmv_tiles.cuh", "sgmv_cc.cuh", "sgmv_cc_f16.cu",
                                "sgmv_cc_bf16.cu"),
}
# which kernels a workload's update call runs (prefill's segments all go to
# the tensor cores; every decode workload to the streaming kernel)
WORKLOAD_KERNELS = {"prefill": "tc", "fused-linear-lora-q": "fused"}


def source_hash(family="stream"):
    """Hash of one kernel family's sources (see KERNEL_SOURCES)."""
    import hashlib

    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "rank_gemv_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[family]):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(workload):
    """DRAM bytes per update call measured by ncu for this workload (from
    profiles/traffic.md), or None when its kernels changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    want = source_hash(WORKLOAD_KERNELS.get(workload, "stream"))
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 3 and cells[0] == workload and cells[1] == want:
            try:
                return float(cells[2])
            except ValueError:
                return None
    return None


def config_of(name, w, l2_note=None):
    cfg = {"workload": name, "T": w.T, "L": w.L, "H1": w.H1, "H2": w.H2, "r": w.r,
           "inputs": str(w.dtype).replace("torch.", ""),
           "y": str(w.y_dtype).replace("torch.", ""),
           "segments": int(len(set(w.row_adapter.tolist()))), "parallelism": "replicas"}
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


def stack_config(l2_note=None, grouped=True):
    cfg = {"workload": "llama7b-stack", "T": 128, "L": 128, "r": 16, "layers": 32,
           "projections": 7, "inputs": "float16", "y": "float16", "segments": 128,
           "parallelism": "replicas",
           "update_launches": ("per layer: q+k+v, o, gate+up and down, one sgmv_apply_multi "
                               "launch each (128 per step)") if grouped
           else "one sgmv_apply per projection (224 per step)"}
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(dev):
    import torch

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(dev.index or 0)


def rotation_copies(touched_bytes, l2_bytes, cap=256):
    """Input copies to rotate over so that one pass touches more than twice the
    L2 cache (at most `cap`; tiny batches then stay in L2, which the caller
    states)."""
    return int(min(cap, max(2, -(-2 * l2_bytes // max(1, touched_bytes)))))


# ------------------------------------------------------- our implementation
class Batch:
    """Device copy of one batch plus its metadata buffers."""

    def __init__(self, w, dev, sgmv):
        import torch

        self.w = w
        self.X = w.X.to(dev)
        self.A = w.A.to(dev)
        self.B = w.B.to(dev)
        self.Y = w.Y0.to(dev).clone()
        self.ra = w.row_adapter.to(dev)
        self.smax = sgmv.sgmv_max_segments(w.T, w.L)
        # lets long segments use the tensor-core path (unused by decode batches)
        self.ws = torch.empty(sgmv.sgmv_workspace_bytes(w.T, w.H1, w.H2, w.r), dtype=torch.uint8,
                              device=dev)
        self.meta = (torch.empty(max(w.T, 1), dtype=torch.int32, device=dev),
                     torch.empty(self.smax + 1, dtype=torch.int32, device=dev),
                     torch.empty(max(self.smax, 1), dtype=torch.int32, device=dev),
                     torch.empty(1, dtype=torch.int32, device=dev))

    n_apply = 1  # update calls per step

    def apply(self, sgmv):
        """One sgmv_apply_rows (grouping + update); returns the kernels it launched."""
        sgmv.sgmv_apply_rows(self.Y, self.X, self.A, self.B, self.ra, self.w.scale, out=self.meta,
                             workspace=self.ws)
        return sgmv.sgmv_last_launch_count()

    def step(self, sgmv):
        self.apply(sgmv)

    def update(self, sgmv):
        """The update kernels alone (roofline): sgmv_apply on the grouping the
        last step wrote, or the single grouped launch for batches of up to 64
        rows (their grouping happens inside the kernel)."""
        if self.w.T <= 64:
            self.apply(sgmv)
            return
        perm, seg_ptr, idx, _ = self.meta
        sgmv.sgmv_apply(self.Y, self.X, self.A, self.B, seg_ptr, idx, self.w.scale, perm=perm,
                        S=self.smax, workspace=self.ws)


def stack_launch_groups(grouped=True):
    """The update launches of one llama7b-stack step: (layer, projections),
    in order.  Grouped: per layer q+k+v (they read the same rows), o, gate+up
    (the same rows again) and down, each one launch; else one per
    projection."""
    from rank_gemv_gb300 import workloads as wl

    n_proj = len(wl.LLAMA7B_PROJ)
    groups = [[0, 1, 2], [3], [4, 5], [6]] if grouped else [[k] for k in range(n_proj)]
    return [(layer, g) for layer in range(wl.LLAMA7B_LAYERS) for g in groups]


class StackBatch:
    """All 224 projections of the llama7b-stack workload, resident on the device.

    grouped (the default): the batch is grouped once per step
    (sgmv_build_segments_device), then a layer's projections run as a model
    runs them -- q, k and v read the same rows and are one sgmv_apply_multi
    launch, gate and up another, o and down (which read the attention output
    and the activation) one sgmv_apply_multi launch each: 4 update launches
    per layer, 128 per step.  Otherwise 224 sgmv_apply calls, one per
    projection, the first one grouping the batch (sgmv_apply_rows)."""

    def __init__(self, seed, dev, sgmv, grouped=True):
        import torch
        from rank_gemv_gb300 import workloads as wl

        self.T, self.L, self.r = 128, 128, 16
        self.grouped = grouped
        self.projs = []
        for layer in range(wl.LLAMA7B_LAYERS):
            for p in range(len(wl.LLAMA7B_PROJ)):
                X, A, B, Y0 = wl.stack_projection(seed, layer, p, device=dev)
                self.projs.append((X, A, B, Y0))
        self.ra = wl.stack_row_adapter(self.T).to(dev)
        self.smax = sgmv.sgmv_max_segments(self.T, self.L)
        self.meta = (torch.empty(self.T, dtype=torch.int32, device=dev),
                     torch.empty(self.smax + 1, dtype=torch.int32, device=dev),
                     torch.empty(self.smax, dtype=torch.int32, device=dev),
                     torch.empty(1, dtype=torch.int32, device=dev))
        self.launches = stack_launch_groups(grouped)
        self.n_apply = len(self.launches)

    def run_group(self, sgmv, layer, g):
        """The update of projections g of a layer, on the last grouping."""
        perm, seg_ptr, idx, _ = self.meta
        pr = [self.projs[layer * 7 + k] for k in g]
        if not self.grouped:
            X, A, B, Y = pr[0]
            sgmv.sgmv_apply(Y, X, A, B, seg_ptr, idx, 1.0, perm=perm, S=self.smax)
        else:  # every launch through the multi-problem entry (one kernel for the step)
            sgmv.sgmv_apply_multi([Y for _, _, _, Y in pr], [X for X, _, _, _ in pr],
                                  [A for _, A, _, _ in pr], [B for _, _, B, _ in pr],
                                  seg_ptr, idx, 1.0, perm=perm, S=self.smax)
        return sgmv.sgmv_last_launch_count()

    def apply(self, sgmv):
        """One decode step over all 224 projections, as a serving loop runs it:
        the batch is grouped once, and every update launch after it reuses
        the grouping (grouped: sgmv_build_segments_device, then the 128
        launches; else the first projection's sgmv_apply_rows writes the
        grouping out).  Returns the kernels launched."""
        if self.grouped:
            sgmv.sgmv_build_segments_device(self.ra, self.L, out=self.meta)
            n = sgmv.sgmv_last_launch_count()
            for layer, g in self.launches:
                n += self.run_group(sgmv, layer, g)
            return n
        X, A, B, Y = self.projs[0]
        sgmv.sgmv_apply_rows(Y, X, A, B, self.ra, 1.0, out=self.meta)
        n = sgmv.sgmv_last_launch_count()
        for layer, g in self.launches:
            if layer == 0 and 0 in g:
                g = [k for k in g if k != 0]  # q of layer 0 went with the grouping
                if not g:
                    continue
            n += self.run_group(sgmv, layer, g)
        return n

    def step(self, sgmv):
        self.apply(sgmv)

    def update(self, sgmv):
        """All update launches of a step on the grouping of the last step
        (roofline)."""
        for layer, g in self.launches:
            self.run_group(sgmv, layer, g)

    @staticmethod
    def proj_bytes(H1, H2, T=128, L=128, r=16):
        return L * (H1 * r + r * H2) * 2 + T * H1 * 2 + 2 * T * H2 * 2

    def group_bytes(self, g):
        from rank_gemv_gb300 import workloads as wl

        return sum(self.proj_bytes(*wl.LLAMA7B_PROJ[k][1:]) for k in g)

    def bytes_moved(self):
        from rank_gemv_gb300 import workloads as wl

        return sum(self.proj_bytes(H1, H2) for _, H1, H2 in wl.LLAMA7B_PROJ) * wl.LLAMA7B_LAYERS


def capture(fns):
    import torch

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for fn in fns:
            fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def timed_replays(graph_full, n_per_graph, graph_rem, K):
    """Seconds of K steps: K // n replays of the rotation graph and one of the
    remainder graph, CUDA events on the replaying stream, synchronised on both
    sides."""
    import torch

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(K // n_per_graph):
        graph_full.replay()
    if graph_rem is not None:
        graph_rem.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def timed_regions(graph_full, n_per_graph, graph_rem, K, repeats, world):
    """`repeats` timed regions of exactly K steps, each bracketed by a barrier
    (N > 1) and a device synchronisation; returns their seconds."""
    out = []
    for _ in range(repeats):
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        out.append(timed_replays(graph_full, n_per_graph, graph_rem, K))
    return out


def isolated_stats(fn, flush, iters):
    """Device time (us) of fn() alone, median and 10th / 90th percentiles:
    before each call a write larger than L2 evicts its inputs, and CUDA events
    bracket the call."""
    import torch

    ts = []
    for i in range(iters):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    ts.sort()
    pick = lambda q: ts[min(len(ts) - 1, int(q * (len(ts) - 1) + 0.5))]
    return {"median": statistics.median(ts), "p10": pick(0.1), "p90": pick(0.9)}


def isolated_us(fn, flush, iters):
    """Median of isolated_stats."""
    return isolated_stats(fn, flush, iters)["median"]


def back_to_back_us(fns, calls, repeats=3):
    """Per-call device time (us) of `calls` calls back to back: a graph of one
    rotation over fns replayed; median of `repeats` timings."""
    n = len(fns)
    g = capture(fns)
    reps = max(1, calls // n)
    times = [timed_replays(g, 1, None, reps) for _ in range(repeats)]
    return statistics.median(times) / (reps * n) * 1e6


def hbm(bytes_, us, peak):
    gbs = bytes_ / (us * 1e-6) / 1e9
    return gbs, gbs / peak


def run_ours(args, rank, world, local):
    import torch

    from rank_gemv_gb300 import build as _build
    from rank_gemv_gb300 import sgmv
    from rank_gemv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    sgmv.load_library()
    K, W, R = args.steps, max(3, args.warmup), max(1, args.repeats)
    seed = args.seed + rank
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
    peak, peak_kind = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    if args.workload == "llama7b-stack":
        stack = StackBatch(seed, dev, sgmv, grouped=args.stack_calls == "grouped")
        batches = [stack]
        T = stack.T
        bytes_step = stack.bytes_moved()
        w0 = None
        l2_note = f"inputs {bytes_step / 1e9:.1f} GB per step, larger than L2 ({l2 / 1e6:.0f} MB)"
    else:
        w0 = wl.make(args.workload, seed)
        T = w0.T
        bytes_step = w0.bytes_moved()
        n_copies = rotation_copies(bytes_step, l2)
        batches = [Batch(w0, dev, sgmv) for _ in range(n_copies)]
        touched = n_copies * bytes_step
        l2_note = (f"rotating {n_copies} input copies, {touched / 1e6:.0f} MB touched per "
                   f"rotation" + (f" > 2 x L2 ({l2 / 1e6:.0f} MB)" if touched > 2 * l2
                                  else f", inside L2 ({l2 / 1e6:.0f} MB)"))

    if world > 1:
        import torch.distributed as dist

        dist.barrier()

    # warm-up (eager), then the graphs of one rotation and of the remainder
    for i in range(W):
        batches[i % len(batches)].step(sgmv)
    launches_step = batches[0].apply(sgmv)  # kernels per step, as the library reports them
    n_apply = batches[0].n_apply
    torch.cuda.synchronize()
    assert sgmv.sgmv_get_device_error(dev) == 0, "device error word set during warm-up"
    n = len(batches)
    g_full = capture([(lambda b=b: b.step(sgmv)) for b in batches])
    g_rem = capture([(lambda b=b: b.step(sgmv)) for b in batches[: K % n]]) if K % n else None
    # the update kernels alone, for the roofline
    k_full = capture([(lambda b=b: b.update(sgmv)) for b in batches])
    k_rem = capture([(lambda b=b: b.update(sgmv)) for b in batches[: K % n]]) if K % n else None
    batches[0].update(sgmv)
    per_call = sgmv.sgmv_last_launch_count()

    # soak under the clock sampler, then the timed regions
    sampler = ClockSampler(gpu_id_for(dev))
    t_end = time.perf_counter() + args.soak_seconds
    while time.perf_counter() < t_end:
        g_full.replay()
        torch.cuda.synchronize()
    regions = timed_regions(g_full, n, g_rem, K, R, world)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    kregions = timed_regions(k_full, n, k_rem, K, R, 1)
    assert sgmv.sgmv_get_device_error(dev) == 0, "device error word set during timing"

    elapsed, kernel_s = max_over_ranks([statistics.median(regions), statistics.median(kregions)],
                                       world, dev)
    value = replica_throughput(world, K, T, elapsed)
    # roofline of one update call, back to back (as a decode step runs its
    # calls) and alone after an L2 flush
    apply_us = kernel_s / (K * n_apply) * 1e6
    bytes_apply = bytes_step / n_apply
    achieved, frac = hbm(bytes_apply, apply_us, peak)
    if args.workload == "llama7b-stack":
        # every launch of layer 0 alone after an L2 flush; the mean over them
        # is one launch of the step on average (all layers have these shapes)
        from rank_gemv_gb300 import workloads as wl

        iso = {}
        for layer, g in stack.launches:
            if layer != 0:
                continue
            name = "+".join(wl.LLAMA7B_PROJ[k][0] for k in g)
            st = isolated_stats(lambda g=g: stack.run_group(sgmv, 0, g), flush, args.latency_iters)
            us = st["median"]
            iso[name] = {"us": us, "us_p10": st["p10"], "us_p90": st["p90"],
                         "bytes": stack.group_bytes(g),
                         "frac": hbm(stack.group_bytes(g), us, peak)[1]}
        iso_us = sum(v["us"] for v in iso.values()) / len(iso)
        iso_note = ("every update launch of layer 0, L2 flushed before each; mean over the "
                    f"layer's {len(iso)} launches")
    else:
        iso = None
        iso_st = isolated_stats(lambda: batches[0].update(sgmv), flush, args.latency_iters)
        iso_us = iso_st["median"]
        iso_note = (f"L2 flushed before each call; p10 {iso_st['p10']:.2f} us, "
                    f"p90 {iso_st['p90']:.2f} us")
    iso_gbs, iso_frac = hbm(bytes_apply, iso_us, peak)
    if args.workload == "prefill":
        kname = "sgmv_tc_shrink_kernel + sgmv_tc_expand_kernel (tensor cores; the streaming kernel gets no short segment)"
    elif w0 is not None and w0.T <= 64:
        kname = "sgmv_stream_kernel (grouping + shrink + expand in one launch, CUDA cores)"
    elif w0 is None and args.stack_calls == "grouped":
        kname = ("sgmv_stream_kernel, multi-problem instantiation (per layer q+k+v, o, gate+up, "
                 "down: 4 launches; shrink + expand on CUDA cores; grouping excluded)")
    else:
        kname = "sgmv_stream_kernel (shrink + expand, CUDA cores; grouping excluded)"
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": elapsed / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": (config_of(args.workload, w0, l2_note) if w0 is not None
                   else stack_config(l2_note, args.stack_calls == "grouped")),
        "repeats": {"n": R, "ms_per_step": [t / K * 1e3 for t in regions],
                    "value_from": "median region"},
        "hbm_gbs": bytes_step * K / elapsed / 1e9,
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "kernel": kname, "kernels_per_call": per_call,
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": frac,
                     "peak_kind": peak_kind, "traffic": profiled_traffic(args.workload),
                     "source_hash": source_hash(WORKLOAD_KERNELS.get(args.workload, "stream")), "bytes_per_call": bytes_apply,
                     "call_us": apply_us,
                     "frac_uses": f"call_us: {n_apply * K} update launches back to back in CUDA "
                                  f"graphs, median of {R} regions",
                     "isolated": {"call_us": iso_us, "achieved": iso_gbs, "frac": iso_frac,
                                  "method": f"median of {args.latency_iters}; {iso_note}",
                                  **({"by_shape": iso} if iso else {})}},
        "gpu_launches": K * launches_step,
        "clocks": clocks,
    }
    if not args.no_extras and rank == 0:
        del g_full, g_rem, k_full, k_rem
        torch.cuda.synchronize()
        side = {}
        for name in SIDE_WORKLOADS:
            if name != args.workload:
                side[name] = measure_workload(name, args, dev, sgmv, wl, l2, peak, flush)
        fl = fused_layer_point(sgmv, wl, dev, 4096, 4096, 128, args.seed + 5, args.latency_iters,
                               flush, l2, peak)
        side["fused-linear-lora-q"] = fl
        if "decode-distinct" in side and "decode-shared" in side:
            d, s = side["decode-distinct"], side["decode-shared"]
            side["distinct_vs_shared"] = {
                "isolated_step_ratio": d["isolated"]["step_us"] / s["isolated"]["step_us"],
                "back_to_back_step_ratio": d["back_to_back"]["step_us"] / s["back_to_back"]["step_us"],
                "target": 1.3}
        out["workloads"] = side
    if not args.no_extras:
        out["e2e"] = e2e(args, dev, sgmv, wl, world, seed, K, W)
    if rank == 0 and world == 1 and not args.no_extras:
        out["cpu_baseline"] = cpu_baseline(args, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_workload(name, args, dev, sgmv, wl, l2, peak, flush):
    """One named workload beside the headline: the update call (and the whole
    step, grouping included) back to back over rotating input copies and alone
    after an L2 flush; for decode batches (up to 64 rows) also the read-only
    floor of the same bytes with the streaming kernel's launch shape."""
    import torch

    w = wl.make(name, args.seed)
    nbytes = w.bytes_moved()
    n_copies = rotation_copies(nbytes, l2)
    batches = [Batch(w, dev, sgmv) for _ in range(n_copies)]
    for b in batches:
        b.step(sgmv)
    torch.cuda.synchronize()
    assert sgmv.sgmv_get_device_error(dev) == 0, f"device error word set on {name}"
    calls = max(4 * n_copies, 200)
    res = {"T": w.T, "bytes_per_call": nbytes,
           "inputs": f"{n_copies} rotating copies, {n_copies * nbytes / 1e6:.0f} MB touched per "
                     "rotation" + (" (> 2 x L2)" if n_copies * nbytes > 2 * l2 else " (inside L2)")}
    b2b_call = back_to_back_us([(lambda b=b: b.update(sgmv)) for b in batches], calls)
    b2b_step = back_to_back_us([(lambda b=b: b.step(sgmv)) for b in batches], calls)
    iso_st = isolated_stats(lambda: batches[0].update(sgmv), flush, args.latency_iters)
    iso_call = iso_st["median"]
    iso_step = isolated_us(lambda: batches[0].step(sgmv), flush, args.latency_iters)
    g1, f1 = hbm(nbytes, b2b_call, peak)
    g2, f2 = hbm(nbytes, iso_call, peak)
    res["back_to_back"] = {"call_us": b2b_call, "gbs": g1, "frac": f1, "step_us": b2b_step,
                           "rows_per_s": w.T / (b2b_step * 1e-6)}
    res["isolated"] = {"call_us": iso_call, "call_us_p10": iso_st["p10"],
                       "call_us_p90": iso_st["p90"], "gbs": g2, "frac": f2, "step_us": iso_step}
    if w.T <= 64 and w.r % 4 == 0 and w.r <= 64:
        nb = (nbytes + 15) // 16 * 16
        src = torch.zeros(n_copies * nb // 4, dtype=torch.int32, device=dev)
        srcs = [src[i * nb // 4:(i + 1) * nb // 4] for i in range(n_copies)]
        shape = {}

        def floor(s):
            shape["grid"] = sgmv.sgmv_read_floor(s, nb, w.T, w.L, w.H1, w.H2, w.r, w.dtype,
                                                 w.y_dtype)
        floor(srcs[0])
        fb = back_to_back_us([(lambda s=s: floor(s)) for s in srcs], calls)
        fi = isolated_us(lambda: floor(srcs[0]), flush, args.latency_iters)
        res["floor"] = {"ctas": shape["grid"][0], "cluster": shape["grid"][1],
                        "back_to_back_us": fb, "isolated_us": fi,
                        "frac_back_to_back": hbm(nb, fb, peak)[1],
                        "frac_isolated": hbm(nb, fi, peak)[1],
                        "call_over_floor_back_to_back": b2b_call / fb,
                        "call_over_floor_isolated": iso_call / fi}
        del src, srcs
    assert sgmv.sgmv_get_device_error(dev) == 0, f"device error word set on {name}"
    del batches
    torch.cuda.empty_cache()
    return res


def _packed(tensors, device, pin=False):
    """One byte buffer holding copies of `tensors` at 256-byte-aligned offsets,
    and a view of each (so a step's inputs move in one copy)."""
    import torch

    offs, n = [], 0
    for t in tensors:
        n = (n + 255) // 256 * 256
        offs.append(n)
        n += t.nbytes
    buf = torch.empty(n, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + t.nbytes].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    for v, t in zip(views, tensors):
        v.copy_(t)
    return buf, views


def e2e(args, dev, sgmv, wl, world, seed, K, W):
    """The metric through the public API with host buffers, as a serving loop
    runs it: every step copies that step's inputs (rows, row -> adapter ids,
    y) from page-locked host memory, groups and applies, and copies y back;
    the host waits for, and reads, each step's result.  Steps are pipelined
    over three streams: the copies in on one (for the stack, all 449 pieces
    in one sgmv_copy_gather call), the update calls on the compute stream,
    the copies out on a third (the stack's 224 results in one
    sgmv_copy_gather call); events order each step's three parts, and D sets
    of buffers (D = 4, 2 for the stack) let step s copy in while step s-1
    computes.  The host waits for step s-D's result just before step s
    reuses its buffers.  The update calls are issued eagerly through the
    Python binding (`value`: argument checks, tensor-map encoding and
    launches inside the loop), and, for comparison, as one CUDA-graph replay
    per step (`graphed`).  A single-projection step's x, y and ids sit in one
    page-locked buffer and move in one copy.  `breakdown_us` times the parts
    alone: the copies in and out (device time), the step's kernels (device
    time), and the host time of issuing the step's API calls."""
    import torch

    gather_ctas = 64  # the host link is saturated by 64 CTAs; the rest compute
    if args.workload == "llama7b-stack":
        # inputs per step: the 224 projections' X and Y rows and the ids
        sets = []
        for _ in range(2):
            stack = StackBatch(seed, dev, sgmv)
            hx = [X.cpu().pin_memory() for X, _, _, _ in stack.projs]
            hy = [Y.cpu().pin_memory() for _, _, _, Y in stack.projs]
            hout = [torch.empty_like(h).pin_memory() for h in hy]
            hra = stack.ra.cpu().pin_memory()
            sets.append((stack, hx, hy, hout, hra))

        def parts(st):
            stack, hx, hy, hout, hra = st
            din = [stack.ra] + [X for X, _, _, _ in stack.projs] + [Y for _, _, _, Y in stack.projs]
            sin = [hra] + hx + hy
            dev_y = [Y for _, _, _, Y in stack.projs]

            def h2d(s):
                sgmv.sgmv_copy_gather(din, sin, stream=s, max_ctas=gather_ctas)

            def d2h(s):
                sgmv.sgmv_copy_gather(hout, dev_y, stream=s, max_ctas=gather_ctas)
            return h2d, (lambda: stack.step(sgmv)), d2h, hout[0]

        stack0, hx0, hy0, hout0, hra0 = sets[0]
        h2d_b = sum(h.nbytes for h in hx0) + sum(h.nbytes for h in hy0) + hra0.nbytes
        d2h_b = sum(h.nbytes for h in hout0)
        T = stack0.T
        K = min(K, 20)
    else:
        w = wl.make(args.workload, seed)
        sets = []
        for _ in range(4):
            b = Batch(w, dev, sgmv)
            dbuf, (b.X, b.Y, b.ra) = _packed([w.X, w.Y0, w.row_adapter], dev)
            hbuf, _ = _packed([w.X, w.Y0, w.row_adapter], "cpu", pin=True)
            sets.append((b, dbuf, hbuf, torch.empty_like(w.Y0).pin_memory()))

        def parts(st):
            b, dbuf, hbuf, hout = st

            def h2d(s):
                with torch.cuda.stream(s):
                    dbuf.copy_(hbuf, non_blocking=True)

            def d2h(s):
                with torch.cuda.stream(s):
                    hout.copy_(b.Y, non_blocking=True)
            return h2d, (lambda: b.step(sgmv)), d2h, hout

        _, _, hbuf0, hout0 = sets[0]
        h2d_b, d2h_b, T = hbuf0.nbytes, hout0.nbytes, w.T
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    steps = [parts(st) for st in sets]
    D = len(steps)
    ev_in = [torch.cuda.Event() for _ in steps]
    ev_k = [torch.cuda.Event() for _ in steps]
    done = [torch.cuda.Event() for _ in steps]  # step's result copied out

    def issue(i, kern):
        h2d, _, d2h, _ = steps[i]
        s_in.wait_event(done[i])  # the last copy out of set i has read its y
        h2d(s_in)
        ev_in[i].record(s_in)
        comp.wait_event(ev_in[i])
        kern()
        ev_k[i].record(comp)
        s_out.wait_event(ev_k[i])
        d2h(s_out)
        done[i].record(s_out)

    for i, (_, kern, _, _) in enumerate(steps):  # eager warm-up
        for _ in range(W):
            issue(i, kern)
    torch.cuda.synchronize()
    graphs = [capture([kern]) for _, kern, _, _ in steps]
    outs = [st[3] for st in steps]
    checksum = 0.0

    def run(n, graphed):
        nonlocal checksum
        for s_ in range(n):
            i = s_ % D
            if s_ >= D:
                done[i].synchronize()                  # step s-D's result is on the host
                checksum += float(outs[i].view(-1)[0])  # ... and read there
            issue(i, graphs[i].replay if graphed else steps[i][1])
        for i in range(min(n, D)):
            done[i].synchronize()
            checksum += float(outs[i].view(-1)[0])

    def timed(graphed):
        run(W, graphed)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run(K, graphed)
        torch.cuda.synchronize()
        return time.perf_counter() - t0  # every stream's work is inside

    el = timed(False)
    el_g = timed(True)
    assert sgmv.sgmv_get_device_error(dev) == 0, "device error word set during e2e"

    # the parts alone
    h2d, kern, d2h, _ = steps[0]

    def dev_us(fn, iters=10):
        ts = []
        for _ in range(iters):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def host_us(fn, iters=10):
        ts = []
        for _ in range(iters):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            ts.append((time.perf_counter() - t0) * 1e6)
            torch.cuda.synchronize()
        return statistics.median(ts)

    h2d_us, d2h_us = dev_us(lambda: h2d(comp)), dev_us(lambda: d2h(comp))
    breakdown = {"h2d_us": h2d_us, "d2h_us": d2h_us, "kernels_us": dev_us(kern),
                 "api_host_us": host_us(kern),
                 "h2d_gbs": h2d_b / (h2d_us * 1e3), "d2h_gbs": d2h_b / (d2h_us * 1e3)}
    return {"value": world * K * T / el, "unit": UNIT, "h2d_bytes_per_step": h2d_b,
            "d2h_bytes_per_step": d2h_b, "steps": K, "ms_per_step": el / K * 1e3,
            "method": "eager API calls each step (Python binding -> C ABI), copies from/to "
                      "page-locked host memory on their own streams (sgmv_copy_gather for "
                      f"the stack's pieces), {D} steps in flight; host waits for and reads "
                      "every step's result; wall clock",
            "graphed": {"value": world * K * T / el_g, "ms_per_step": el_g / K * 1e3,
                        "method": "the same, with each step's update calls as one CUDA-graph "
                                  "replay (host-side checks and launches not in the loop)"},
            "breakdown_us": breakdown}


# -------------------------------------------------- oracle (host cores)
def oracle_tasks(perm, seg_ptr, idx, n_tasks):
    """Split the sorted positions of a grouped batch into about n_tasks ranges
    of consecutive positions; each task is (rows, seg_ptr, idx) of an
    independent SGMV problem on those rows (the segments clipped to the
    range, positions re-based to 0)."""
    import numpy as np

    total = int(seg_ptr[-1]) if len(seg_ptr) else 0
    n_tasks = max(1, min(n_tasks, total))
    cuts = [round(i * total / n_tasks) for i in range(n_tasks + 1)]
    tasks = []
    for p0, p1 in zip(cuts[:-1], cuts[1:]):
        if p1 <= p0:
            continue
        sp, ix = [0], []
        for s in range(len(idx)):
            a, b = max(int(seg_ptr[s]), p0), min(int(seg_ptr[s + 1]), p1)
            if a < b:
                ix.append(int(idx[s]))
                sp.append(sp[-1] + b - a)
        tasks.append((np.asarray(perm[p0:p1], dtype=np.int64), np.asarray(sp, np.int32),
                      np.asarray(ix, np.int32)))
    return tasks


def oracle_apply_parallel(o, pool, Y, X, A, B, perm, seg_ptr, idx, scale, n_tasks):
    """The oracle's SGMV update of a grouped batch, as independent oracle calls
    on ranges of its rows run by the threads of `pool` (the C code releases
    the interpreter lock).  Every output element is computed by the same
    oracle arithmetic as in one call, so the result is identical to
    o.sgmv_apply(Y, X, A, B, seg_ptr, idx, scale, perm=perm)."""
    out = Y.copy()

    def one(task):
        rows, sp, ix = task
        out[rows] = o.sgmv_apply(Y[rows], X[rows], A, B, sp, ix, scale, widened=True)

    list(pool.map(one, oracle_tasks(perm, seg_ptr, idx, n_tasks)))
    return out


def _oracle_sample(name, seed):
    """(problems, metric rows per pass, description) of a bounded sample of the
    workload for the oracle; a problem is (Y, X, A, B, row_adapter, L, scale)
    widened to float64."""
    import oracle
    from rank_gemv_gb300 import workloads as wl

    if name == "llama7b-stack":
        problems = []
        for p in range(len(wl.LLAMA7B_PROJ)):
            X, A, B, Y = wl.stack_projection(seed, 0, p)
            problems.append((oracle.widen(Y), oracle.widen(X), oracle.widen(A), oracle.widen(B),
                             wl.stack_row_adapter(128), 128, 1.0))
        # one layer of 7 projections on all 128 rows stands for 1/32 of a pass
        return problems, 128 / 32.0, "all 128 rows of layer 0 (7 of 224 projections = 1/32 of a step)"
    w = wl.make(name, seed)
    per_row = w.H1 * w.r + w.r * w.H2
    rows = int(max(1, min(w.T, 4e8 // per_row)))
    problems = [(oracle.widen(w.Y0[:rows]), oracle.widen(w.X[:rows]), oracle.widen(w.A),
                 oracle.widen(w.B), w.row_adapter[:rows], w.L, w.scale)]
    desc = "whole batch" if rows == w.T else f"first {rows} of {w.T} rows"
    return problems, float(rows), desc


def oracle_step(problems, threads):
    """One oracle pass (grouping + fp64 update of every problem) on `threads`
    host threads; returns the step function and a closer for its pool."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    o = oracle.default()
    pool = ThreadPoolExecutor(threads) if threads > 1 else None

    def step():
        for Y, X, A, B, ra, L, scale in problems:
            perm, seg_ptr, idx = o.build_segments(ra, L)
            if pool is None:
                o.sgmv_apply(Y, X, A, B, seg_ptr, idx, scale, perm=perm, widened=True)
            else:
                oracle_apply_parallel(o, pool, Y, X, A, B, perm, seg_ptr, idx, scale,
                                      4 * threads)

    return step, (pool.shutdown if pool is not None else (lambda: None))


def _time_passes(step, budget_s):
    step()
    n, t0 = 0, time.perf_counter()
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return n, el


def cpu_baseline(args, budget_s):
    """The oracle on the host cores: all cores (`value`, `cores` = threads
    used) and one thread, each for about budget_s seconds."""
    problems, rows, desc = _oracle_sample(args.workload, args.seed)
    nthr = host_threads()
    res = {}
    for threads in (nthr, 1):
        step, close = oracle_step(problems, threads)
        try:
            n, el = _time_passes(step, budget_s)
        finally:
            close()
        res[threads] = (n * rows / el, n, el)
    v, n, el = res[nthr]
    v1, n1, el1 = res[1]
    return {"value": v, "unit": UNIT, "cores": nthr, "kind": "oracle",
            "sample": f"{desc}; {n} oracle passes (grouping + fp64 update, {nthr} threads over "
                      f"ranges of rows) in {el:.1f} s",
            "single_core": {"value": v1, "cores": 1,
                            "sample": f"{n1} passes on one thread in {el1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from rank_gemv_gb300 import workloads as wl

    problems, rows, desc = _oracle_sample(args.workload, args.seed)
    nthr = host_threads()
    step, close = oracle_step(problems, nthr)
    try:
        W = max(3, args.warmup)
        for _ in range(W):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    finally:
        close()
    value = args.steps * rows / el
    w = None if args.workload == "llama7b-stack" else wl.make(args.workload, args.seed)
    cfg = (config_of(args.workload, w) if w is not None
           else stack_config(None, args.stack_calls == "grouped"))
    sample = (f"{desc}; one oracle pass (grouping + fp64 update, {nthr} threads over ranges of "
              "rows) per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": W, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def max_over_ranks(values, world, device=None):
    """The largest of each value over all ranks (the job's time is its slowest
    replica's); the values themselves when there is one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def replica_throughput(world, K, T, elapsed):
    """Rows/s of the whole job: every replica ran K steps of T rows within
    `elapsed` seconds (the slowest rank's time)."""
    return world * K * T / elapsed


def figure_point(sgmv, dev, W, A, B, T, n_adapters, seed):
    """One point of the latency-vs-batch figure: T rows over n_adapters adapters
    (round robin, shuffled).  Returns the three methods as callables on shared
    buffers, the largest difference between the per-adapter loop and SGMV
    relative to RMS(y), and the inputs (x, row -> adapter ids, y)."""
    import torch

    H1, H2 = W.shape
    g = torch.Generator().manual_seed(seed)
    ids = (torch.arange(T) % n_adapters)[torch.randperm(T, generator=g)].to(torch.int32)
    x = torch.randn(T, H1, generator=g).to(W.dtype).to(dev)
    y = torch.empty(T, H2, dtype=W.dtype, device=dev)
    ra = ids.to(dev)
    groups = [(int(a), (ids == a).nonzero().flatten().to(dev)) for a in torch.unique(ids)]
    smax = sgmv.sgmv_max_segments(T, A.shape[0])
    meta = (torch.empty(T, dtype=torch.int32, device=dev),
            torch.empty(smax + 1, dtype=torch.int32, device=dev),
            torch.empty(smax, dtype=torch.int32, device=dev),
            torch.empty(1, dtype=torch.int32, device=dev))

    def base():
        torch.matmul(x, W, out=y)

    def naive():  # the loop the pages compare against: one pair of matmuls per adapter
        base()
        for a, rows in groups:
            y.index_add_(0, rows, (x.index_select(0, rows) @ A[a]) @ B[a])

    def with_sgmv():
        base()
        sgmv.sgmv_apply_rows(y, x, A, B, ra, 1.0, out=meta)

    naive()
    y_naive = y.float().clone()
    with_sgmv()
    y_sgmv = y.float()
    rms = y_naive.pow(2).mean().sqrt().item()
    err = (y_naive - y_sgmv).abs().max().item() / max(rms, 1e-30)
    return {"base": base, "naive": naive, "sgmv": with_sgmv}, err, (x, ids, y)


def fused_layer_point(sgmv, wl, dev, H1, H2, T, seed, iters, flush, l2, peak):
    """The LoRA layer y = x W + (x A[a]) B[a] for T decode rows, each on its own
    adapter out of 128 (r = 16, fp16): cuBLAS x W alone ("base"), x W then
    sgmv_apply ("two_step", the grouping built once and reused, as a model's
    layers reuse it), and sgmv_fused_linear_lora ("fused", same grouping).
    Each method alone after an L2 flush (median of `iters`) and back to back
    over rotating copies of the weights whose pass exceeds twice the L2."""
    import torch

    L, r = 128, 16
    per_copy = H1 * H2 * 2 + L * (H1 * r + r * H2) * 2
    n_copies = rotation_copies(per_copy, l2, cap=8)
    sets = []
    for c in range(n_copies):
        X, A, B = _fused_inputs(wl, dev, H1, H2, T, L, r, seed + c)
        W = wl.base_weight(H1, H2, seed=seed + 31 + c, device=dev)
        sets.append((X, A, B, W, torch.empty(T, H2, dtype=torch.float16, device=dev)))
    g = torch.Generator().manual_seed(seed)
    ra = torch.randperm(L, generator=g)[:T].to(torch.int32).to(dev)
    perm, seg_ptr, idx, _ = sgmv.sgmv_build_segments_device(ra, L)
    ws = torch.empty(sgmv.sgmv_fused_workspace_bytes(T, H2, r), dtype=torch.uint8, device=dev)

    def base(st):
        X, A, B, W, y = st
        torch.matmul(X, W, out=y)

    def two_step(st):
        X, A, B, W, y = st
        torch.matmul(X, W, out=y)
        sgmv.sgmv_apply(y, X, A, B, seg_ptr, idx, 1.0, perm=perm)

    def fused(st):
        X, A, B, W, y = st
        sgmv.sgmv_fused_linear_lora(y, X, W, A, B, seg_ptr, idx, 1.0, perm=perm, workspace=ws)

    two_step(sets[0])
    y_two = sets[0][4].float().clone()
    fused(sets[0])
    y_fused = sets[0][4].float()
    rms = y_two.pow(2).mean().sqrt().item()
    err = (y_two - y_fused).abs().max().item() / max(rms, 1e-30)
    nbytes = (H1 * H2 + T * (H1 * r + r * H2) + T * H1 + T * H2) * 2
    out = {"T": T, "H1": H1, "H2": H2, "adapters": T, "r": r, "unit": "us",
           "bytes_per_call": nbytes, "max_diff_over_rms": err}
    for name, fn in (("base", base), ("two_step", two_step), ("fused", fused)):
        for _ in range(3):
            fn(sets[0])
        torch.cuda.synchronize()
        graph = capture([lambda: fn(sets[0])])
        out[name] = isolated_us(graph.replay, flush, iters)
        out[name + "_back_to_back"] = back_to_back_us([(lambda st=st: fn(st)) for st in sets],
                                                      max(8 * n_copies, 64))
    assert sgmv.sgmv_get_device_error(dev) == 0
    out["fused_frac"] = hbm(nbytes, out["fused"], peak)[1]
    out["fused_frac_back_to_back"] = hbm(nbytes, out["fused_back_to_back"], peak)[1]
    out["fused_over_two_step"] = out["fused"] / out["two_step"]
    return out


def _fused_inputs(wl, dev, H1, H2, T, L, r, seed):
    """x [T, H1], A [L, H1, r], B [L, r, H2] (fp16, the workloads' distributions),
    drawn on the device."""
    import torch

    g = torch.Generator(device=dev).manual_seed(seed)
    X = wl._normal(g, (T, H1), 1.0, wl.F16, dev)
    A = wl._normal(g, (L, H1, r), H1 ** -0.5, wl.F16, dev)
    B = wl._normal(g, (L, r, H2), r ** -0.5, wl.F16, dev)
    return X, A, B


def run_fused(args):
    """The fused LoRA layer ("Punica: when LoRA fine-tuned models need
    multi-tenant serving", omica.com.cn article, §2.1: y = xW + xAB; "How to
    deploy several LoRA adapters without reloading the base model", aivaro.ru,
    §3.2, fused kernel) on one GB300: for each point, the layer with cuBLAS x W
    alone, with x W then SGMV, and fused.  Prints one JSON line per point."""
    import torch

    from rank_gemv_gb300 import build as _build
    from rank_gemv_gb300 import sgmv
    from rank_gemv_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sgmv.load_library()
    peak, _ = measured_peak()
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    points = [(4096, 4096, T) for T in (1, 8, 32, 64, 128)]
    points += [(4096, 11008, 128), (11008, 4096, 128)]
    if args.fused_point:
        points = [tuple(int(v) for v in args.fused_point.split(","))]
    for i, (H1, H2, T) in enumerate(points):
        out = fused_layer_point(sgmv, wl, dev, H1, H2, T, args.seed + 97 * i, args.latency_iters,
                                flush, l2, peak)
        out["bench"] = "fused_linear_lora"
        print(json.dumps(out), flush=True)


def run_figure(args):
    """The pages' micro-benchmark (the "Punica: when LoRA fine-tuned models need
    multi-tenant serving" article, §2.2 figure): one Llama-2-7B q projection,
    4096 -> 4096, r = 16, fp16, base weight W and 128 stacked adapters.  For
    each point, the latency of y = x W alone, of that plus a per-adapter loop
    of matmuls, and of that plus SGMV; one step after a 256 MB L2 flush, each
    method captured as a CUDA graph, median of --latency-iters.  Batches of
    1..128 rows on distinct adapters, then 2..100 adapters over 128 rows.
    Prints one JSON line per point."""
    import torch

    from rank_gemv_gb300 import build as _build
    from rank_gemv_gb300 import sgmv

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sgmv.load_library()
    H, r, L = 4096, 16, 128
    g = torch.Generator().manual_seed(args.seed)
    W = (torch.randn(H, H, generator=g) * H ** -0.5).half().to(dev)
    A = (torch.randn(L, H, r, generator=g) * H ** -0.5).half().to(dev)
    B = (torch.randn(L, r, H, generator=g) * r ** -0.5).half().to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    points = [(T, T) for T in (1, 2, 4, 8, 16, 32, 64, 128)]
    points += [(128, n) for n in (2, 4, 8, 16, 32, 64, 100)]
    for i, (T, n) in enumerate(points):
        fns, err, _ = figure_point(sgmv, dev, W, A, B, T, n, args.seed + i)
        assert err < 2e-2, f"per-adapter loop and SGMV disagree at T={T}, adapters={n}: {err}"
        out = {"figure": "latency_vs_batch", "layer": "llama2-7b q 4096x4096, r=16, fp16",
               "T": T, "adapters": n, "unit": "us", "max_diff_over_rms": err}
        for name, fn in fns.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fn()
            ts = []
            for it in range(args.latency_iters):
                flush.fill_(it & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                graph.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            out[name] = statistics.median(ts)
        assert sgmv.sgmv_get_device_error(dev) == 0
        print(json.dumps(out), flush=True)


def run_load(args):
    """On-demand adapter loading (the "Punica: Multi-Tenant LoRA Serving" review:
    adapters are loaded on demand, in milliseconds).  One Llama-2-7B adapter =
    32 layers x 7 projections of A [H1, 16] and B [16, H2], fp16, 80 MB, in
    page-locked host memory, loaded on a copy stream (a) as 448 copy-engine
    transfers (sgmv_load_adapter) and (b) as one sgmv_copy_gather kernel that
    reads the host memory directly, at several CTA caps: (1) alone; (2) while
    the compute stream replays llama7b-stack steps (all 224 SGMV calls over 128
    resident adapters), the loads going to spare pools so that no slot a
    running call reads is overwritten.  Prints one JSON line."""
    import torch

    from rank_gemv_gb300 import build as _build
    from rank_gemv_gb300 import sgmv
    from rank_gemv_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sgmv.load_library()
    r = 16
    g = torch.Generator().manual_seed(args.seed)
    host = []
    spare = []
    for _ in range(wl.LLAMA7B_LAYERS):
        for _, H1, H2 in wl.LLAMA7B_PROJ:
            host.append(((torch.randn(H1, r, generator=g) * H1 ** -0.5).half().pin_memory(),
                         (torch.randn(r, H2, generator=g) * r ** -0.5).half().pin_memory()))
            spare.append((torch.empty(2, H1, r, dtype=torch.half, device=dev),
                          torch.empty(2, r, H2, dtype=torch.half, device=dev)))
    adapter_bytes = sum(a.nbytes + b.nbytes for a, b in host)
    cs = torch.cuda.Stream(dev)

    def load(slot):
        for (A, B), (a, b) in zip(spare, host):
            sgmv.sgmv_load_adapter(A, B, slot, a, b, stream=cs)

    # one adapter's 448 copies as a graph on the copy stream (GPU-side time,
    # not the host's time to issue 448 calls), one graph per spare slot
    load(0)
    load(1)
    torch.cuda.synchronize()
    load_graphs = []
    for slot in (0, 1):
        lg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(lg, stream=cs):
            load(slot)
        load_graphs.append(lg)
    torch.cuda.synchronize()
    n = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        for i in range(3):
            load_graphs[i & 1].replay()
        torch.cuda.synchronize()
        e0.record(cs)
        for i in range(n):
            load_graphs[i & 1].replay()
        e1.record(cs)
    torch.cuda.synchronize()
    alone_ms = e0.elapsed_time(e1) / n
    ok = all(torch.equal(A[(n - 1) & 1].cpu(), a) and torch.equal(B[(n - 1) & 1].cpu(), b)
             for (A, B), (a, b) in zip(spare, host))

    stack = StackBatch(args.seed, dev, sgmv)
    stack.step(sgmv)
    torch.cuda.synchronize()
    graph = capture([lambda: stack.step(sgmv)])
    steps = 8  # longer than the loads below, which run inside this window
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(steps):
        graph.replay()
    s1.record()
    torch.cuda.synchronize()
    step_alone = s0.elapsed_time(s1) / steps
    # both at once: steps enqueued first, then the loads on the copy stream
    s0.record()
    for _ in range(steps):
        graph.replay()
    s1.record()
    with torch.cuda.stream(cs):
        e0.record(cs)
        for i in range(n):
            load_graphs[i & 1].replay()
        e1.record(cs)
    torch.cuda.synchronize()
    busy_load_ms = e0.elapsed_time(e1) / n
    step_busy = s0.elapsed_time(s1) / steps

    # host time to issue one adapter's loads
    def host_ms(fn, reps=5):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            ts.append((time.perf_counter() - t0) * 1e3)
        torch.cuda.synchronize()
        return statistics.median(ts)

    issue_copy_ms = host_ms(lambda: load(0))
    # the link's reference: the same bytes as ONE copy-engine transfer
    big_h = torch.empty(adapter_bytes, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(adapter_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(cs):
        for _ in range(3):
            big_d.copy_(big_h, non_blocking=True)
        torch.cuda.synchronize()
        e0.record(cs)
        for _ in range(n):
            big_d.copy_(big_h, non_blocking=True)
        e1.record(cs)
    torch.cuda.synchronize()
    one_transfer_ms = e0.elapsed_time(e1) / n
    del big_h, big_d
    dsts = [[t[slot] for A, B in spare for t in (A, B)] for slot in (0, 1)]
    srcs = [t for a, b in host for t in (a, b)]
    gather = {}
    for ctas in (0, 304, 152, 64, 32, 16):
        def gload(slot, ctas=ctas):
            sgmv.sgmv_copy_gather(dsts[slot], srcs, stream=cs, max_ctas=ctas)
            assert sgmv.load_library().sgmv_last_launch_count() == 1

        for A, B in spare:
            A.zero_()
            B.zero_()
        torch.cuda.synchronize()
        issue_ms = host_ms(lambda: gload(0))
        gload(1)
        torch.cuda.synchronize()
        g_ok = all(torch.equal(A[i].cpu(), a) and torch.equal(B[i].cpu(), b)
                   for (A, B), (a, b) in zip(spare, host) for i in (0, 1))
        ggraphs = []
        for slot in (0, 1):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=cs, capture_error_mode="relaxed"):
                gload(slot)
            ggraphs.append(gg)
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            for i in range(3):
                ggraphs[i & 1].replay()
            torch.cuda.synchronize()
            e0.record(cs)
            for i in range(n):
                ggraphs[i & 1].replay()
            e1.record(cs)
        torch.cuda.synchronize()
        g_alone = e0.elapsed_time(e1) / n
        s0.record()
        for _ in range(steps):
            graph.replay()
        s1.record()
        with torch.cuda.stream(cs):
            e0.record(cs)
            for i in range(n):
                ggraphs[i & 1].replay()
            e1.record(cs)
        torch.cuda.synchronize()
        gather[str(ctas or "4 per SM")] = {
            "load_ms_alone": g_alone, "load_gbs_alone": adapter_bytes / g_alone / 1e6,
            "load_ms_during_sgmv": e0.elapsed_time(e1) / n,
            "stack_step_ms_during_loads": s0.elapsed_time(s1) / steps,
            "host_issue_ms": issue_ms, "bit_exact": g_ok}
        del ggraphs

    # cold start: 50 adapters of rank 32 (160 MB each, Llama-2-7B shapes) into
    # empty pools, one sgmv_copy_gather call per adapter, back to back on the
    # copy stream (one page-locked source adapter, loaded into every slot:
    # the same bytes cross the link as for 50 different adapters)
    n_cold, r_cold = 50, 32
    src32, pools32 = [], []
    for _ in range(wl.LLAMA7B_LAYERS):
        for _, H1, H2 in wl.LLAMA7B_PROJ:
            src32.append(((torch.randn(H1, r_cold, generator=g) * H1 ** -0.5).half().pin_memory(),
                          (torch.randn(r_cold, H2, generator=g) * r_cold ** -0.5).half()
                          .pin_memory()))
            pools32.append((torch.empty(n_cold, H1, r_cold, dtype=torch.half, device=dev),
                            torch.empty(n_cold, r_cold, H2, dtype=torch.half, device=dev)))
    cold_bytes = sum(a.nbytes + b.nbytes for a, b in src32)
    srcs32 = [t for a, b in src32 for t in (a, b)]

    def cold_start():
        for slot in range(n_cold):
            sgmv.sgmv_copy_gather([t[slot] for A, B in pools32 for t in (A, B)], srcs32,
                                  stream=cs, max_ctas=64)

    cold_start()  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(cs)
    cold_start()
    e1.record(cs)
    torch.cuda.synchronize()
    cold = {"adapters": n_cold, "rank": r_cold, "bytes_per_adapter": cold_bytes,
            "ms": e0.elapsed_time(e1), "wall_ms": (time.perf_counter() - t0) * 1e3,
            "gbs": n_cold * cold_bytes / e0.elapsed_time(e1) / 1e6,
            "bit_exact": all(torch.equal(A[n_cold - 1].cpu(), a) and torch.equal(B[0].cpu(), b)
                             for (A, B), (a, b) in zip(pools32, src32))}
    del pools32, src32, srcs32
    assert sgmv.sgmv_get_device_error(dev) == 0
    print(json.dumps({
        "bench": "adapter_load", "adapter": "llama2-7b, 224 projections, r=16, fp16",
        "adapter_bytes": adapter_bytes, "copies_per_adapter": 2 * len(host),
        "load_ms_alone": alone_ms, "load_gbs_alone": adapter_bytes / alone_ms / 1e6,
        "load_ms_during_sgmv": busy_load_ms,
        "stack_step_ms_alone": step_alone, "stack_step_ms_during_loads": step_busy,
        "host_issue_ms": issue_copy_ms,
        "one_transfer_ms": one_transfer_ms,
        "one_transfer_gbs": adapter_bytes / one_transfer_ms / 1e6,
        "loads_during_run": n, "steps_during_run": steps, "copies_bit_exact": ok,
        "gather_by_cta_cap": gather,
        "cold_start": cold,
        "host_memory": "page-locked"}), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.load:
        if rank == 0:
            run_load(args)
        return
    if args.figure:
        if rank == 0:
            run_figure(args)
        return
    if args.fused:
        if rank == 0:
            run_fused(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
