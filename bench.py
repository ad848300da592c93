#!/usr/bin/env python3
"""Benchmark of the SGMV multi-LoRA hot path on GB300.

One step = one pass of the whole path over one batch through the C ABI:
sgmv_apply_rows groups the batch's rows by adapter, gathers x, shrinks,
expands and scatters into y (one kernel for decode batches; grouping kernel +
CUDA-core + tensor-core kernels for prefill).  The llama7b-stack workload runs
it for all 224 projections of one decode step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the fp64 oracle on the host cores

Prints one JSON line (rank 0).  `value` is rows/s with inputs resident in HBM;
inputs are rotated over enough copies that one pass over them exceeds twice
the L2 cache, and the K timed steps run as CUDA-graph replays.  `e2e` is the
same metric with each step's inputs copied from pinned host memory and its
result read back.  With N > 1 (torchrun) every rank runs an independent
replica: the path has no exchange step.
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


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode-distinct",
                   choices=["tiny", "decode-distinct", "decode-shared", "decode-zipf", "prefill",
                            "llama7b-q", "llama7b-stack"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="host-core budget of the oracle baseline sample")
    p.add_argument("--soak-seconds", type=float, default=1.0,
                   help="load before the timed region while clocks are sampled")
    p.add_argument("--latency-iters", type=int, default=50)
    p.add_argument("--no-extras", action="store_true",
                   help="skip e2e, cpu baseline and latency (for profiling runs)")
    p.add_argument("--load", action="store_true",
                   help="on-demand adapter loading instead: one Llama-2-7B adapter (224 "
                        "projections) from pinned host memory, alone and during the stack's SGMV")
    p.add_argument("--figure", action="store_true",
                   help="the pages' micro-benchmark instead: latency of the base layer alone, "
                        "with a per-adapter loop and with SGMV, over batch sizes and adapter counts")
    return p.parse_args()


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


# Sources of the C ABI's host-side argument checks and dispatch: they launch
# kernels but hold none, so a change there leaves the kernels' counters valid.
HOST_ONLY_SOURCES = ("sgmv_api.cu", "sgmv_noalloc.cu")


def source_hash():
    """Hash of the kernel sources: a profile's counters stand only for this code."""
    import hashlib

    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "rank_gemv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in HOST_ONLY_SOURCES:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(workload):
    """DRAM bytes per update call measured by ncu for this workload (from
    profiles/traffic.md), or None when the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    want = source_hash()
    for line in lines:
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 3 and cells[0] == workload and cells[1] == want:
            try:
                return float(cells[2])
            except ValueError:
                return None
    return None


def config_of(name, w, n_copies=None, l2_note=None):
    cfg = {"workload": name, "T": w.T, "L": w.L, "H1": w.H1, "H2": w.H2, "r": w.r,
           "inputs": str(w.dtype).replace("torch.", ""),
           "y": str(w.y_dtype).replace("torch.", ""),
           "segments": int(len(set(w.row_adapter.tolist()))), "parallelism": "replicas"}
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

    def group(self, sgmv):
        sgmv.sgmv_build_segments_device(self.ra, self.w.L, out=self.meta)

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


class StackBatch:
    """All 224 projections of the llama7b-stack workload, resident on the device."""

    def __init__(self, seed, dev, sgmv):
        import torch
        from rank_gemv_gb300 import workloads as wl

        self.T, self.L, self.r = 128, 128, 16
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

    def group(self, sgmv):
        sgmv.sgmv_build_segments_device(self.ra, self.L, out=self.meta)

    n_apply = 224

    def apply(self, sgmv):
        """One decode step over all 224 projections, as a serving loop runs it:
        the first call groups the batch (sgmv_apply_rows writes the grouping
        out), the other 223 reuse it through sgmv_apply."""
        perm, seg_ptr, idx, _ = self.meta
        n = 0
        for i, (X, A, B, Y) in enumerate(self.projs):
            if i == 0:
                sgmv.sgmv_apply_rows(Y, X, A, B, self.ra, 1.0, out=self.meta)
            else:
                sgmv.sgmv_apply(Y, X, A, B, seg_ptr, idx, 1.0, perm=perm, S=self.smax)
            n += sgmv.sgmv_last_launch_count()
        return n

    def step(self, sgmv):
        self.apply(sgmv)

    def update(self, sgmv):
        """All 224 update calls on the grouping of the last step (roofline)."""
        perm, seg_ptr, idx, _ = self.meta
        for X, A, B, Y in self.projs:
            sgmv.sgmv_apply(Y, X, A, B, seg_ptr, idx, 1.0, perm=perm, S=self.smax)

    def bytes_moved(self):
        from rank_gemv_gb300 import workloads as wl

        tot = 0
        for _, H1, H2 in wl.LLAMA7B_PROJ:
            tot += self.L * (H1 * self.r + self.r * H2) * 2 + self.T * H1 * 2 + 2 * self.T * H2 * 2
        return tot * wl.LLAMA7B_LAYERS


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
    return start.elapsed_time(end) / 1e3  # seconds


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from rank_gemv_gb300 import build as _build
    from rank_gemv_gb300 import sgmv
    from rank_gemv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    sgmv.load_library()
    K, W = args.steps, max(3, args.warmup)
    seed = args.seed + rank
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)

    if args.workload == "llama7b-stack":
        stack = StackBatch(seed, dev, sgmv)
        batches = [stack]
        T = stack.T
        bytes_step = stack.bytes_moved()
        w0 = None
        l2_note = f"inputs {bytes_step / 1e9:.1f} GB per step, larger than L2 ({l2 / 1e6:.0f} MB)"
    else:
        w0 = wl.make(args.workload, seed)
        T = w0.T
        bytes_step = w0.bytes_moved()
        per_copy = (w0.X.nbytes + w0.A.nbytes + w0.B.nbytes + 2 * w0.Y0.nbytes)
        n_copies = max(2, -(-2 * l2 // per_copy))
        batches = [Batch(w0, dev, sgmv) for _ in range(n_copies)]
        l2_note = (f"rotating {n_copies} input copies, {n_copies * per_copy / 1e6:.0f} MB per "
                   f"rotation > 2 x L2 ({l2 / 1e6:.0f} MB)")

    if world > 1:
        dist.barrier()

    # warm-up (eager), then the graphs of one rotation and of the remainder
    for i in range(W):
        batches[i % len(batches)].step(sgmv)
    # kernels per step, as reported by the library
    launches_apply = batches[0].apply(sgmv)
    launches_step = launches_apply
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

    # soak under the clock sampler, then the timed steps
    sampler = ClockSampler(gpu_id_for(dev))
    t_end = time.perf_counter() + args.soak_seconds
    while time.perf_counter() < t_end:
        g_full.replay()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed = timed_replays(g_full, n, g_rem, K)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    kernel_s = timed_replays(k_full, n, k_rem, K)
    assert sgmv.sgmv_get_device_error(dev) == 0, "device error word set during timing"

    elapsed, kernel_s = max_over_ranks([elapsed, kernel_s], world, dev)
    value = replica_throughput(world, K, T, elapsed)
    peak, peak_kind = measured_peak()
    # roofline of one update call (the streaming kernel for decode batches;
    # streaming + tensor-core shrink + expand for prefill), timed alone in a
    # graph of K steps' worth of calls
    apply_s = kernel_s / (K * n_apply)
    bytes_apply = bytes_step / n_apply
    achieved = bytes_apply / apply_s / 1e9
    if args.workload == "prefill":
        kname = "sgmv_tc_shrink_kernel + sgmv_tc_expand_kernel (tensor cores; the streaming kernel gets no short segment)"
    elif w0 is not None and w0.T <= 64:
        kname = "sgmv_stream_kernel (grouping + shrink + expand in one launch, CUDA cores)"
    else:
        kname = "sgmv_stream_kernel (shrink + expand, CUDA cores; grouping excluded)"
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": elapsed / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(args.workload, w0, l2_note=l2_note) if w0 is not None else {
            "workload": "llama7b-stack", "T": T, "L": 128, "r": 16, "layers": 32,
            "projections": 7, "inputs": "float16", "y": "float16", "segments": 128,
            "parallelism": "replicas", "l2": l2_note},
        "hbm_gbs": bytes_step * K / elapsed / 1e9,
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "kernel": kname, "kernels_per_call": per_call,
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": profiled_traffic(args.workload), "source_hash": source_hash(),
                     "bytes_per_call": bytes_apply, "call_us": apply_s * 1e6},
        "gpu_launches": K * launches_step,
        "clocks": clocks,
    }
    if args.workload == "decode-distinct" and not args.no_extras:
        out["latency_us"] = distinct_vs_shared(args, dev, sgmv, wl)
    if not args.no_extras:
        out["e2e"] = e2e(args, dev, sgmv, wl, world, seed, K, W)
    if rank == 0 and world == 1 and not args.no_extras:
        out["cpu_baseline"] = cpu_baseline(args, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)


def distinct_vs_shared(args, dev, sgmv, wl):
    """Median latency of one step with L2 flushed before it, for the batch of
    32 distinct adapters and for the same batch on one shared adapter."""
    import torch

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {}
    for name in ("decode-distinct", "decode-shared"):
        b = Batch(wl.make(name, args.seed), dev, sgmv)
        for _ in range(5):
            b.step(sgmv)
        ts = []
        for i in range(args.latency_iters):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            b.step(sgmv)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        res[name] = statistics.median(ts)
    return {"distinct": res["decode-distinct"], "shared": res["decode-shared"],
            "ratio": res["decode-distinct"] / res["decode-shared"],
            "method": f"median of {args.latency_iters}, L2 flushed (256 MB write) before each"}


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
    the host waits for, and reads, each step's result.  Steps are pipelined:
    D sets of buffers (D = 4, 2 for the stack), each step one CUDA-graph
    replay of those copies and API calls, and the host waits for step s-D's
    result just before step s reuses its buffers.  A single-projection step's
    x, y and ids sit in one page-locked buffer and move in one copy."""
    import torch

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

        def make_step(st):
            stack, hx, hy, hout, hra = st

            def one():
                stack.ra.copy_(hra, non_blocking=True)
                for (X, _, _, Y), a, b in zip(stack.projs, hx, hy):
                    X.copy_(a, non_blocking=True)
                    Y.copy_(b, non_blocking=True)
                stack.step(sgmv)
                for (_, _, _, Y), o in zip(stack.projs, hout):
                    o.copy_(Y, non_blocking=True)
            return one, hout[0]

        stack0, hx0, hy0, hout0, hra0 = sets[0]
        h2d = sum(h.nbytes for h in hx0) + sum(h.nbytes for h in hy0) + hra0.nbytes
        d2h = sum(h.nbytes for h in hout0)
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

        def make_step(st):
            b, dbuf, hbuf, hout = st

            def one():
                dbuf.copy_(hbuf, non_blocking=True)
                b.step(sgmv)
                hout.copy_(b.Y, non_blocking=True)
            return one, hout

        _, _, hbuf0, hout0 = sets[0]
        h2d, d2h, T = hbuf0.nbytes, hout0.nbytes, w.T
    steps = [make_step(st) for st in sets]
    for one, _ in steps:  # eager warm-up, then one graph per buffer set
        for _ in range(W):
            one()
    torch.cuda.synchronize()
    graphs = [capture([one]) for one, _ in steps]
    outs = [out for _, out in steps]
    done = [torch.cuda.Event() for _ in steps]
    checksum = 0.0

    D = len(steps)

    def run(n):
        nonlocal checksum
        for s_ in range(n):
            i = s_ % D
            if s_ >= D:
                done[i].synchronize()                  # step s-D's result is on the host
                checksum += float(outs[i].view(-1)[0])  # ... and read there
            graphs[i].replay()
            done[i].record()
        for i in range(min(n, D)):
            done[i].synchronize()
            checksum += float(outs[i].view(-1)[0])

    run(W)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    run(K)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    el = max(e0.elapsed_time(e1) / 1e3, wall)
    return {"value": world * K * T / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "ms_per_step": el / K * 1e3,
            "pipelining": f"{D} steps in flight; host waits for and reads every step's result"}


# -------------------------------------------------- oracle (host cores)
def _oracle_sample(name, seed):
    """(step function, rows per step, rows/s scale, sample description) for the
    oracle on a bounded sample of the workload."""
    import oracle
    from rank_gemv_gb300 import workloads as wl

    if name == "llama7b-stack":
        rows = 16
        projs = [wl.stack_projection(seed, 0, p) for p in range(len(wl.LLAMA7B_PROJ))]
        ra = wl.stack_row_adapter(128)[:rows]
        widened = [tuple(oracle.widen(t[:rows] if i in (0, 3) else t) for i, t in enumerate(pr))
                   for pr in projs]

        def step():
            perm, seg_ptr, idx = oracle.build_segments(ra, 128)
            for X, A, B, Y in widened:
                oracle.sgmv_apply(Y, X, A, B, seg_ptr, idx, 1.0, perm=perm, widened=True)

        # one layer of 7 projections stands for 1/32 of a pass
        return step, rows / 32.0, f"{rows} of 128 rows, layer 0 (7 of 224 projections)"
    w = wl.make(name, seed)
    per_row = w.H1 * w.r + w.r * w.H2
    rows = int(max(1, min(w.T, 20e6 // per_row)))
    X, A, B, Y = (oracle.widen(w.X[:rows]), oracle.widen(w.A), oracle.widen(w.B),
                  oracle.widen(w.Y0[:rows]))
    ra = w.row_adapter[:rows]

    def step():
        perm, seg_ptr, idx = oracle.build_segments(ra, w.L)
        oracle.sgmv_apply(Y, X, A, B, seg_ptr, idx, w.scale, perm=perm, widened=True)

    desc = "whole batch" if rows == w.T else f"first {rows} of {w.T} rows"
    return step, float(rows), desc


def cpu_baseline(args, budget_s):
    step, rows, desc = _oracle_sample(args.workload, args.seed)
    step()
    n, t0 = 0, time.perf_counter()
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": n * rows / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{desc}; {n} oracle passes (grouping + fp64 apply, one thread) "
                      f"in {el:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from rank_gemv_gb300 import workloads as wl

    step, rows, desc = _oracle_sample(args.workload, args.seed)
    W = max(3, args.warmup)
    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * rows / el
    w = None if args.workload == "llama7b-stack" else wl.make(args.workload, args.seed)
    cfg = config_of(args.workload, w) if w is not None else {"workload": "llama7b-stack"}
    sample = f"{desc}; one oracle pass (grouping + fp64 apply, one thread) per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": W, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
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
    page-locked host memory, copied with sgmv_load_adapter on a copy stream:
    (1) alone; (2) while the compute stream replays llama7b-stack steps (all
    224 SGMV calls over 128 resident adapters), the loads going to spare pools
    so that no slot a running call reads is overwritten.  Prints one JSON line."""
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
    assert sgmv.sgmv_get_device_error(dev) == 0
    print(json.dumps({
        "bench": "adapter_load", "adapter": "llama2-7b, 224 projections, r=16, fp16",
        "adapter_bytes": adapter_bytes, "copies_per_adapter": 2 * len(host),
        "load_ms_alone": alone_ms, "load_gbs_alone": adapter_bytes / alone_ms / 1e6,
        "load_ms_during_sgmv": busy_load_ms,
        "stack_step_ms_alone": step_alone, "stack_step_ms_during_loads": step_busy,
        "loads_during_run": n, "steps_during_run": steps, "copies_bit_exact": ok,
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
