"""RMSNorm forward + backward benchmark on GB300.

One step = rmsnorm_fwd then rmsnorm_bwd (main kernel + dW finalizer) over a
bf16 16384 x 8192 activation matrix (llama mode, eps 1e-6, offset 0, 1%
outlier columns), inputs resident in HBM. The metric is achieved HBM
bandwidth: algorithmic bytes (every tensor read and written, including the
backward's fp32 workspace, written then read) per step / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0. Under torchrun each rank runs the same
workload on its own GPU (independent batches, no collective on the data
path): weak scaling, value = bytes of all ranks / max time over ranks.
`--impl reference` times the CPU oracle (fp64 C, all host cores) on a
bounded row sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "wide_bf16_16384x8192"
WORKLOAD_DESC = ("rmsnorm fwd+bwd bf16 M=16384 N=8192, llama mode eps=1e-6 offset=0, "
                 "1% outlier columns x20")
METRIC = "RMSNorm fwd/bwd achieved HBM GB/s (% of GB300 peak) and us/call, bf16 16384x8192"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time fwd and bwd over the shape sweep, fused-add and misaligned cases; "
                         "one JSON line per point (not the headline line)")
    ap.add_argument("--sweep-iters", type=int, default=40)
    ap.add_argument("--sweep-filter", default="", help="only points whose label contains this text")
    ap.add_argument("--packed-ab", action="store_true",
                    help="time the staged backward with packed f32x2 and with scalar fp32 arithmetic at the "
                         "wide-row shapes (bf16 16384x8192, fp32 16384x6144); one JSON line per variant")
    ap.add_argument("--ab-iters", type=int, default=50)
    ap.add_argument("--ab-reps", type=int, default=4)
    ap.add_argument("--profile-run", action="store_true",
                    help="warm-up and timed steps only (no host-enqueue, workspace-NULL, per-op split, e2e, "
                         "oracle or clock legs): a short program for ncu captures of the bench's kernels")
    return ap.parse_args()


# ------------------------------------------------------------- helpers --

def bytes_fwd(M, N, s):
    return 2 * M * N * s + N * s + 4 * M


def bytes_bwd_main(M, N, s, P):
    return 3 * M * N * s + N * s + 4 * M + 4 * P * N


def bytes_bwd_finalize(N, s, P):
    return 4 * P * N + N * s


def bytes_bwd(M, N, s, P):
    return 3 * M * N * s + 2 * N * s + 4 * M + 8 * P * N


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (x itself with one rank)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_rank_step per step and
    the step time is the slowest rank's."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the kernel sources' code: comments and blank space are dropped
    first, so that a change of wording alone keeps the stored counters."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_normalization_rmsnorm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8", errors="replace") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())
        h.update(f.encode() + text.encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    k = d.get("kernels", {}).get(kernel_key)
    return None if k is None else k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True, busy=None):
        """busy: optional callable that keeps the GPU working (one short,
        synchronised burst a call) while nvidia-smi starts, so the timed
        region does not begin on a GPU that sat idle meanwhile."""
        import tempfile
        self.index, self.proc, self.enabled, self.busy = index, None, enabled, busy
        self.busy_calls = 0
        self.path = os.path.join(tempfile.gettempdir(), f"rmsnorm_bench_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # the sampler's start-up (about 0.3 s) before the timed region
        t0 = time.time()
        while time.time() - t0 < 0.3:
            if self.busy is None:
                time.sleep(0.3)
                break
            self.busy()
            self.busy_calls += 1
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except OSError:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ CPU legs --

def oracle_sample(arrays, p, rows, nthreads):
    import oracle
    x = arrays["x"][:rows]
    dy = arrays["dy"][:rows]
    t0 = time.perf_counter()
    f = oracle.fwd(x, arrays["w"], dtype=p["dtype"], eps=p["eps"], offset=p["offset"], nthreads=nthreads)
    oracle.bwd(dy, x, arrays["w"], dtype=p["dtype"], eps=p["eps"], offset=p["offset"], rstd=f["rstd32"],
               nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(arrays, p, target_s=8.0, single_s=4.0):
    """The oracle on the host's cores (row-parallel, one thread a core) and
    on one thread, each on a bounded sample of the workload's rows."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    M, N = arrays["x"].shape
    s = 2 if p["dtype"] == "bf16" else 4
    t = oracle_sample(arrays, p, 64, cores)
    rows = int(min(M, max(64, 64 * target_s / max(t, 1e-3))))
    rows = max(cores, rows // cores * cores)
    t = oracle_sample(arrays, p, rows, cores)
    by = bytes_fwd(rows, N, s) + bytes_bwd(rows, N, s, 0)
    t1 = oracle_sample(arrays, p, 16, 1)
    rows1 = int(min(M, max(16, 16 * single_s / max(t1, 1e-3))))
    t1 = oracle_sample(arrays, p, rows1, 1)
    by1 = bytes_fwd(rows1, N, s) + bytes_bwd(rows1, N, s, 0)
    return {"value": by / t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {M} rows of the workload, fwd + bwd, fp64 C oracle, "
                      f"row-parallel on {cores} threads, {t:.2f} s wall",
            "single_thread": {"value": by1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"first {rows1} rows, one thread, {t1:.2f} s wall"}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from row_wise_normalization_rmsnorm_gb300 import inputs
    import oracle
    oracle.build()
    arrays, p = inputs.workload_inputs(WORKLOAD)
    M, N = arrays["x"].shape
    s = 2
    cores = os.cpu_count() or 1
    t1 = oracle_sample(arrays, p, cores, cores)
    # rows per step so that warmup + steps end within about a minute
    per_row = t1 / cores
    rows = int(max(1, min(512, 60.0 / max(1, args.steps + args.warmup) / max(per_row, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(arrays, p, rows, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(arrays, p, rows, cores)
    dt = time.perf_counter() - t0
    by = (bytes_fwd(rows, N, s) + bytes_bwd(rows, N, s, 0)) * args.steps
    val = by / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "M": M, "N": N, "rows_per_step": rows,
                   "eps": p["eps"], "offset": p["offset"]},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows per step of the {M}x{N} workload, fwd+bwd, fp64 C oracle"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------- GPU arm --

def sweep_points():
    """(label, dtype, M, N, fused, misaligned) of the shape sweep (N x M grid,
    N = 128 as per-head rows), the fused-add shapes and one misaligned case
    per dtype."""
    from row_wise_normalization_rmsnorm_gb300 import inputs
    pts = []
    for dt in ("bf16", "f32"):
        for M, N in inputs.sweep_points(dt):
            pts.append((f"{dt} {M}x{N}", dt, M, N, False, False))
    for M, N in ((4096, 4096), (1024, 8192), (4096, 16384)):
        pts.append((f"add bf16 {M}x{N}", "bf16", M, N, True, False))
    for M, N in ((16384, 8192), (4096, 8192), (16384, 16384)):
        pts.append((f"f16 {M}x{N}", "f16", M, N, False, False))
    pts.append(("nonaffine bf16 16384x8192", "bf16", 16384, 8192, False, False))
    pts.append(("nonaffine f32 16384x6144", "f32", 16384, 6144, False, False))
    # fp32 weight and dW beside 16-bit activations
    pts.append(("w32 bf16 16384x8192", "bf16", 16384, 8192, False, False))
    pts.append(("w32 f16 4096x8192", "f16", 4096, 8192, False, False))
    # E4M3 output of the forward (forward only)
    pts.append(("fp8row bf16 16384x8192", "bf16", 16384, 8192, False, False))
    pts.append(("fp8tensor bf16 16384x8192", "bf16", 16384, 8192, False, False))
    pts.append(("fp8row bf16 4096x4096", "bf16", 4096, 4096, False, False))
    pts.append(("fp8row bf16 8192x32768", "bf16", 8192, 32768, False, False))
    # LayerNorm (gamma and beta, dgamma and dbeta)
    for dt, M, N in (("bf16", 16384, 8192), ("bf16", 4096, 4096), ("bf16", 16384, 2048), ("f32", 16384, 4096),
                     ("bf16", 4096, 16384), ("bf16", 16384, 16384), ("bf16", 8192, 12288)):
        pts.append((f"ln {dt} {M}x{N}", dt, M, N, False, False))
    pts.append(("misaligned bf16 4096x7168", "bf16", 4096, 7168, False, True))
    pts.append(("misaligned f32 4096x2048", "f32", 4096, 2048, False, True))
    pts.append(("ln misaligned bf16 4096x7168", "bf16", 4096, 7168, False, True))
    # a row length that is no multiple of 16 bytes, and rows whose x and dy
    # sit at different addresses mod 16: the generic kernels
    pts.append(("oddn bf16 4096x7169", "bf16", 4096, 7169, False, False))
    pts.append(("skew bf16 4096x7168", "bf16", 4096, 7168, False, True))
    pts.append(("wide f32 16384x6144", "f32", 16384, 6144, False, False))
    # rows wider than one CTA's stages: a cluster of CTAs shares each row
    for M, N in ((16384, 20480), (8192, 32768), (2048, 65536)):
        pts.append((f"wide bf16 {M}x{N}", "bf16", M, N, False, False))
    pts.append(("ln bf16 4096x32768", "bf16", 4096, 32768, False, False))
    pts.append(("small f32 64x256", "f32", 64, 256, False, False))
    return pts


def run_sweep(args):
    """Per-call device time of fwd and bwd at every sweep point, two ways.
    Inputs are N(0,1) draws made on the device (timing only; parity uses the
    seeded host recipe).

    sustained: calls back to back, cycling over R sets of the call's arrays
      whose inputs together exceed three times the L2 size, so every call
      reads its inputs from HBM while the launches overlap as in a training
      step. The calls are captured once into a CUDA graph (programmatic
      dependencies included) and the graph replayed between one pair of
      events, so host-side call overhead cannot starve the GPU on short
      calls; us = elapsed / calls.
    isolated: before every call a buffer twice the L2 size is read (a sum),
      outside the event bracket, then one event pair brackets the call; the
      bracket itself costs what the empty-kernel line reports (launch and
      event overhead), which a short call cannot hide. (A read-based flush
      leaves clean lines: a write-based one would leave dirty lines whose
      write-back the timed call would pay for.)"""
    import torch
    from row_wise_normalization_rmsnorm_gb300 import build as rn_build
    rn_build.build()
    import row_wise_normalization_rmsnorm_gb300 as rn

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1005)

    def isolated(fn, iters):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            torch.sum(flush, 0, out=sink)
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        ts = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
        return ts[len(ts) // 2]

    def sustained(fn, R, iters):
        for i in range(2 * R):
            fn(i)
        torch.cuda.synchronize()
        K = 4 * R   # calls in the graph: every set four times
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(K):
                    fn(i)
        torch.cuda.current_stream().wait_stream(side)
        reps = max(1, -(-iters // K))
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        del graph
        return a.elapsed_time(b) * 1e3 / (K * reps)

    # the bracket's own cost: an empty kernel, and a forward of one 8-element row
    one = torch.zeros(1, device=dev)
    x1 = torch.ones(1, 8, device=dev, dtype=torch.bfloat16)
    w1 = torch.ones(8, device=dev, dtype=torch.bfloat16)
    print(json.dumps({"sweep": "bracket floor", "empty_kernel_us": round(isolated(lambda: one.add_(1.0), 40), 2),
                      "fwd_1x8_us": round(isolated(lambda: rn.rmsnorm_fwd(x1, w1), 40), 2)}), flush=True)

    for label, dt, M, N, fused, mis in sweep_points():
        if args.sweep_filter and args.sweep_filter not in label:
            continue
        td = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dt]
        s = 4 if dt == "f32" else 2
        off = 1 if mis else 0

        def mk(n, dtype=td, o=None):
            o = off if o is None else o
            buf = torch.randn(n + o, generator=g, device=dev, dtype=torch.float32).to(dtype)
            return buf[o:o + n]

        affine = not label.startswith("nonaffine")
        skew = label.startswith("skew")
        ln = label.startswith("ln ")
        fp8 = label.startswith("fp8")
        wtd = torch.float32 if label.startswith("w32") else td
        sw = 4 if wtd == torch.float32 else s
        w = mk(N, wtd)
        w.copy_(1 + 0.1 * torch.randn(N, generator=g, device=dev))
        dw = torch.empty_like(w)
        bvec = mk(N)
        bvec.mul_(0.1)
        dbv = torch.empty_like(bvec)
        if not affine:
            w, dw = None, None
        # sets of the per-call arrays, enough that their inputs exceed 3 x L2
        in_bytes = (2 + (1 if fused else 0)) * M * N * s
        R = max(2, -(-3 * l2 // in_bytes))

        def make_set():
            # skew: dy (and dx) one element further from a 16-byte boundary than x
            st = {"x": mk(M * N).view(M, N), "dy": mk(M * N, o=2 if skew else None).view(M, N),
                  "y": mk(M * N).view(M, N),
                  "dx": mk(M * N).view(M, N), "rstd": torch.empty(M, dtype=torch.float32, device=dev),
                  "mean": torch.empty(M, dtype=torch.float32, device=dev)}
            if fused:
                st["res"], st["hout"], st["dres"] = (mk(M * N).view(M, N) for _ in range(3))
            if fp8:
                st["yq"] = torch.empty((M, N), dtype=torch.uint8, device=dev)
                st["sinv"] = torch.empty(M, dtype=torch.float32, device=dev)
            return st
        sets = [make_set() for _ in range(R)]
        code = rn.TORCH_DTYPE[td] | (rn.RMSNORM_WEIGHT_F32 if sw != s else 0)
        nb = rn.rmsnorm_bwd_workspace_bytes(M, N, code)
        if ln:
            nb = rn.layernorm_bwd_workspace_bytes(M, N, td)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        sc = torch.tensor([2.0], dtype=torch.float32, device=dev)
        row = label.startswith("fp8row")

        def fwd(i):
            t = sets[i % R]
            if ln:
                return rn.layernorm_fwd(t["x"], w, bvec, y=t["y"], mean=t["mean"], rstd=t["rstd"])["plan"]
            if fp8:
                return rn.rmsnorm_fwd_fp8(t["x"], w, scaling="row" if row else "tensor", scale=None if row else sc,
                                          y=t["yq"], rstd=t["rstd"], scale_inv=t["sinv"] if row else t["sinv"][:1])[
                    "plan"]
            if fused:
                rn.rmsnorm_add_fwd(t["x"], t["res"], w, y=t["y"], residual_out=t["hout"], rstd=t["rstd"])
            else:
                rn.rmsnorm_fwd(t["x"], w, y=t["y"], rstd=t["rstd"])
            return None

        def bwd(i):
            t = sets[i % R]
            if ln:
                return rn.layernorm_bwd(t["dy"], t["x"], w, t["mean"], t["rstd"], dx=t["dx"], dgamma=dw, dbeta=dbv,
                                        workspace=ws)["plan"]
            if fused:
                rn.rmsnorm_add_bwd(t["dy"], t["dres"], t["hout"], w, t["rstd"], dx=t["dx"], dw=dw, workspace=ws)
            else:
                rn.rmsnorm_bwd(t["dy"], t["x"], w, t["rstd"], dx=t["dx"], dw=dw, workspace=ws)
            return None

        t0 = sets[0]
        if ln:
            fplan, bplan = fwd(0), bwd(0)
        elif fp8:
            fplan, bplan = fwd(0), None
        else:
            _, _, _, fplan = rn.rmsnorm_fwd_ex(t0["x"], w, residual=t0.get("res"), residual_out=t0.get("hout"),
                                               y=t0["y"], rstd=t0["rstd"])
            _, _, bplan = rn.rmsnorm_bwd_ex(t0["dy"], t0["hout"] if fused else t0["x"], w, t0["rstd"],
                                            dresidual_out=t0.get("dres"), fused=fused, dx=t0["dx"], dw=dw,
                                            workspace=ws)
        P = bplan["ws_rows"] if bplan else 0   # partial rows (a cluster shares one)
        k = 1 if fused else 0
        wb = 1 if affine else 0   # the weight, dW and the workspace exist only with a weight
        by = {"fwd": (2 + 2 * k) * M * N * s + wb * N * sw + 4 * M,
              "bwd": (3 + k) * M * N * s + wb * (2 * N * sw + 8 * P * N) + 4 * M}
        if ln:
            # LayerNorm: forward reads x, gamma, beta and writes y, mean, rstd;
            # backward reads dy, x, gamma, mean, rstd, writes dx, and moves
            # the [P, 2N] partial rows and dgamma, dbeta
            by["fwd"] = 2 * M * N * s + 2 * N * s + 8 * M
            by["bwd"] = 3 * M * N * s + N * s + 8 * M + 2 * (8 * P * N) + 2 * N * s
        if fp8:
            # reads x and w, writes one byte per element, rstd and (per row) 1/s
            by["fwd"] = M * N * s + N * s + M * N + 4 * M + (4 * M if row else 0)
        ops = (("fwd", fwd, fplan),) if fp8 else (("fwd", fwd, fplan), ("bwd", bwd, bplan))
        for op, fn, plan in ops:
            us = sustained(fn, R, args.sweep_iters)
            iso = isolated(lambda: fn(0), args.sweep_iters)
            gbs = by[op] / us / 1e3
            print(json.dumps({"sweep": label, "op": op, "dtype": dt, "M": M, "N": N, "fused": fused,
                              "misaligned": mis, "us": round(us, 2), "gbs": round(gbs, 1),
                              "frac_of_peak": round(gbs / peak, 4), "us_isolated": round(iso, 2),
                              "frac_isolated": round(by[op] / iso / 1e3 / peak, 4), "buffer_sets": R,
                              "peak": peak, "peak_source": peak_kind,
                              "plan": plan["plan_id"], "path": plan["path_name"], "peel": plan.get("peel", 0),
                              "ctas": plan["ctas"], "bytes": by[op]}), flush=True)
        del sets, ws, w, dw, dbv
        torch.cuda.empty_cache()
    return 0


def run_packed_ab(args):
    """The staged backward's two arithmetic variants (same plan, same CTA
    count, bit-identical results) timed back to back on the wide-row shapes
    where the packed f32x2 math was credited with speeding up an issue-bound
    kernel, inputs larger than L2, K calls between one pair of events,
    alternating variants in blocks so clock drift affects both alike."""
    import torch
    from row_wise_normalization_rmsnorm_gb300 import build as rn_build
    rn_build.build()
    import row_wise_normalization_rmsnorm_gb300 as rn
    dev = torch.device("cuda", 0)
    peak, peak_kind = peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(1006)
    for dt, M, N in (("bf16", 16384, 8192), ("f32", 16384, 6144)):
        td = torch.bfloat16 if dt == "bf16" else torch.float32
        s = 2 if dt == "bf16" else 4
        x, dy, dx = (torch.randn(M, N, generator=g, device=dev).to(td) for _ in range(3))
        w = (1 + 0.1 * torch.randn(N, generator=g, device=dev)).to(td)
        dw = torch.empty_like(w)
        _, rstd = rn.rmsnorm_fwd(x, w)
        ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, N, td), dtype=torch.uint8, device=dev)
        times = {0: [], 1: []}
        plans = {}
        for rep in range(args.ab_reps):
            for pk in (1, 0):
                for _ in range(3):
                    _, _, plans[pk] = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx, dw=dw, workspace=ws, force_packed=pk)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(args.ab_iters):
                    rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx, dw=dw, workspace=ws, force_packed=pk)
                b.record()
                torch.cuda.synchronize()
                times[pk].append(a.elapsed_time(b) * 1e3 / args.ab_iters)
        P = plans[1]["ws_rows"]
        by = bytes_bwd(M, N, s, P)
        for pk in (1, 0):
            us = statistics.median(times[pk])
            print(json.dumps({"packed_ab": f"{dt} {M}x{N}", "packed": pk, "us": round(us, 2),
                              "gbs": round(by / us / 1e3, 1), "frac_of_peak": round(by / us / 1e3 / peak, 4),
                              "plan": plans[pk]["plan_id"], "ctas": plans[pk]["ctas"],
                              "variant_packed": plans[pk]["packed"], "peak_source": peak_kind}), flush=True)
        del x, dy, dx, ws
        torch.cuda.empty_cache()
    return 0


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.packed_ab:
        return run_packed_ab(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from row_wise_normalization_rmsnorm_gb300 import build as rn_build
    rn_build.build()
    import row_wise_normalization_rmsnorm_gb300 as rn
    from row_wise_normalization_rmsnorm_gb300 import inputs

    arrays, p = inputs.workload_inputs(WORKLOAD)
    M, N, eps = p["M"], p["N"], p["eps"]
    s = 2

    def up(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    x, dy, w = up(arrays["x"]), up(arrays["dy"]), up(arrays["w"])
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    ws_bytes = rn.rmsnorm_bwd_workspace_bytes(M, N, torch.bfloat16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    _, _, _, fplan = rn.rmsnorm_fwd_ex(x, w, y=y, rstd=rstd, eps=eps)
    _, _, bplan = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx, dw=dw, workspace=ws, eps=eps)
    P = bplan["ws_rows"]   # partial rows (a cluster shares one)

    K, W = args.steps, args.warmup
    # per-op split, measured outside the timed region: an event between two
    # kernels also ends the programmatic dependency between them
    nsplit = K
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nsplit)]
    # torch creates an event on its first record(); materialise them up front
    for e in ev:
        for q in e:
            q.record(stream)
    torch.cuda.synchronize()

    def step(e=None, mid=None):
        if e is not None:
            e[0].record(stream)
        rn.rmsnorm_fwd(x, w, y=y, rstd=rstd, eps=eps)
        if e is not None:
            e[1].record(stream)
        rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx, dw=dw, workspace=ws, eps=eps, event_after_main=mid)
        if e is not None:
            e[2].record(stream)

    # While the clock sampler starts, the GPU keeps running the step in
    # bursts of 20 (each synchronised, so the launch queue never runs far
    # ahead): the W warm-up steps and the timed ones then follow a busy GPU,
    # not one left idle for the sampler's 0.3 s start-up (which cost a
    # 20-step run about 3% against a 200-step one). Counted in the JSON line.
    def preheat():
        for _ in range(20):
            step()
        torch.cuda.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, enabled=not (args.no_clocks or args.profile_run), busy=preheat) as clk:
        for _ in range(W):
            step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        start.record(stream)
        for i in range(K):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), dist if world > 1 else None, dev)
    if args.profile_run:
        if rank == 0:
            print(json.dumps({"profile_run": WORKLOAD_DESC, "steps": K, "ms_per_step": total_ms / K,
                              "gpu_launches": 3 * K}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return 0
    for i in range(nsplit):
        step(ev[i])
    torch.cuda.synchronize()
    t_fwd = [e[0].elapsed_time(e[1]) for e in ev]
    t_bwd = [e[1].elapsed_time(e[2]) for e in ev]
    ms_per_step = total_ms / K
    step_bytes = bytes_fwd(M, N, s) + bytes_bwd(M, N, s, P)
    value = whole_job_gbs(step_bytes, world, ms_per_step)

    # Diagnostic split of the backward into its two kernels, outside the
    # timed region: an event between them serialises the finalizer's launch.
    nd = min(K, 50)
    dg = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nd)]
    for e in dg:
        for q in e:
            q.record(stream)
    torch.cuda.synchronize()
    for i in range(nd):
        step(None)
        dg[i][0].record(stream)
        rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx, dw=dw, workspace=ws, eps=eps, event_after_main=dg[i][1])
        dg[i][2].record(stream)
    torch.cuda.synchronize()
    t_main = [e[0].elapsed_time(e[1]) for e in dg]
    t_fin = [e[1].elapsed_time(e[2]) for e in dg]

    # Host cost of one ABI call (the wall time of enqueueing it, the
    # counterpart of the per-call host cost the direct-call launch path was
    # built to cut): ctypes calls with the arguments marshalled once, in
    # bursts of 50 followed by a synchronize so the launch queue never fills
    # (a full queue would make the call wait for the GPU); median per call.
    L = rn.lib()
    hs = stream.cuda_stream
    fargs = (x.data_ptr(), w.data_ptr(), y.data_ptr(), rstd.data_ptr(), M, N, 1, eps, 0.0, hs)
    bargs = (dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), dx.data_ptr(), dw.data_ptr(),
             ws.data_ptr(), ws_bytes, M, N, 1, eps, 0.0, hs)
    host = {}
    for name, fn, cargs in (("fwd", L.rmsnorm_fwd, fargs), ("bwd", L.rmsnorm_bwd, bargs)):
        per = []
        for _ in range(20):
            torch.cuda.synchronize()
            for _ in range(50):
                t0 = time.perf_counter_ns()
                st = fn(*cargs)
                per.append((time.perf_counter_ns() - t0) / 1e3)
                assert st == 0, st
        torch.cuda.synchronize()
        host[name] = {"median_us": statistics.median(per), "p90_us": sorted(per)[int(0.9 * len(per))],
                      "calls": len(per)}
    host["how"] = ("wall time of the ctypes call into the C ABI, arguments marshalled once, "
                   "bursts of 50 calls between synchronizes, median over 1000 calls")

    # The backward with workspace NULL: the library takes stream-ordered
    # memory (cudaMallocAsync / cudaFreeAsync on the stream) inside the call,
    # so the allocation is inside the timed bracket.
    nn = min(K, 200)
    en = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nn)]
    for a, b in en:
        a.record(stream)
        b.record(stream)
    for _ in range(3):
        rn.rmsnorm_bwd(dy, x, w, rstd, dx=dx, dw=dw, workspace=None, eps=eps)
    torch.cuda.synchronize()
    for a, b in en:
        a.record(stream)
        rn.rmsnorm_bwd(dy, x, w, rstd, dx=dx, dw=dw, workspace=None, eps=eps)
        b.record(stream)
    torch.cuda.synchronize()
    t_null = [a.elapsed_time(b) for a, b in en]

    peak, peak_kind = peaks()
    comp = {}
    for name, ts, by in (("fwd", t_fwd, bytes_fwd(M, N, s)), ("bwd", t_bwd, bytes_bwd(M, N, s, P)),
                         ("bwd_workspace_null", t_null, bytes_bwd(M, N, s, P)),
                         ("bwd_main_serialised", t_main, bytes_bwd_main(M, N, s, P)),
                         ("bwd_finalize_serialised", t_fin, bytes_bwd_finalize(N, s, P))):
        avg = sum(ts) / len(ts)
        comp[name] = {"us": avg * 1e3, "median_us": statistics.median(ts) * 1e3, "bytes": by,
                      "gbs": by / (avg * 1e-3) / 1e9, "frac_of_peak": by / (avg * 1e-3) / 1e9 / peak}
    comp["bwd"]["kernels"] = "main + finalizer (programmatic dependent launch)"
    comp["split_how"] = ("fwd and bwd each between their own events in steps run after the timed region "
                         "(events between kernels end the programmatic dependency, so the split sums to "
                         "more than ms_per_step)")
    comp["bwd_workspace_null"]["kernels"] = ("main + finalizer, workspace NULL: stream-ordered allocation "
                                             "and free inside the call")
    dom = "bwd" if comp["bwd"]["us"] >= comp["fwd"]["us"] else "fwd"
    bwd_main = {"staged": "rmsnorm_bwd_staged", "vector": "rmsnorm_bwd_vector"}.get(bplan["path_name"],
                                                                                   "rmsnorm_bwd_generic")
    kname = {"fwd": "rmsnorm_fwd_vector", "bwd": bwd_main + " + rmsnorm_dw_finalize4"}[dom]
    roof = {"kernel": kname, "bound": "hbm", "achieved": comp[dom]["gbs"], "peak": peak, "unit": "GB/s",
            "frac": comp[dom]["gbs"] / peak, "traffic": ncu_traffic(dom), "peak_source": peak_kind,
            "bytes_per_launch": comp[dom]["bytes"]}

    # end to end: pinned host buffers, copies inside the timed region. Steps
    # are independent batches, so they are pipelined over two sets of device
    # buffers: step k+1's host-to-device copies (one stream) and step k-1's
    # device-to-host copies (another) run while step k computes; events
    # order each buffer's reuse, and the timed region brackets every copy.
    # (Splitting a direction's copies over more streams measured no faster:
    # the host link is the limit, about 165 GB/s each way with both busy.)
    h_x = torch.empty_like(x, device="cpu").pin_memory()
    h_dy = torch.empty_like(dy, device="cpu").pin_memory()
    h_w = torch.empty_like(w, device="cpu").pin_memory()
    h_x.copy_(x.cpu())
    h_dy.copy_(dy.cpu())
    h_w.copy_(w.cpu())
    o_y = torch.empty_like(y, device="cpu").pin_memory()
    o_dx = torch.empty_like(dx, device="cpu").pin_memory()
    o_dw = torch.empty_like(dw, device="cpu").pin_memory()
    o_r = torch.empty_like(rstd, device="cpu").pin_memory()
    bufs = [dict(x=torch.empty_like(x), dy=torch.empty_like(dy), w=torch.empty_like(w), y=torch.empty_like(y),
                 r=torch.empty_like(rstd), dx=torch.empty_like(dx), dw=torch.empty_like(dw),
                 ws=torch.empty_like(ws), loaded=torch.cuda.Event(), computed=torch.cuda.Event(),
                 drained=torch.cuda.Event()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    for bf in bufs:  # every buffer starts free
        bf["computed"].record(stream)
        bf["drained"].record(stream)

    def e2e_step(k):
        bf = bufs[k % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(bf["computed"])   # the last kernels that read this buffer's inputs
            bf["x"].copy_(h_x, non_blocking=True)
            bf["dy"].copy_(h_dy, non_blocking=True)
            bf["w"].copy_(h_w, non_blocking=True)
            bf["loaded"].record(s_in)
        stream.wait_event(bf["loaded"])
        stream.wait_event(bf["drained"])      # the last copies out of this buffer's outputs
        rn.rmsnorm_fwd(bf["x"], bf["w"], y=bf["y"], rstd=bf["r"], eps=eps)
        rn.rmsnorm_bwd(bf["dy"], bf["x"], bf["w"], bf["r"], dx=bf["dx"], dw=bf["dw"], workspace=bf["ws"], eps=eps)
        bf["computed"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(bf["computed"])
            o_y.copy_(bf["y"], non_blocking=True)
            o_r.copy_(bf["r"], non_blocking=True)
            o_dx.copy_(bf["dx"], non_blocking=True)
            o_dw.copy_(bf["dw"], non_blocking=True)
            bf["drained"].record(s_out)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for k in range(args.e2e_steps):
        e2e_step(k)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dist if world > 1 else None, dev)
    h2d = (h_x.numel() + h_dy.numel() + h_w.numel()) * s
    d2h = (o_y.numel() + o_dx.numel() + o_dw.numel()) * s + o_r.numel() * 4
    e2e = {"value": whole_job_gbs(step_bytes, world, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "preheat_steps": 20 * clk.busy_calls,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "M": M, "N": N, "per_rank_rows": M,
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "inputs larger than L2 (268 MB per tensor, 126 MB L2); no flush",
                   "fwd_plan": fplan["plan_id"], "bwd_plan": bplan["plan_id"], "bwd_ctas": P,
                   "workspace_bytes": ws_bytes},
        "frac_of_peak": value / world / peak,
        "components": comp,
        "host_enqueue": host,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(arrays, p)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
