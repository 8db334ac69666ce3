#!/usr/bin/env python
"""Benchmark: forward + backward of the weighted sum and the scaled SiLU.

One step is one pass of the whole hot path over the synthetic workloads:

    silu_fwd(c2)  ws_fwd(c3) ws_fwd(c4) ws_fwd(c5)       forwards
    ws_bwd(c5)    ws_bwd(c4) ws_bwd(c3) silu_bwd(c2)     backwards, reverse order

(c2: scaled SiLU, fp16 x[8192,4096]; c3: bf16 x[1048576,1024];
c4: fp16 x[16777216,64]; c5: fp32 x[4096,65536]).  Every input is larger
than L2 or is separated from its reuse by gigabytes of other traffic, as in a
real network where a layer's backward runs long after its forward.

The metric is effective HBM bandwidth: the algorithmic bytes the method must
move (fwd: read x and w, write y; bwd: read x, dy and w, write dx and the
parameter gradient) divided by device time.  `value` is measured with CUDA
events around K steps on resident inputs; `e2e` runs the same step through
the public API with host buffers: every step copies its inputs from pinned
host memory and its result (the parameter gradients) back, inside the timed
region (`e2e.all_outputs`: y and dx copied back as well).

The worked 100 x 64 example (c1, 32-row tiles) is latency-bound: it is timed
alone, outside the step (device time per op from CUDA graphs, and the host's
call-to-result latency), and reported beside the isolated per-op table.
`cpu_baseline` times the fp64 oracle per workload and per op on the host's
cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]
       [--workload all|c1,c2,c3,c4,c5,...]
Under torchrun each rank runs its own replica of the workload (weak scaling,
no collective on the data path); rank 0 prints one JSON line.
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

METRIC = "fwd+bwd effective HBM GB/s and % of GB300 peak; elements/s per op"
ORDER_FWD = ["c2", "c3", "c4", "c5"]
ORDER_BWD = ["c5", "c4", "c3", "c2"]
KERNELS_PER_OP = {"ws_fwd": 1, "ws_bwd": 2, "silu_fwd": 1, "silu_bwd": 2, "softmax_fwd": 1,
                  "softmax_bwd": 1, "rmsnorm_fwd": 1, "rmsnorm_bwd": 2, "layernorm_fwd": 1,
                  "layernorm_bwd": 2}
EXTRA = ["s1", "n1", "n2", "s2", "n3", "n4", "s3", "s4"]  # measured only when named
LATENCY = ["c1"]  # latency-bound: timed alone, outside the step
NORMS = ("rmsnorm", "layernorm")


# ------------------------------------------------------------------ byte model
def elt_size(dt: str) -> int:
    return 4 if dt == "f32" else 2


def op_bytes(wl, op: str, rows: int | None = None) -> int:
    """Algorithmic bytes of one op on workload wl (optionally on `rows` rows)."""
    N = wl.N if rows is None else rows
    es = elt_size(wl.dtype)
    if wl.op == "ws":
        D = wl.D
        if op == "fwd":
            return N * D * es + D * 4 + N * es
        return 2 * N * D * es + N * es + 2 * D * 4
    n = N * wl.D
    if wl.op == "softmax":
        return 2 * n * es if op == "fwd" else 3 * n * es
    if wl.op in NORMS:
        # x (and dy) read, y (dx) written; w (and b) read, grad_w (and grad_b)
        # written once; the backward's per-tile partials are not counted
        params = 4 * wl.D * (2 if wl.op == "layernorm" else 1)
        return 2 * n * es + params if op == "fwd" else 3 * n * es + 4 * wl.D + params
    return 2 * n * es + 4 if op == "fwd" else 3 * n * es + 8


def op_elems(wl, rows: int | None = None) -> int:
    return (wl.N if rows is None else rows) * wl.D


def steps_ops(names):
    fwd = [(n, "fwd") for n in ORDER_FWD + EXTRA if n in names]
    bwd = [(n, "bwd") for n in ORDER_BWD + EXTRA if n in names]
    return fwd + bwd


def op_name(wl, op):
    return f"{wl.op}_{op}"


# ------------------------------------------------------------------ helpers
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
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
            out = ""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(v: float, device=None) -> float:
    """Maximum of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU (oracle) leg
def oracle_sample(names, frac: float):
    """Host inputs for a bounded sample of each workload: the first
    max(1, round(N·frac)) rows (for the scaled SiLU, rows of the [8192, 4096]
    tensor)."""
    from inputgen.workloads import WORKLOADS
    return oracle_sample_wl([(WORKLOADS[n], max(1, int(round(WORKLOADS[n].N * frac))))
                             for n in names])


def oracle_sample_wl(pairs):
    """Host inputs of the first `rows` rows of each (workload, rows) pair."""
    import torch
    import inputgen
    samples = []
    for wl, rows in pairs:
        x = inputgen.make((rows, wl.D), wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0)
        if wl.op == "ws":
            w = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1)
            dy = inputgen.make((rows,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
        elif wl.op == "softmax":
            w = None
            dy = inputgen.make((rows, wl.D), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
        elif wl.op in NORMS:
            w = [inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1),
                 inputgen.make((wl.D,), "f32", wl.b.kind, wl.b.a, wl.b.b, 0, 3)
                 if wl.b is not None else None]
            dy = inputgen.make((rows, wl.D), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
        else:
            w = torch.tensor([wl.w_scalar], dtype=torch.float32)
            dy = inputgen.make((rows, wl.D), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2)
        samples.append((wl, rows, x, w, dy))
    return samples


def oracle_step(samples):
    import oracle
    nbytes = 0
    for wl, rows, x, w, dy in samples:
        if wl.op == "ws":
            oracle.ws_fwd(x, w)
            oracle.ws_bwd(x, w, dy)
        elif wl.op == "softmax":
            _, y = oracle.softmax_fwd(x)
            oracle.softmax_bwd(y, dy)
        elif wl.op in NORMS:
            layer = wl.op == "layernorm"
            oracle.norm_fwd(x, w[0], w[1], wl.eps, layer)
            oracle.norm_bwd(x, w[0], dy, wl.eps, layer)
        else:
            oracle.silu_fwd(x.reshape(-1), wl.w_scalar)
            oracle.silu_bwd(dy.reshape(-1), x.reshape(-1), wl.w_scalar)
        nbytes += op_bytes(wl, "fwd", rows) + op_bytes(wl, "bwd", rows)
    return nbytes


def sample_desc(samples):
    return ", ".join(f"{wl.name}: first {rows} of {wl.N} rows" for wl, rows, *_ in samples)


def calibrated_fraction(names, budget_s: float, max_frac: float = 1 / 16):
    """Largest row fraction (<= max_frac) whose oracle step takes about budget_s."""
    f0 = 1 / 4096
    s = oracle_sample(names, f0)
    t = time.perf_counter()
    oracle_step(s)
    dt = max(time.perf_counter() - t, 1e-4)
    return max(f0, min(max_frac, f0 * budget_s / dt))


def _time_repeated(fn, budget_s: float) -> float:
    """Mean seconds of one call of fn, repeated until budget_s have passed."""
    reps = 0
    t = time.perf_counter()
    while reps == 0 or time.perf_counter() - t < budget_s:
        fn()
        reps += 1
    return (time.perf_counter() - t) / reps


def oracle_ops(wl, rows):
    """The oracle's forward and backward of the first `rows` rows of wl (host
    inputs generated here, outside any timing), as two callables."""
    import oracle
    (_, _, x, w, dy), = oracle_sample_wl([(wl, rows)])
    if wl.op == "ws":
        return (lambda: oracle.ws_fwd(x, w)), (lambda: oracle.ws_bwd(x, w, dy))
    if wl.op == "softmax":
        _, y = oracle.softmax_fwd(x)
        return (lambda: oracle.softmax_fwd(x)), (lambda: oracle.softmax_bwd(y, dy))
    if wl.op in NORMS:
        layer = wl.op == "layernorm"
        return (lambda: oracle.norm_fwd(x, w[0], w[1], wl.eps, layer),
                lambda: oracle.norm_bwd(x, w[0], dy, wl.eps, layer))
    xf, gf = x.reshape(-1), dy.reshape(-1)
    return (lambda: oracle.silu_fwd(xf, wl.w_scalar)), (lambda: oracle.silu_bwd(gf, xf, wl.w_scalar))


def cpu_baseline(names, per_op_budget_s: float = 0.4):
    """The oracle on this host, per workload and per op: forward, backward and
    fwd+bwd as effective bytes/s and elements/s, on all cores (OpenMP) and on
    one.  Each workload runs on a bounded sample (its first rows: at most a
    sixteenth of a large workload, sized so that an op takes ~per_op_budget_s
    on all cores), every op repeated for ~per_op_budget_s.  `value` is the
    sum of the sampled bytes over the sum of the times on all cores."""
    import oracle
    from inputgen.workloads import WORKLOADS
    oracle.build()
    cores = oracle.threads()
    per_op, desc = {}, []
    tot = {"all": [0, 0.0], "one": [0, 0.0]}
    for n in names:
        wl = WORKLOADS[n]
        cap = wl.N if wl.N <= 1600 else wl.N // 16
        rows0 = max(1, min(cap, wl.N // 4096))
        fwd, bwd = oracle_ops(wl, rows0)
        t0 = time.perf_counter()
        fwd()
        bwd()
        t0 = max(time.perf_counter() - t0, 1e-5)
        rows = max(1, min(cap, int(rows0 * 2 * per_op_budget_s / t0)))
        fwd, bwd = oracle_ops(wl, rows) if rows != rows0 else (fwd, bwd)
        bf, bb, el = op_bytes(wl, "fwd", rows), op_bytes(wl, "bwd", rows), op_elems(wl, rows)
        for label, threads in (("all", cores), ("one", 1)):
            old = oracle.set_threads(threads)
            try:
                tf = _time_repeated(fwd, per_op_budget_s)
                tb = _time_repeated(bwd, per_op_budget_s)
            finally:
                oracle.set_threads(old)
            sfx = "" if label == "all" else "_1core"
            for op, b, t in (("fwd", bf, tf), ("bwd", bb, tb), ("fwd+bwd", bf + bb, tf + tb)):
                row = per_op.setdefault(f"{n}.{op}", {})
                row["GB/s" + sfx] = round(b / t / 1e9, 4)
                row["elements_per_s" + sfx] = round(el / t, 1)
            tot[label][0] += bf + bb
            tot[label][1] += tf + tb
        desc.append(f"{n}: first {rows} of {wl.N} rows")
    return {"value": round(tot["all"][0] / tot["all"][1] / 1e9, 4), "unit": "GB/s",
            "cores": cores, "kind": "oracle",
            "sample": ", ".join(desc) + f"; each op repeated for ~{per_op_budget_s} s on "
                      f"{cores} threads and on 1 (fp64 CPU work)",
            "single_thread": {"value": round(tot["one"][0] / tot["one"][1] / 1e9, 4),
                              "unit": "GB/s", "cores": 1},
            "per_op": per_op}


def run_reference(args, names):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.threads()
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    frac = calibrated_fraction(names, budget_s=budget)
    samples = oracle_sample(names, frac)
    for _ in range(args.warmup):
        oracle_step(samples)
    nbytes = 0
    t = time.perf_counter()
    for _ in range(args.steps):
        nbytes += oracle_step(samples)
    dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": workload_label(names) + (f" (rows x {args.scale})"
                                                             if args.scale != 1.0 else ""), "reference": "fp64 CPU oracle"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample_desc(samples)},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


EXTRA_LABELS = {"s1": "row softmax s1 (bf16 x[65536,4096])",
                "n1": "RMSNorm n1 (bf16 x[65536,4096])",
                "n2": "LayerNorm n2 (bf16 x[65536,4096])",
                "s2": "row softmax s2 (bf16 x[4096,131072])",
                "n3": "RMSNorm n3 (bf16 x[16384,16384])",
                "n4": "LayerNorm n4 (bf16 x[16384,16384])",
                "s3": "row softmax s3 (bf16 x[8192,50257])",
                "s4": "row softmax s4 (fp32 x[2048,262144])"}


def workload_label(names):
    if all(n in EXTRA for n in names):
        return " + ".join(EXTRA_LABELS[n] for n in names) + ", fwd+bwd"
    return ("weighted sum " + "+".join(n for n in ["c3", "c4", "c5"] if n in names) +
            (" and " if "c2" in names and len(names) > 1 else "") +
            ("scaled-SiLU c2" if "c2" in names else "") + ", fwd+bwd")


# ------------------------------------------------------------------ GPU leg
class Buffers:
    """Device tensors of one workload (inputs resident, outputs, workspace)
    plus, for e2e, pinned host copies of inputs and outputs."""

    def __init__(self, wl, dev, wsf, host_io: bool):
        import torch
        import inputgen
        self.wl = wl
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
        shape = (wl.N, wl.D)
        self.hx = inputgen.make(shape, wl.dtype, wl.x.kind, wl.x.a, wl.x.b, 0, 0, pin=host_io)
        if wl.op == "ws":
            self.hw = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1, pin=host_io)
            self.hdy = inputgen.make((wl.N,), wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2,
                                     pin=host_io)
        elif wl.op == "softmax":
            self.hw = torch.zeros(1, dtype=torch.float32)
            self.hdy = inputgen.make(shape, wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2,
                                     pin=host_io)
        elif wl.op in NORMS:
            self.hw = inputgen.make((wl.D,), "f32", wl.w.kind, wl.w.a, wl.w.b, 0, 1, pin=host_io)
            if wl.b is not None:
                self.hb = inputgen.make((wl.D,), "f32", wl.b.kind, wl.b.a, wl.b.b, 0, 3,
                                        pin=host_io)
            self.hdy = inputgen.make(shape, wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2,
                                     pin=host_io)
        else:
            self.hw = torch.tensor([wl.w_scalar], dtype=torch.float32)
            if host_io:
                self.hw = self.hw.pin_memory()
            self.hdy = inputgen.make(shape, wl.dtype, wl.dy.kind, wl.dy.a, wl.dy.b, 0, 2,
                                     pin=host_io)
        self.x = self.hx.to(dev)
        self.w = self.hw.to(dev)
        self.dy = self.hdy.to(dev)
        self.hb = getattr(self, "hb", None)
        self.b = self.hb.to(dev) if self.hb is not None else None
        self.gb = None
        if wl.op == "ws":
            self.y = torch.empty(wl.N, dtype=tdt, device=dev)
            self.gw = torch.empty(wl.D, dtype=torch.float32, device=dev)
            nbytes = wsf.ws_bwd_workspace_bytes(wl.N, wl.D, tdt, wl.block_n)
        elif wl.op == "softmax":
            self.y = torch.empty(shape, dtype=tdt, device=dev)
            self.gw = torch.zeros(1, dtype=torch.float32, device=dev)
            nbytes = 0
        elif wl.op in NORMS:
            layer = wl.op == "layernorm"
            self.y = torch.empty(shape, dtype=tdt, device=dev)
            self.gw = torch.empty(wl.D, dtype=torch.float32, device=dev)
            self.gb = torch.empty(wl.D, dtype=torch.float32, device=dev) if layer else None
            nbytes = wsf.norm_bwd_workspace_bytes(wl.N, wl.D, tdt, layer)
        else:
            self.y = torch.empty(shape, dtype=tdt, device=dev)
            self.gw = torch.empty(1, dtype=torch.float32, device=dev)
            nbytes = wsf.silu_bwd_workspace_bytes(wl.N * wl.D, tdt)
        self.dx = torch.empty(shape, dtype=tdt, device=dev)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        if host_io:
            self.hy = torch.empty(self.y.shape, dtype=tdt, pin_memory=True)
            self.hdx = torch.empty(shape, dtype=tdt, pin_memory=True)
            self.hgw = torch.empty(self.gw.shape, dtype=torch.float32, pin_memory=True)
            self.hgb = (torch.empty(self.gb.shape, dtype=torch.float32, pin_memory=True)
                        if self.gb is not None else None)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in (self.hx, self.hw, self.hdy, self.hb)
                   if t is not None)

    def d2h_bytes(self, all_outputs=False):
        outs = (self.y, self.dx, self.gw, self.gb) if all_outputs else (self.gw, self.gb)
        return sum(t.numel() * t.element_size() for t in outs if t is not None)

    def norm(self, wsf, op, x, y, dy, dx, accumulate=False, stream=None):
        eps = self.wl.eps
        if self.wl.op == "layernorm":
            if op == "fwd":
                wsf.layernorm_fwd(x, self.w, self.b, eps, y=y, stream=stream)
            else:
                wsf.layernorm_bwd(x, self.w, dy, eps, dx=dx, grad_w=self.gw, grad_b=self.gb,
                                  accumulate=accumulate, workspace=self.ws, stream=stream)
        elif op == "fwd":
            wsf.rmsnorm_fwd(x, self.w, eps, y=y, stream=stream)
        else:
            wsf.rmsnorm_bwd(x, self.w, dy, eps, dx=dx, grad_w=self.gw, accumulate=accumulate,
                            workspace=self.ws, stream=stream)

    def run_rows(self, wsf, r0, r1, accumulate, stream):
        """Forward and backward of rows [r0, r1) (for the scaled SiLU, rows of
        the [N, D] view), the parameter gradient accumulated when asked."""
        x, dy, y, dx = self.x[r0:r1], self.dy[r0:r1], self.y[r0:r1], self.dx[r0:r1]
        if self.wl.op == "softmax":
            wsf.softmax_fwd(x, y=y, stream=stream)
            wsf.softmax_bwd(y, dy, dx=dx, stream=stream)
        elif self.wl.op in NORMS:
            self.norm(wsf, "fwd", x, y, dy, dx, stream=stream)
            self.norm(wsf, "bwd", x, y, dy, dx, accumulate=accumulate, stream=stream)
        elif self.wl.op == "ws":
            wsf.ws_fwd(x, self.w, y=y, stream=stream)
            wsf.ws_bwd(x, self.w, dy, dx=dx, grad_w=self.gw, accumulate=accumulate,
                       workspace=self.ws, block_n=self.wl.block_n, stream=stream)
        else:
            wsf.silu_fwd(x, self.w, y=y, stream=stream)
            wsf.silu_bwd(dy, x, self.w, dx=dx, dw=self.gw, accumulate=accumulate,
                         workspace=self.ws, stream=stream)

    def run(self, wsf, op):
        if self.wl.op in NORMS:
            self.norm(wsf, op, self.x, self.y, self.dy, self.dx)
        elif self.wl.op == "softmax":
            if op == "fwd":
                wsf.softmax_fwd(self.x, y=self.y)
            else:
                wsf.softmax_bwd(self.y, self.dy, dx=self.dx)
        elif self.wl.op == "ws":
            if op == "fwd":
                wsf.ws_fwd(self.x, self.w, y=self.y)
            else:
                wsf.ws_bwd(self.x, self.w, self.dy, dx=self.dx, grad_w=self.gw,
                           workspace=self.ws, block_n=self.wl.block_n)
        else:
            if op == "fwd":
                wsf.silu_fwd(self.x, self.w, y=self.y)
            else:
                wsf.silu_bwd(self.dy, self.x, self.w, dx=self.dx, dw=self.gw, workspace=self.ws)


def run_cuda(args, names):
    import torch
    import torch.distributed as dist
    import __graft_entry__
    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import backward_ws_fwd_gb300 as wsf

    host_io = not args.no_e2e
    WORKLOADS = scaled_workloads(args.scale)
    bufs = {n: Buffers(WORKLOADS[n], dev, wsf, host_io) for n in names}
    ops = steps_ops(names)
    step_bytes = sum(op_bytes(WORKLOADS[n], op) for n, op in ops)
    launches_per_step = sum(KERNELS_PER_OP[op_name(WORKLOADS[n], op)] for n, op in ops)

    def step():
        for n, op in ops:
            bufs[n].run(wsf, op)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # timed region: K steps bracketed by a barrier + device sync and two
    # events on the launching (current) stream, nothing in between (an event
    # between two kernels would stop the second from starting early).
    stream = torch.cuda.current_stream()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = Clocks(uuid or str(local))
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # per-op pass: the same K steps again with an event after every op, for
    # the per-op table and the roofline of the dominant op
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        e = evs[k]
        e[0].record(stream)
        for j, (n, op) in enumerate(ops):
            bufs[n].run(wsf, op)
            e[j + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    per_op_ms = [sum(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps)) / args.steps
                 for j in range(len(ops))]

    # isolated per-op protocol: an L2 flush (a write of twice the L2 size, then
    # a read of another such buffer, so that the flush's own dirty lines are
    # written back before the op starts) before every timed op, 5 warm-ups,
    # the median of 20; fwd+bwd is the two ops back to back after one flush
    isolated = isolated_per_op(bufs, names, wsf, dev, stream, WORKLOADS) if args.isolated else None
    if args.latency_names:
        lat = latency_per_op(lambda n: Buffers(WORKLOADS[n], dev, wsf, False), args.latency_names,
                             wsf, dev, WORKLOADS)
        isolated = dict(isolated or {}, **lat)

    # end to end through the public API with host buffers: every input is
    # copied from pinned host memory and the step's result back, inside the
    # timed region.  The result of a forward + backward step is the parameter
    # gradients (grad_w / dw, grad_b), what an optimizer step consumes; y and dx
    # stay on the device, where the next layer would use them.  A second figure
    # copies every output back too (y and dx as well).  Each workload is cut
    # into row chunks on three streams (H2D, compute, D2H) so that copies in
    # both directions overlap each other and the kernels; the chunked backward
    # accumulates grad_w / dw with the library's accumulate flag
    # (micro-batches), as a caller would.
    e2e = None
    if host_io:
        e2e_steps = max(1, min(args.steps, 10))
        streams = [torch.cuda.Stream(device=dev) for _ in range(3)]
        chunks = {"c2": 2, "c3": 8, "c4": 8, "c5": 4}

        def e2e_step(all_outputs):
            h2d, comp, d2h = streams
            for n in names:
                b = bufs[n]
                nc = min(chunks.get(n, 4), b.wl.N)
                bounds = [b.wl.N * j // nc for j in range(nc + 1)]
                with torch.cuda.stream(h2d):
                    b.w.copy_(b.hw, non_blocking=True)
                    if b.hb is not None:
                        b.b.copy_(b.hb, non_blocking=True)
                for j in range(nc):
                    r0, r1 = bounds[j], bounds[j + 1]
                    with torch.cuda.stream(h2d):
                        b.x[r0:r1].copy_(b.hx[r0:r1], non_blocking=True)
                        b.dy[r0:r1].copy_(b.hdy[r0:r1], non_blocking=True)
                        ready = torch.cuda.Event()
                        ready.record(h2d)
                    comp.wait_event(ready)
                    b.run_rows(wsf, r0, r1, accumulate=j > 0, stream=comp)
                    if all_outputs:
                        done = torch.cuda.Event()
                        done.record(comp)
                        d2h.wait_event(done)
                        with torch.cuda.stream(d2h):
                            b.hy[r0:r1].copy_(b.y[r0:r1], non_blocking=True)
                            b.hdx[r0:r1].copy_(b.dx[r0:r1], non_blocking=True)
                done = torch.cuda.Event()
                done.record(comp)
                d2h.wait_event(done)
                with torch.cuda.stream(d2h):
                    b.hgw.copy_(b.gw, non_blocking=True)
                    if b.hgb is not None:
                        b.hgb.copy_(b.gb, non_blocking=True)

        def e2e_time(all_outputs, nsteps):
            e2e_step(all_outputs)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            # each step ends when its result is on the host (a sync, as a
            # training loop that reads its loss); the median step time is the
            # value, so that a stall of the shared host does not decide it
            step_ms = []
            for _ in range(nsteps):
                t_a = time.perf_counter()
                e2e_step(all_outputs)
                torch.cuda.synchronize()
                step_ms.append((time.perf_counter() - t_a) * 1e3)
            med = max_over_ranks(statistics.median(step_ms), dev)
            return {"value": round(world * step_bytes / (med * 1e-3) / 1e9, 3), "unit": "GB/s",
                    "h2d_bytes_per_step": sum(bufs[n].h2d_bytes() for n in names),
                    "d2h_bytes_per_step": sum(bufs[n].d2h_bytes(all_outputs) for n in names),
                    "ms_per_step": round(med, 3), "ms_mean": round(statistics.mean(step_ms), 3),
                    "ms_max": round(max(step_ms), 3), "steps": nsteps}

        e2e = e2e_time(False, e2e_steps)
        e2e["how"] = ("pinned host buffers; inputs (x, w, dy, b) to the device and the step's "
                      "result, the parameter gradients, back to the host; per workload 2-8 row "
                      "chunks pipelined over H2D, compute and D2H streams; wall clock per step "
                      "from the first copy to the result on the host (device sync); median over "
                      "the steps")
        e2e["all_outputs"] = e2e_time(True, max(1, min(args.steps, 5)))
        e2e["all_outputs"]["how"] = "the same, with y and dx also copied back to the host"

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = read_peaks()
    ms_per_step = elapsed_ms / args.steps
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    per_op = {}
    for (n, op), ms in zip(ops, per_op_ms):
        wl = WORKLOADS[n]
        b = op_bytes(wl, op)
        per_op[f"{n}.{op}"] = {"ms": round(ms, 4), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                               "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                               "elements_per_s": round(op_elems(wl) / (ms * 1e-3), 1)}
    for n in names:
        wl = WORKLOADS[n]
        ms = per_op[f"{n}.fwd"]["ms"] + per_op[f"{n}.bwd"]["ms"]
        b = op_bytes(wl, "fwd") + op_bytes(wl, "bwd")
        per_op[f"{n}.fwd+bwd"] = {"ms": round(ms, 4), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                                  "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                                  "frac_of_8TBs": round(b / (ms * 1e-3) / 1e9 / 8000.0, 4)}
    # dominant op: the largest share of the step
    j = max(range(len(ops)), key=lambda i: per_op_ms[i])
    dn, dop = ops[j]
    dwl = WORKLOADS[dn]
    dbytes = op_bytes(dwl, dop)
    achieved = dbytes / (per_op_ms[j] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": f"{op_name(dwl, dop)} ({dn})",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": read_traffic(op_name(dwl, dop), dn),
                "algorithmic_bytes_per_launch": dbytes,
                "note": "achieved = algorithmic bytes / mean CUDA-event time of the op "
                        f"({KERNELS_PER_OP[op_name(dwl, dop)]} kernel(s)) over K steps of the "
                        "per-op pass (events after every op; the headline step time has none)"}
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64/Box-Muller, workload recipes)",
            "config": {"workload": workload_label(names) + (f" (rows x {args.scale})"
                                                             if args.scale != 1.0 else ""),
                       "step": [f"{n}.{op}" for n, op in ops],
                       "bytes_per_step": step_bytes,
                       "frac_of_peak": round(value / world / peak, 4),
                       "frac_of_8TBs": round(value / world / 8000.0, 4),
                       "l2": "inputs larger than L2; each fwd and its bwd are separated by "
                             ">= 1 GB of other traffic"},
            "roofline": roofline, "per_op": per_op, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "per_op_pass_ms_per_step": round(sum(per_op_ms), 4), "clocks": clk}
    if isolated is not None:
        line["per_op_isolated"] = isolated
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(args.latency_names + names)
        line["cpu_baseline"] = cpu
        # the oracle's rate beside each GPU row of the isolated protocol
        for k, row in (line.get("per_op_isolated") or {}).items():
            o = cpu["per_op"].get(k)
            if o and isinstance(row, dict):
                row["oracle_GB/s"] = o["GB/s"]
                row["oracle_GB/s_1core"] = o["GB/s_1core"]
                row["oracle_elements_per_s"] = o["elements_per_s"]
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def isolated_per_op(bufs, names, wsf, dev, stream, WORKLOADS, warmup=5, reps=20):
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    clean = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
    out = {}

    def timed(fn):
        for _ in range(warmup):
            flush.fill_(0)
            clean.sum()
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(1)
            clean.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    for n in names:
        wl, b = WORKLOADS[n], bufs[n]
        t = {op: timed(lambda op=op: b.run(wsf, op)) for op in ("fwd", "bwd")}
        t["fwd+bwd"] = timed(lambda: (b.run(wsf, "fwd"), b.run(wsf, "bwd")))
        for op, ms in t.items():
            nb = (op_bytes(wl, "fwd") + op_bytes(wl, "bwd")) if op == "fwd+bwd" else op_bytes(wl, op)
            out[f"{n}.{op}"] = {"ms": round(ms, 4), "GB/s": round(nb / (ms * 1e-3) / 1e9, 1),
                                "frac_of_8TBs": round(nb / (ms * 1e-3) / 1e9 / 8000.0, 4),
                                "elements_per_s": round(op_elems(wl) / (ms * 1e-3), 1)}
    out["_how"] = (f"L2 flush before every timed op: a write of {2 * l2 >> 20} MiB, then a read of "
                   f"another {2 * l2 >> 20} MiB (no dirty lines left for the op to write back); "
                   f"{warmup} warm-ups, median of {reps}; fwd+bwd = both ops back to back after one flush")
    return out


def latency_per_op(bufs_for, names, wsf, dev, WORKLOADS, reps=100, rounds=7, host_reps=50):
    """Small workloads that a launch's latency, not HBM, bounds (c1: the
    worked 100 x 64 shape with 32-row tiles), timed alone.  `ms` is the
    device time of one op: a CUDA graph of `reps` back-to-back calls is
    replayed `rounds` times (median), so no host launch cost is included;
    `host_us` is the wall-clock latency a caller sees for one call followed by
    a device synchronisation (median of host_reps)."""
    import torch
    out = {}
    for n in names:
        wl = WORKLOADS[n]
        b = bufs_for(n)
        ops = {"fwd": lambda: b.run(wsf, "fwd"), "bwd": lambda: b.run(wsf, "bwd"),
               "fwd+bwd": lambda: (b.run(wsf, "fwd"), b.run(wsf, "bwd"))}
        for op, fn in ops.items():
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for _ in range(3):
                    fn()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(reps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(rounds):
                a = torch.cuda.Event(enable_timing=True)
                c = torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                c.record()
                c.synchronize()
                ts.append(a.elapsed_time(c) / reps)
            hs = []
            for _ in range(host_reps):
                t = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                hs.append(time.perf_counter() - t)
            del g
            ms = statistics.median(ts)
            nb = (op_bytes(wl, "fwd") + op_bytes(wl, "bwd")) if op == "fwd+bwd" else op_bytes(wl, op)
            out[f"{n}.{op}"] = {"ms": round(ms, 5), "us": round(ms * 1e3, 2),
                                "GB/s": round(nb / (ms * 1e-3) / 1e9, 2),
                                "frac_of_8TBs": round(nb / (ms * 1e-3) / 1e9 / 8000.0, 6),
                                "elements_per_s": round(op_elems(wl) / (ms * 1e-3), 1),
                                "host_us": round(statistics.median(hs) * 1e6, 1),
                                "protocol": "latency"}
    out["_how_latency"] = (f"latency-bound workloads ({', '.join(names)}): ms = device time of one "
                           f"op from a CUDA graph of {reps} back-to-back calls (median of {rounds} "
                           f"replays); host_us = wall clock of one call plus a device sync "
                           f"(median of {host_reps})")
    return out


def scaled_workloads(scale: float):
    """The workload table with every row count multiplied by `scale`."""
    import dataclasses
    from inputgen.workloads import WORKLOADS
    if scale == 1.0:
        return WORKLOADS
    return {k: dataclasses.replace(v, N=max(1, int(round(v.N * scale)))) for k, v in WORKLOADS.items()}


def run_compare_atomic(args, names):
    """Measured comparison of the deterministic two-pass backward with the
    atomic-add variant (the pages' own scheme): mean backward time over K
    launches each, and how many distinct bit patterns grad_w / dw takes over
    the same K runs.  Prints one JSON line."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as wsf
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    WL = scaled_workloads(args.scale)
    out = {}
    for n in names:
        b = Buffers(WL[n], dev, wsf, host_io=False)
        wl = b.wl

        def two():
            b.run(wsf, "bwd")
            return b.gw

        def atom():
            if wl.op == "ws":
                wsf.ws_bwd_atomic(b.x, b.w, b.dy, dx=b.dx, grad_w=b.gw)
            else:
                wsf.silu_bwd_atomic(b.dy, b.x, b.w, dx=b.dx, dw=b.gw)
            return b.gw

        res = {}
        for label, fn in (("two_pass", two), ("atomic", atom)):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            pats = set()
            ms = []
            for _ in range(args.steps):
                a = torch.cuda.Event(enable_timing=True)
                c = torch.cuda.Event(enable_timing=True)
                a.record()
                g = fn()
                c.record()
                torch.cuda.synchronize()
                ms.append(a.elapsed_time(c))
                pats.add(bytes(g.view(torch.int32).cpu().numpy()))
            mean = sum(ms) / len(ms)
            res[label] = {"ms": round(mean, 4),
                          "GB/s": round(op_bytes(wl, "bwd") / (mean * 1e-3) / 1e9, 1),
                          "distinct_gradient_bit_patterns": len(pats)}
        res["atomic_speedup"] = round(res["two_pass"]["ms"] / res["atomic"]["ms"], 4)
        out[n] = res
        del b
        torch.cuda.empty_cache()
    print(json.dumps({"comparison": "backward: deterministic two-pass vs atomic-add parameter "
                                    "gradient", "runs_per_variant": args.steps,
                      "note": "each run timed alone with events (sync between runs)",
                      "per_workload": out}), flush=True)
    return 0


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch measured by ncu for this kernel and workload,
    from profiles/traffic.json, if a capture of the current source exists."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(f"{kernel}:{workload}")
        if e and e.get("source_hash") == source_hash(kernel.rsplit("_", 1)[0]):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# the kernel source of each operator; every operator also depends on the
# shared device helpers, the launch helpers and the C entry points
OP_SOURCES = {"silu": "silu.cu", "ws": "ws.cu", "rmsnorm": "norm.cu", "layernorm": "norm.cu",
              "softmax": "softmax.cu"}
SHARED_SOURCES = ("abi.cu", "wsf_device.cuh", "wsf_internal.h")


def _code_only(src: str) -> str:
    """C/C++/CUDA source with its comments removed and its whitespace
    collapsed (string and character literals kept as written)."""
    import re
    token = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|/\*.*?\*/|//[^\n]*',
                       re.S)
    src = token.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    return " ".join(src.split())


def source_hash(op: str | None = None) -> str:
    """Hash of the code of the kernel sources an operator is built from (all
    of them for op=None; comments and layout aside): a DRAM-traffic capture
    stays valid while its operator's hash is unchanged."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "backward_ws_fwd_gb300", "csrc")
    files = sorted(os.listdir(d)) if op is None else sorted((OP_SOURCES[op],) + SHARED_SOURCES)
    for f in files:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default="all",
                    help="all (c2..c5) or a comma list of c2,c3,c4,c5,s1,n1,n2,s2,n3,n4,s3,s4")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="multiply every workload's row count (profiling on small cases)")
    ap.add_argument("--compare-atomic", action="store_true",
                    help="measure the atomic-add backward variants against the two-pass ones")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--isolated", action=argparse.BooleanOptionalAction, default=True,
                    help="also time every op alone after an L2 flush (median of 20)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-latency", action="store_true",
                    help="skip the latency-bound workload c1 (timed alone, outside the step)")
    args = ap.parse_args(argv)
    names = ORDER_FWD if args.workload == "all" else [s.strip() for s in args.workload.split(",")]
    assert all(n in ORDER_FWD + EXTRA + LATENCY for n in names), names
    args.latency_names = [] if args.no_latency else (
        LATENCY if args.workload == "all" else [n for n in names if n in LATENCY])
    names = [n for n in names if n not in LATENCY]
    if not names:
        ap.error("name at least one workload of the step (c2..c5 or a row workload) besides c1")
    if args.warmup < 3 and args.impl == "cuda":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, names)
    if args.compare_atomic:
        return run_compare_atomic(args, names)
    return run_cuda(args, names)


if __name__ == "__main__":
    sys.exit(main())
