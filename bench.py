#!/usr/bin/env python3
"""Benchmark of the few-row packed-weight verify matmul on GB300.

One step = one verify pass of M drafted rows through a stack of distinct
packed weight matrices of the workload (a model-like stack, so consecutive
calls never find their weights in L2: the stack is larger than 4x L2), run
back to back on one stream through the C ABI.  Metric: packed-weight GB/s
(algorithmic bytes: packed weights + X + Y per call) and us per call, at
M = 1..8 rows, as a fraction of the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|NAME] [--impl lbv|reference]

With no --workload every configuration is timed (the rotated output head,
the 1-bit MLP-up, both 2-bit g64 shapes, the Q4_0 stack per call and as one
grouped launch); the JSON line's headline is the rotated head and "configs"
holds one entry per configuration.

N > 1 (under torchrun): independent replicas, one per GPU; no data-path
collective (the verify path shards by output columns, and each replica here
owns its own stack).  value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "us/call and packed-weight GB/s at M=1..8 rows, as % of GB300 HBM peak"
FMT_IDS = {synth.SIGN1_G128: 0, synth.AFFINE2: 1, synth.Q4_0: 2}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lbv", choices=["lbv", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(synth.WORKLOADS),
                    help="one workload, or all of them (the default; the first, the rotated "
                         "head, is the headline)")
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--no-sweep", action="store_true", help="skip the M=1..8 table")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-measure", action="store_true",
                    help="plans without LBV_PLAN_MEASURE (default launch shapes)")
    ap.add_argument("--shape", default="", help="warps,tpw,splits[,ctas] override of the launch shape")
    ap.add_argument("--kernel", default="mma", choices=["mma", "tc", "tc8"],
                    help="few-row kernel: mma.sync (default plans), tcgen05 with fp16 operands "
                         "(PLAN_TCGEN05) or tcgen05 with e4m3 operands (PLAN_TC_E4M3)")
    ap.add_argument("--head", default="fused", choices=["fused", "two-call", "greedy"],
                    help="rotated head: rotation fused into the verify launch (default), "
                         "lbv_fwht128 then lbv_verify_gemm, or fused rotation and per-row "
                         "argmax without writing the logits")
    ap.add_argument("--stack", default="grouped", choices=["grouped", "calls"],
                    help="multi-matrix workloads: every matrix in one grouped launch "
                         "(default) or one verify call per matrix")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense fp16 cuBLAS context timing")
    ap.add_argument("--no-graph", action="store_true", help="launch each call from Python")
    ap.add_argument("--quick", action="store_true", help="no sustained clock window (profiling)")
    ap.add_argument("--json-out", default="")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def packed_weight_bytes(mat):
    """Algorithmic packed bytes of one matrix from its format: 1 bit per
    weight + an fp16 scale per 128 (sign g128), 2 bits + fp16 scale and bias
    per group (2-bit affine), 18 bytes per 32 weights (Q4_0)."""
    K, N = mat.K, mat.N
    if mat.fmt == synth.SIGN1_G128:
        return N * K // 8 + N * (K // 128) * 2
    if mat.fmt == synth.AFFINE2:
        return N * K // 4 + N * (K // mat.group) * 4
    return N * (K // 32) * 18


def call_bytes(mat, M, head="fused"):
    """Algorithmic bytes of one call: packed weights, X, and Y (or, for the
    greedy head, the argmax column and logit of each row)."""
    out = M * 8 if (mat.rotate and head == "greedy") else M * mat.N * 4
    return packed_weight_bytes(mat) + M * mat.K * 2 + out


# ---------------------------------------------------------------------------
# clocks during the measurement

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the lbv arm

_GEN = {"workload": None}


def gen_cached(workload, mat, seed):
    """synth.gen_matrix, kept while the configurations of one workload run."""
    if _GEN["workload"] != workload:
        _GEN.clear()
        _GEN["workload"] = workload
    key = (mat, str(seed))
    if key not in _GEN:
        _GEN[key] = synth.gen_matrix(mat, seed)
    return _GEN[key]


class Stack:
    """Distinct packed matrices of a workload resident on the device."""

    def __init__(self, workload, pdl: bool, shape: str, l2_bytes: int, M: int,
                 use_graphs: bool = True, kernel: str = "mma", head: str = "fused",
                 stack: str = "grouped", measure: bool = True):
        import torch
        self.use_graphs = use_graphs
        self.graphs = {}
        self.head = head

        import few_row_packed_gb300 as lbv
        wl = synth.WORKLOADS[workload]
        self.mats = list(wl.matrices)
        flags = ((lbv.PLAN_PDL if pdl else 0) | (lbv.PLAN_TCGEN05 if kernel == "tc" else 0) |
                 (lbv.PLAN_TC_E4M3 if kernel == "tc8" else 0))
        # plans are set up once per weight shape, timing their candidate launch
        # shapes and the 1-row crossover (LBV_PLAN_MEASURE)
        mflag = lbv.PLAN_MEASURE if measure else 0
        self.layers = []
        if len(self.mats) == 1:
            mat = self.mats[0]
            per = packed_weight_bytes(mat)
            L = max(64 if per < 100e6 else 3, math.ceil(4 * l2_bytes / per))
            ndistinct = min(L, 4)
            gens = [gen_cached(workload, mat, [wl.seed, i]) for i in range(ndistinct)]
            mats = [mat] * L
            gen_of = [gens[i % ndistinct] for i in range(L)]
        else:
            mats = self.mats
            gen_of = [gen_cached(workload, m, synth.matrix_seed(wl, i)) for i, m in enumerate(mats)]
        plans = {}
        packed_cache = {}
        for i, (mat, (parts, xb)) in enumerate(zip(mats, gen_of)):
            key = (mat.fmt, mat.K, mat.N, mat.group, mat.xdtype)
            if key not in plans:
                plans[key] = lbv.Plan(FMT_IDS[mat.fmt], mat.K, mat.N, mat.group,
                                      lbv.DTYPE_BY_NAME[mat.xdtype],
                                      flags | (mflag if not shape else 0))
                if shape and (len(self.mats) == 1 or stack != "grouped"):
                    plans[key].set_shape(*[int(v) for v in shape.split(",")])
            pid = id(parts[0])
            if pid not in packed_cache:
                packed_cache[pid] = lbv.pack(FMT_IDS[mat.fmt], parts, mat.K, mat.N, mat.group,
                                             plan=plans[key])
            Wp = torch.from_numpy(packed_cache[pid]).cuda()       # a distinct allocation
            X = torch.from_numpy(xb.view(np.int16)).cuda()
            Xr = torch.zeros_like(X) if mat.rotate else None
            Y = torch.zeros((8, mat.N), dtype=torch.float32, device="cuda")
            self.layers.append((mat, plans[key], Wp, X, Xr, Y))
        self.plans = plans
        self.bytes_per_step = {m: sum(call_bytes(l[0], m, head) for l in self.layers)
                               for m in range(1, 9)}
        self.calls = len(self.layers)
        self.launches_per_step = sum(2 if (l[0].rotate and head == "two-call") else 1
                                     for l in self.layers)
        # a model's matrices in grouped launches
        self.group = None
        if len(self.mats) > 1 and stack == "grouped" and kernel == "mma":
            m0 = self.mats[0]
            self.group = lbv.Group(FMT_IDS[m0.fmt], m0.group, lbv.DTYPE_BY_NAME[m0.xdtype],
                                   [(m.K, m.N) for m in mats], flags | (mflag if not shape else 0))
            if shape:
                self.group.set_shape(*[int(v) for v in shape.split(",")])
            self.launches_per_step = self.group.launches()
        # greedy head: argmax outputs and the (zeroed) workspace the calls share
        self.idx = torch.zeros(8, dtype=torch.int32, device="cuda")
        self.val = torch.zeros(8, dtype=torch.float32, device="cuda")
        self.ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")

    def shape_desc(self):
        """The launch shapes the step uses."""
        if self.group is not None:
            return [{"warps": 16, "tiles_per_warp": t, "splits": sp, "cluster_rows": r,
                     "matrices": sum(self.group.problem_launch(i) == c
                                     for i in range(self.group.count))}
                    for c in range(self.group.launches())
                    for t, sp, r in [self.group.shape(c)]]
        out = []
        for key, plan in self.plans.items():
            w, t, sp, ctas = plan.shape()
            out.append({"K": key[1], "N": key[2], "warps": w, "tiles_per_warp": t, "splits": sp,
                        "ctas_n": ctas})
        return out if len(out) > 1 else out[0]

    def dispatch_desc(self):
        """Per shape, the row-count dispatch the plan chose (LBV_PLAN_MEASURE
        times the few-row kernel and the 1-row path run M times)."""
        if self.group is not None:
            return None
        import few_row_packed_gb300 as lbv
        out = []
        for key, plan in self.plans.items():
            per = {}
            crossover = None
            for M in range(1, 9):
                few, gemv, crossover = plan.measured(M)
                kernel = plan.query(M)[0]
                per[str(M)] = {"kernel": ("1-row" if kernel == lbv.KERNEL_GEMV else "few-row"),
                               "fewrow_us": round(few, 3), "one_row_times_M_us": round(gemv, 3)}
            out.append({"K": key[1], "N": key[2], "crossover": crossover, "per_M": per})
        return out if len(out) > 1 else out[0]

    def graph(self, M, verify_only=False):
        """A CUDA graph of one step (launches captured through the C ABI)."""
        import torch
        key = (M, verify_only)
        if key not in self.graphs:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                self.step(M, verify_only)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(M, verify_only)
            self.graphs[key] = g
        return self.graphs[key]

    def run(self, M, verify_only=False):
        if self.use_graphs:
            self.graph(M, verify_only).replay()
        else:
            self.step(M, verify_only)

    def step(self, M, verify_only=False):
        import few_row_packed_gb300 as lbv
        if self.group is not None:
            lbv.verify_grouped(self.group, [(X, M, Wp, Y) for _, _, Wp, X, _, Y in self.layers])
            return
        for mat, plan, Wp, X, Xr, Y in self.layers:
            if not mat.rotate or verify_only:
                lbv.verify_gemm(plan, X, M, Wp, Y)
            elif self.head == "two-call":
                lbv.fwht128(X, Xr, M, mat.K, lbv.DTYPE_BY_NAME[mat.xdtype])
                lbv.verify_gemm(plan, Xr, M, Wp, Y)
            elif self.head == "fused":
                lbv.verify_fused(plan, X, M, Wp, lbv.FUSED_ROTATE, Y=Y)
            else:
                lbv.verify_fused(plan, X, M, Wp, lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX,
                                 idx=self.idx, val=self.val, workspace=self.ws)


@contextlib.contextmanager
def nvtx_range(name):
    """An NVTX range around a phase of the bench, for Nsight timelines; a
    no-op where torch was built without NVTX.  Host-side markers only."""
    import torch
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pushed = False
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


def timed(torch, fn, steps, warmup, barrier):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def dense_context(stack, M, l2_bytes, steps, warmup, peak, barrier, reduce_max):
    """Context, not the product: the step's matrices as a dense fp16 GEMM in
    cuBLAS (torch.matmul, fp16 x fp16 -> fp16) on the weights expanded once
    by lbv_dequant_fp16, with enough dense copies that a step's weights
    exceed 4x L2, captured in a CUDA graph like the packed step."""
    import torch

    import few_row_packed_gb300 as lbv
    dense_b = [l[0].K * l[0].N * 2 for l in stack.layers]
    if len(stack.mats) == 1:
        n = min(len(stack.layers), max(2, math.ceil(4 * l2_bytes / dense_b[0])))
    else:
        n = len(stack.layers)
    calls = []
    for mat, plan, Wp, X, _, _ in stack.layers[:n]:
        W = torch.empty((mat.K, mat.N), dtype=torch.float16, device="cuda")
        lbv.dequant_fp16(plan, Wp, W.view(torch.int16))
        Xh = X[:M].view(torch.float16 if mat.xdtype == "f16" else torch.bfloat16)
        Xh = Xh.to(torch.float16).contiguous()
        Yh = torch.empty((M, mat.N), dtype=torch.float16, device="cuda")
        calls.append((Xh, W, Yh))

    def step():
        for Xh, W, Yh in calls:
            torch.matmul(Xh, W, out=Yh)

    how = "CUDA graph of the step"
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        run = g.replay
    except Exception as e:                       # eager launches, said so below
        torch.cuda.synchronize()
        run, how = step, f"eager launches (graph capture failed: {type(e).__name__})"
    ms = reduce_max(timed(torch, run, steps, warmup, barrier))
    us = ms * 1e3 / (steps * n)
    bytes_call = sum(b + M * mat.K * 2 + M * mat.N * 2
                     for b, (mat, *_r) in zip(dense_b[:n], stack.layers[:n])) / n
    gbs = bytes_call / (us * 1e-6) / 1e9
    del calls
    torch.cuda.empty_cache()
    return {"us_per_call": round(us, 3), "GBps": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "bytes_per_call": round(bytes_call),
            "matrices_per_step": n,
            "how": f"cuBLAS fp16 GEMM (torch.matmul) on the dequantized weights, {how}; "
                   "rotation not included; context only"}


def code_text(src: str) -> str:
    """C/C++ source without its comments, trailing blanks and empty lines."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] in "\"'":                    # string or character literal
            q, j = src[i], i + 1
            while j < n and src[j] != q:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_hash():
    """Hash of the device code (kernels and the headers they include, without
    comments); the host-side planning in the .cpp files does not change what a
    captured launch executes."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "few_row_packed_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, M, kernel):
    """DRAM bytes per verify launch from the committed ncu capture of this
    workload and kernel ("mma", "tc", "tc8" or "grouped"), if it was taken on
    the current kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[f"{workload}/{kernel}"]
        if e.get("kernel_hash") == kernel_hash() and int(e.get("M", -1)) == M:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def host_cpu():
    """The host's processor model and core counts (where the oracle runs)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"model": model or os.uname().machine, "nproc": os.cpu_count(),
            "usable": len(os.sched_getaffinity(0))}


def oracle_columns(oracle, fmt, parts, Xf, mat, cols, nthreads):
    """The oracle's verify over `cols`, split into contiguous column ranges
    run on `nthreads` host threads (the C call releases the GIL; columns are
    independent, so this is the oracle unchanged, over N in parallel)."""
    if nthreads <= 1:
        oracle.verify(fmt, parts, Xf, mat.K, mat.N, mat.group, cols=cols)
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(lambda c: oracle.verify(fmt, parts, Xf, mat.K, mat.N, mat.group, cols=c),
                    np.array_split(cols, nthreads)))


def oracle_sample(workload, M, budget_s, head, nthreads):
    """GB/s of the fp64 oracle on nthreads host threads: verify calls on the
    workload's matrices (whole, or a slice of columns) until about budget_s
    has passed."""
    import oracle
    oracle.build()
    wl = synth.WORKLOADS[workload]
    done_bytes, t_total, calls, cols_done = 0, 0.0, 0, 0
    i = 0
    while t_total < budget_s and i < 64:
        mat = wl.matrices[i % len(wl.matrices)]
        parts, xb = synth.gen_matrix(mat, synth.matrix_seed(wl, i % len(wl.matrices)))
        Xf = oracle.x_to_f64(xb[:M], mat.xdtype)
        if mat.rotate:
            Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(Xf), mat.xdtype), mat.xdtype)
        # columns: the whole matrix if it is small enough, else a slice
        ncols = mat.N if mat.N <= 20000 * nthreads else min(mat.N, 16384 * nthreads)
        cols = np.arange(ncols)
        t0 = time.perf_counter()
        oracle_columns(oracle, FMT_IDS[mat.fmt], parts, Xf, mat, cols, nthreads)
        dt = time.perf_counter() - t0
        done_bytes += call_bytes(mat, M, head) * ncols / mat.N
        t_total += dt
        cols_done += ncols
        calls += 1
        i += 1
    gbs = done_bytes / t_total / 1e9
    us_per_call = t_total / (done_bytes / call_bytes(wl.matrices[0], M, head)) * 1e6
    how = "single-threaded" if nthreads == 1 else f"on {nthreads} threads over column ranges"
    return {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "us_per_call": us_per_call,
            "sample": f"{calls} oracle verify call(s), {cols_done} output columns x {M} rows "
                      f"of {workload}, {t_total:.1f} s {how}; GB/s of the sample's "
                      "algorithmic bytes"}


def cpu_baseline(workload, M, budget_s=10.0, head="fused"):
    """The fp64 oracle as it stands on the host: single-threaded (the reported
    baseline), and the same calls spread over every usable core."""
    line = oracle_sample(workload, M, budget_s, head, 1)
    host = host_cpu()
    line["host"] = host
    if host["usable"] > 1:
        line["all_cores"] = oracle_sample(workload, M, budget_s / 2, head, host["usable"])
    return line


# The configurations timed by default, in order; the headline line is the
# first: the rotated output head, the largest single verify call (219 MB of
# packed weights) and one of the shapes with a 70 % bandwidth target.  The
# Q4_0 layer stack is larger in all (767 MB) but is 28 calls; it is reported
# per call and as one grouped launch of its 28 independent problems.
ALL_CONFIGS = [
    ("head_rot_affine2_g128_5120x151936", "grouped"),
    ("sign1_mlp_up_5120x17408", "grouped"),
    ("affine2_g64_6144x6144", "grouped"),
    ("affine2_g64_kv_5120x1024", "grouped"),
    ("q4_0_stack_4x7", "calls"),
    ("q4_0_stack_4x7", "grouped"),
]


def config_label(workload, stack_mode, multi):
    if not multi:
        return workload
    return (f"{workload} (one verify call per matrix)" if stack_mode == "calls" else
            f"{workload} (one grouped launch of its independent problems)")


def measure_config(args, workload, stack_mode, l2, peak, barrier, reduce_max, world,
                   headline):
    """Times one configuration: the step (args.steps steps after args.warmup),
    the M = 1..8 sweep, and for the headline the end-to-end and dense-GEMM
    context.  Returns (summary dict, Stack, extra headline fields)."""
    import torch

    tag = f"lbv/{workload}" + (f"/{stack_mode}" if stack_mode else "")
    with nvtx_range(f"{tag}/setup"):
        stack = Stack(workload, not args.no_pdl, args.shape, l2, args.M, kernel=args.kernel,
                      use_graphs=not args.no_graph, head=args.head, stack=stack_mode,
                      measure=not args.no_measure)
        grouped = stack.group is not None
        rotated = any(l[0].rotate for l in stack.layers)
        stack.run(args.M)
        t_end = time.time() + (0.0 if args.quick else 1.0)
        while time.time() < t_end:
            for _ in range(max(1, args.warmup)):
                stack.run(args.M)
            torch.cuda.synchronize()
    with nvtx_range(f"{tag}/timed M={args.M}"):
        ms = reduce_max(timed(torch, lambda: stack.run(args.M), args.steps, args.warmup,
                              barrier))
    ms_per_step = ms / args.steps
    bytes_step = stack.bytes_per_step[args.M]
    value = replica_value(bytes_step, world, ms_per_step)

    # the dominant kernel: the verify launch, timed alone (verify-only loop)
    # when the step also launches the separate rotation
    if rotated and args.head == "two-call":
        with nvtx_range(f"{tag}/verify only"):
            ms_v = reduce_max(timed(torch, lambda: stack.run(args.M, verify_only=True),
                                    args.steps, args.warmup, barrier))
    else:
        ms_v = ms
    verify_launches = stack.group.launches() if grouped else stack.calls
    us_launch = ms_v * 1e3 / (args.steps * verify_launches)
    bytes_launch = bytes_step / verify_launches
    achieved = bytes_launch / (us_launch * 1e-6) / 1e9

    per_M = {}
    if not args.no_sweep:
        for M in range(1, 9):
            n = max(10, args.steps // 2)
            with nvtx_range(f"{tag}/sweep M={M}"):
                msm = reduce_max(timed(torch, lambda: stack.run(M), n, args.warmup, barrier))
            us = msm * 1e3 / (n * stack.calls)
            gbs = stack.bytes_per_step[M] / stack.calls / (us * 1e-6) / 1e9
            per_M[str(M)] = {"us_per_call": round(us, 3), "GBps": round(gbs, 1),
                             "frac_of_measured_hbm": round(gbs / peak, 4)}

    multi = len(stack.mats) > 1
    summary = {
        "workload": workload,
        "label": config_label(workload, stack_mode, multi),
        "M": args.M,
        "calls_per_step": stack.calls,
        "us_per_call": round(ms_per_step * 1e3 / stack.calls, 3),
        "GBps": round(value / world, 1),
        "frac_of_measured_hbm": round(value / world / peak, 4),
        "per_M": per_M,
        "m8_over_m1": (round(per_M["8"]["us_per_call"] / per_M["1"]["us_per_call"], 3)
                       if per_M else None),
        "launches_per_step": stack.launches_per_step,
        "shape": stack.shape_desc(),
        "dispatch": stack.dispatch_desc(),
        "head": args.head if rotated else None,
    }
    if grouped:
        summary["note"] = ("one launch over the stack's matrices as independent problems, each "
                           "with its own X; us_per_call is the launch time divided by the "
                           "matrices")
    extra = {"ms_per_step": ms_per_step, "bytes_step": bytes_step, "value": value,
             "achieved": achieved, "bytes_launch": bytes_launch, "us_launch": us_launch,
             "grouped": grouped, "rotated": rotated, "kernel_key": "grouped" if grouped else args.kernel}
    if headline:
        with nvtx_range(f"{tag}/e2e"):
            extra["e2e"] = e2e_measure(args, stack, bytes_step, world, barrier, reduce_max)
        if not args.no_dense:
            with nvtx_range(f"{tag}/dense fp16 context"):
                dense = dense_context(stack, args.M, l2, max(3, args.steps // 4), args.warmup,
                                      peak, barrier, reduce_max)
            dense["packed_speedup"] = round(dense["us_per_call"] / (ms_per_step * 1e3 / stack.calls), 2)
            extra["dense"] = dense
    return summary, stack, extra


def e2e_measure(args, stack, bytes_step, world, barrier, reduce_max):
    """End to end through the public API with host buffers: per step, X from
    pinned host memory to the device, the verify stack, the result back."""
    import torch
    rotated = any(l[0].rotate for l in stack.layers)
    greedy = rotated and args.head == "greedy"
    mat0 = stack.layers[0][0]
    x_host = torch.from_numpy(stack.layers[0][3].cpu().numpy()).pin_memory()
    X_dev = stack.layers[0][3]
    if greedy:       # the result of a greedy step: each row's column and logit
        outs = [(stack.idx, torch.zeros(8, dtype=torch.int32).pin_memory()),
                (stack.val, torch.zeros(8, dtype=torch.float32).pin_memory())]
    else:
        outs = [(stack.layers[-1][5], torch.zeros((args.M, stack.layers[-1][0].N),
                                                  dtype=torch.float32).pin_memory())]
    d2h = sum(h[:args.M].numel() * h.element_size() for _, h in outs)

    def e2e_step():
        X_dev[:args.M].copy_(x_host[:args.M], non_blocking=True)
        stack.run(args.M)
        for d, h in outs:
            h[:args.M].copy_(d[:args.M], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    t_e2e = reduce_max((time.perf_counter() - t0) * 1e3)
    return {"value": round(replica_value(bytes_step, world, t_e2e / args.steps), 2),
            "unit": "GB/s", "h2d_bytes_per_step": args.M * mat0.K * 2,
            "d2h_bytes_per_step": d2h}


def run_lbv(args, rank, world, barrier, reduce_max):
    import torch

    import few_row_packed_gb300 as lbv
    lbv.build()
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    peak, peak_kind = peaks()
    phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(dev)).split(",")[dev]
    configs = ([(args.workload, args.stack)] if args.workload != "all" else ALL_CONFIGS)
    skipped = []
    if args.kernel == "tc8":
        # the e4m3 tensor-memory kernel reads the g128 formats only
        keep = [c for c in configs if all(m.group == 128 and m.fmt != synth.Q4_0
                                          for m in synth.WORKLOADS[c[0]].matrices)]
        skipped = [{"workload": w, "stack": st, "skipped": "the e4m3 kernel reads sign1 g128 "
                    "and affine2 g128 only"} for w, st in configs if (w, st) not in keep]
        configs = keep
    if not configs:
        raise SystemExit("no configuration runs on the chosen kernel")

    sampler = ClockSampler(int(phys) if phys.isdigit() else dev)
    sampler.start()
    results = []
    head_summary = head_stack = head_extra = None
    for i, (workload, stack_mode) in enumerate(configs):
        summary, stack, extra = measure_config(args, workload, stack_mode, l2, peak, barrier,
                                               reduce_max, world, headline=(i == 0))
        results.append(summary)
        if i == 0:
            head_summary, head_stack, head_extra = summary, stack, extra
        else:
            del stack
            torch.cuda.empty_cache()
    clocks = sampler.stop()

    workload = configs[0][0]
    mat0 = head_stack.layers[0][0]
    traffic = recorded_traffic(workload, args.M, head_extra["kernel_key"])
    line = {
        "metric": METRIC,
        "value": round(head_extra["value"], 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head_extra["ms_per_step"], 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16" if mat0.xdtype == "f16" else "bf16",
        "data": "synthetic",
        "config": {
            "workload": workload,
            "label": head_summary["label"],
            "M": args.M,
            "calls_per_step": head_stack.calls,
            "us_per_call": head_summary["us_per_call"],
            "l2": f"inputs larger than L2: {head_stack.calls} distinct resident matrices, "
                  f"{head_extra['bytes_step'] / 1e6:.0f} MB per step vs {l2 / 1e6:.0f} MB L2",
            "plans": "launch shapes measured at plan creation (LBV_PLAN_MEASURE)"
                     if not (args.no_measure or args.shape) else "default launch shapes",
            "launch": ("CUDA graph of the step, " if not args.no_graph else "") +
                      ("programmatic dependent launch, " if not args.no_pdl else "") +
                      "back to back on one stream",
            "shape": head_summary["shape"],
            "kernel": {"tc": "tcgen05 (fp16 operands)", "tc8": "tcgen05 (e4m3 operands)"}.get(
                args.kernel, "mma.sync"),
            "head": head_summary["head"],
            "us_per_step": round(head_extra["ms_per_step"] * 1e3, 3),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "per_M": head_summary["per_M"],
        "m8_over_m1": head_summary["m8_over_m1"],
        "roofline": {"bound": "hbm", "achieved": round(head_extra["achieved"], 1), "peak": peak,
                     "unit": "GB/s", "frac": round(head_extra["achieved"] / peak, 4),
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": ("lbv_verify_grouped_kernel" if head_extra["grouped"] else
                                {"tc": "lbv_tc_kernel", "tc8": "lbv_t8_kernel"}.get(
                                    args.kernel, "lbv_verify_kernel")),
                     "bytes_per_launch": head_extra["bytes_launch"],
                     "us_per_launch": round(head_extra["us_launch"], 3)},
        "e2e": head_extra["e2e"],
        "gpu_launches": args.steps * head_stack.launches_per_step,
        "clocks": clocks,
        "dense_fp16_context": head_extra.get("dense"),
        "configs": results + skipped,
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(workload, args.M, budget_s=10.0, head=args.head)
        if len(configs) > 1:
            nthr = line["cpu_baseline"]["host"]["usable"]
            for r in results[1:]:
                r["cpu_baseline"] = oracle_sample(r["workload"], args.M, 2.0, args.head, nthr)
    return line


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands on the host cores
    (threads over column ranges, every usable core); each step is a bounded
    sample (a slice of output columns) of the workload."""
    import oracle
    oracle.build()
    workload = ALL_CONFIGS[0][0] if args.workload == "all" else args.workload
    wl = synth.WORKLOADS[workload]
    mat = wl.matrices[0]
    parts, xb = synth.gen_matrix(mat, synth.matrix_seed(wl, 0))
    M = args.M
    Xf = oracle.x_to_f64(xb[:M], mat.xdtype)
    if mat.rotate:
        Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(Xf), mat.xdtype), mat.xdtype)
    host = host_cpu()
    nthr = host["usable"]
    ncols = min(mat.N, 256 * nthr)
    cols = np.arange(ncols)
    fmt = FMT_IDS[mat.fmt]
    for _ in range(max(0, args.warmup)):
        oracle_columns(oracle, fmt, parts, Xf, mat, cols, nthr)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_columns(oracle, fmt, parts, Xf, mat, cols, nthr)
    dt = time.perf_counter() - t0
    sample_bytes = call_bytes(mat, M, args.head) * ncols / mat.N
    gbs = sample_bytes * args.steps / dt / 1e9
    sample = (f"{ncols} of {mat.N} output columns x {M} rows of {workload} per step, "
              f"fp64 oracle on {nthr} threads over column ranges")
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload, "M": M, "sample_columns": ncols},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nthr, "kind": "oracle",
                         "sample": sample, "host": host},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def replica_helpers(dist, device):
    """Barrier and max-over-ranks for N independent replicas (no data-path
    collective: every rank streams its own copy of the workload)."""
    import torch

    def barrier():
        dist.barrier()

    def reduce_max(v):
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, reduce_max


def replica_value(bytes_per_step_per_rank, world, ms_per_step_max):
    """Whole-job GB/s: the bytes all ranks streamed over the slowest rank's time."""
    return bytes_per_step_per_rank * world / (ms_per_step_max * 1e-3) / 1e9


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            line = run_reference(args)
            print(json.dumps(line))
        return

    import torch
    torch.cuda.set_device(local)
    barrier = lambda: None  # noqa: E731
    reduce_max = lambda v: v  # noqa: E731
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier, reduce_max = replica_helpers(dist, "cuda")

    line = run_lbv(args, rank, world, barrier, reduce_max)
    if rank == 0:
        print(json.dumps(line))
        if args.json_out:
            with open(args.json_out, "w") as f:
                json.dump(line, f, indent=1)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
