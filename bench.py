"""Benchmark: dense linear-layer GEMM throughput on GB300 through the C ABI.

One step = one pass over a workload's GEMMs (default: the bf16 ragged-shape
set -- decode batches of 1/8/16 tokens, 48x4096x48, 333/528/3402-token
prefill shapes, the 1024x50257x512 lm_head, 2048x11007x1024, 4095^2x1024 --
with N(0,1) activations, N(0,0.02) weights and bf16 C).  Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W]
                  [--workload ragged|llama7b_mlp|square|fp8|mxfp4|w4a8|linear|gpt3xl_train|square256]
  python bench.py --impl reference      # the fp64 CPU oracle, timed on the host cores

value = 2*m*n*K summed over the step's GEMMs (valid extents only) / step time,
TFLOP/s, summed over ranks (each rank runs the workload independently).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) & % GB300 tensor peak; decode GB/s vs HBM"
WORKLOAD_TEXT = {
    "ragged": "bf16 ragged-shape sweep, fp32 accumulate, bf16 C: (1,11008,4096) (8,4096,4096) (16,4096,4096) "
              "(48,4096,48) (333,4096,1024) (528,528,1024) (3402,4096,1024) (1024,50257,512) "
              "(2048,11007,1024) (4095,4095,1024); A~N(0,1), B~N(0,0.02)",
    "llama7b_mlp": "LLaMA-2-7B MLP up/gate shapes, bf16: (597,11008,4096) prefill, decode M in {1,4,16}",
    "square": "bf16 squares M=N=K in {2048,4096,8192}, A,B~N(0,1), bf16 C",
    "fp8": "E4M3 with per-row/per-column fp32 scales, bf16 C: (4096,4096,4096) (597,11008,4096) (16,11008,4096)",
    "mxfp4": "MXFP4 (E2M1, one E8M0 scale per 32 of K), bf16 C: (4096,4096,4096) (597,11008,4096) "
             "(16,11008,4096)",
    "w4a8": "W4A8 (E4M3 activations, per-row-scaled E2M1 weights), bf16 C: (4096,4096,4096) (597,11008,4096) "
            "(16,11008,4096) (1,11008,4096)",
    "square256": "bf16 256^3, fp32 C: uniform[-1,1] and integer [-4,4] variants",
    "gpt3xl_train": "GPT-3-XL feed-forward projection, one training step, bf16 C: forward 10240x8192x2048 + bias "
                    "+ GELU; dX = dY W 10240x2048x8192 (W read MN-major); dW = dY^T X 8192x2048x10240 "
                    "(both operands MN-major)",
    "linear": "linear layers with fused epilogues, bf16 C: GPT-3-XL forward addmm 10240x8192x2048 + bias + GELU; "
              "LLaMA-2-7B prefill up/gate pair 597x(2x11008)x4096 as one gated SiLU call, bf16 and E4M3",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="dgl", choices=["dgl", "reference"])
    ap.add_argument("--workload", default="ragged", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--shape", default=None,
                    help="single GEMM m,n,k[,bf16|fp8[,bf16|f32]] instead of a workload (profiling)")
    ap.add_argument("--tile", default=None,
                    help="force the tcgen05 tile MxN (e.g. 256x256) instead of the planner's choice (profiling)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-macs", type=float, default=4e9,
                    help="multiply-adds of the bounded CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the torch.matmul (cuBLAS) context column")
    ap.add_argument("--no-headline", action="store_true",
                    help="skip the headline shapes (4096^3 bf16 / E4M3, decode) timed one by one")
    return ap.parse_args()


def csrc_digest():
    """sha256 over the CUDA sources, as recorded beside the ncu traffic figures."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "dense_gemm_linear_gb300", "csrc", "*"))):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None
    when there is none for this workload or the kernels changed since."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}_sweep.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("csrc_sha256") != csrc_digest():
        return None
    k = rec.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing
def oracle_band(oracle, lib, c, rows):
    """The oracle on the first `rows` rows of case c (the GEMM, or the linear layer)."""
    if c.dtype == "mxfp4":
        oracle.mxfp4_gemm(c.A[:rows], c.B, c.sa[:rows], c.sb, lib=lib)
        return
    if c.dtype == "w4a8":
        oracle.w4a8_gemm(c.A[:rows], c.B, c.sa[:rows], c.sb, lib=lib)
        return
    dt = oracle.BF16 if c.dtype == "bf16" else oracle.E4M3
    sa = c.sa[:rows] if c.sa is not None else None
    if c.linear:
        oracle.linear(dt, c.A[:rows], c.B, sa, c.sb, bias=c.bias, act=c.act, gated=c.gated, lib=lib)
    else:
        oracle.gemm(dt, c.A[:rows], c.B, sa, c.sb, lib=lib)


def oracle_sample_run(cases, mac_budget):
    """Time the oracle on a bounded band of rows of every case; returns (flops, seconds, threads, text)."""
    import oracle
    lib = oracle.load()
    per_case = mac_budget / max(1, len(cases))
    flops, secs, parts = 0.0, 0.0, []
    for c in cases:
        rows = int(max(1, min(c.m, per_case // max(1, c.b_rows * c.K))))
        t0 = time.perf_counter()
        oracle_band(oracle, lib, c, rows)
        secs += time.perf_counter() - t0
        flops += 2.0 * rows * c.b_rows * c.K
        parts.append(f"{rows}x{c.b_rows}x{c.K}")
    return flops, secs, oracle.threads(lib), "first rows of each GEMM: " + ", ".join(parts)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from synthetic import WORKLOADS, make_workload_case
    entries = WORKLOADS[args.workload] if args.shape is None else [shape_entry(args.shape)]
    cases = [make_workload_case(e) for e in entries]
    # each step: a bounded band of one GEMM (round robin), sized so the whole run stays within minutes
    total_steps = args.steps + args.warmup
    budget_macs = min(args.cpu_macs, 3e10 / max(1, total_steps)) if total_steps else args.cpu_macs
    import oracle
    lib = oracle.load()
    flops_t, secs_t = 0.0, 0.0
    desc = []
    for s in range(total_steps):
        c = cases[s % len(cases)]
        rows = int(max(1, min(c.m, budget_macs // max(1, c.b_rows * c.K))))
        t0 = time.perf_counter()
        oracle_band(oracle, lib, c, rows)
        el = time.perf_counter() - t0
        if s >= args.warmup:
            flops_t += 2.0 * rows * c.b_rows * c.K
            secs_t += el
            if len(desc) < len(cases):
                desc.append(f"{rows}x{c.b_rows}x{c.K}")
    value = flops_t / secs_t / 1e12 if secs_t > 0 else 0.0
    cores = oracle.threads(lib)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs_t / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_text(args), "sample": "one GEMM per step, round robin"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: first rows of one GEMM: " + ", ".join(desc)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def over_ranks(ms_per_step, step_flops, dist=None, device=None):
    """The job's step time and throughput from each rank's own step time.

    Every rank runs the whole step on its own GPU (replicas, no data-path
    collective), so the job does `world` steps' work in the slowest rank's
    time: returns (max over ranks of ms_per_step, TFLOP/s of the whole job).
    dist: torch.distributed when initialised, else None (one process)."""
    world = 1
    ms_max = ms_per_step
    if dist is not None:
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, step_flops * world / (ms_max * 1e-3) / 1e12


def shape_entry(text):
    parts = text.split(",")
    m, n, k = (int(v) for v in parts[:3])
    dtype = parts[3] if len(parts) > 3 else "bf16"
    out = parts[4] if len(parts) > 4 else "bf16"
    return (dtype, m, n, k, out, {"fp8": "fp8", "mxfp4": "mx", "w4a8": "w4a8"}.get(dtype, "normal"))


def workload_text(args):
    if args.shape is not None:
        dtype, m, n, k, out, dist = shape_entry(args.shape)
        return f"single GEMM {m}x{n}x{k} {dtype} inputs, {out} C ({dist} draws)"
    return WORKLOAD_TEXT[args.workload]


# ------------------------------------------------------------------ GPU arm
def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    import dense_gemm_linear_gb300 as dgl
    from dense_gemm_linear_gb300 import _build
    if not os.path.exists(dgl.LIB_PATH):
        _build.build()
    lib = dgl.load_library()
    from synthetic import WORKLOADS, make_workload_case

    entries = WORKLOADS[args.workload] if args.shape is None else [shape_entry(args.shape)]
    cases = [make_workload_case(e) for e in entries]
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    s_handle = stream.cuda_stream

    ops = []
    for c in cases:
        if c.dtype == "bf16":
            # MN-major operands are stored transposed ([K][m], [K][n])
            a_host = c.A if c.a_major == 0 else np.ascontiguousarray(c.A.T)
            b_host = c.B if c.b_major == 0 else np.ascontiguousarray(c.B.T)
            A = torch.from_numpy(a_host.view(np.int16)).to(dev)
            B = torch.from_numpy(b_host.view(np.int16)).to(dev)
            sa = sb = None
        else:
            A = torch.from_numpy(c.A).to(dev)
            B = torch.from_numpy(c.B).to(dev)
            sa = torch.from_numpy(c.sa).to(dev)
            sb = torch.from_numpy(c.sb).to(dev)
        out_dtype = dgl.OUT_F32 if c.out == "f32" else dgl.OUT_BF16
        C = torch.empty((c.m, c.n), dtype=torch.float32 if c.out == "f32" else torch.bfloat16, device=dev)
        bias = torch.from_numpy(c.bias).to(dev) if c.bias is not None else None
        ops.append((c, A, B, sa, sb, C, out_dtype, bias))

    forced = None
    if args.tile is not None:
        tm_, tn_ = (int(v) for v in args.tile.lower().split("x"))
        forced = dgl.PlanInfo(path=dgl.PATH_TC, tile_m=tm_, tile_n=tn_)

    def make_call(c, A, B, sa, sb, C, out_dtype, bias):
        if c.a_major or c.b_major:
            args_ = (c.a_major, c.b_major, A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1], C.data_ptr(), c.n,
                     c.m, c.n, c.K, out_dtype, ctypes.byref(forced) if forced is not None else None, s_handle)
            fn = lib.dgl_gemm_bf16_ex
        elif c.linear:
            dt = dgl.DTYPE_BF16 if c.dtype == "bf16" else dgl.DTYPE_E4M3
            args_ = (dt, A.data_ptr(), B.data_ptr(), sa.data_ptr() if sa is not None else None,
                     sb.data_ptr() if sb is not None else None, bias.data_ptr() if bias is not None else None,
                     C.data_ptr(), c.m, c.n, c.K, c.m, c.n, out_dtype, c.act, int(c.gated),
                     ctypes.byref(forced) if forced is not None else None, s_handle)
            fn = lib.dgl_linear
        elif forced is not None:
            dt = {"bf16": dgl.DTYPE_BF16, "fp8": dgl.DTYPE_E4M3, "w4a8": dgl.DTYPE_W4A8}[c.dtype]
            args_ = (dt, A.data_ptr(), B.data_ptr(), sa.data_ptr() if sa is not None else None,
                     sb.data_ptr() if sb is not None else None, C.data_ptr(), c.m, c.n, c.K, c.m, c.n, out_dtype,
                     ctypes.byref(forced), s_handle)
            fn = lib.dgl_gemm_planned
        elif c.dtype == "w4a8":
            args_ = (A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), c.m, c.n, c.K, c.m,
                     c.n, out_dtype, s_handle)
            fn = lib.dgl_gemm_w4a8
        elif c.dtype == "mxfp4":
            args_ = (A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), c.m, c.n, c.K, c.m,
                     c.n, out_dtype, s_handle)
            fn = lib.dgl_gemm_mxfp4
        elif c.dtype == "bf16":
            args_ = (A.data_ptr(), B.data_ptr(), C.data_ptr(), c.m, c.n, c.K, c.m, c.n, out_dtype, s_handle)
            fn = lib.dgl_gemm_bf16
        else:
            args_ = (A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), c.m, c.n, c.K, c.m,
                     c.n, out_dtype, s_handle)
            fn = lib.dgl_gemm_fp8

        def call(s=s_handle):
            st = fn(*args_[:-1], s)
            if st != 0:
                raise RuntimeError(f"GEMM {c.name} failed: {dgl.status_string(st)}")
        return call

    calls = [make_call(*o) for o in ops]
    dtype_ids = {"bf16": dgl.DTYPE_BF16, "fp8": dgl.DTYPE_E4M3, "mxfp4": dgl.DTYPE_MXFP4, "w4a8": dgl.DTYPE_W4A8}

    def make_desc(c, A, B, sa, sb, C, out_dtype, bias):
        """The GEMM as a dgl_gemm_batch item, or None where the batch call has no
        field for it (linear epilogue, operand layouts, a forced plan)."""
        if forced is not None or c.linear or c.a_major or c.b_major:
            return None
        return dgl.GemmDesc(dtype=dtype_ids[c.dtype], out_dtype=out_dtype, A=A.data_ptr(), B=B.data_ptr(),
                            scale_a=sa.data_ptr() if sa is not None else None,
                            scale_b=sb.data_ptr() if sb is not None else None, C=C.data_ptr(),
                            M=c.m, N=c.n, K=c.K, m_valid=c.m, n_valid=c.n)

    # The step's GEMMs are independent (no GEMM reads another's C), so they go
    # out as one dgl_gemm_batch: each kernel after the first loads its operands
    # while the previous one finishes.  Workloads with fused epilogues or
    # operand layouts the batch call does not take run as single calls.
    descs = [make_desc(*o) for o in ops]
    batched = all(d is not None for d in descs)
    if batched:
        desc_arr = dgl.gemm_descs(descs)

        def step_call(s=s_handle):
            st = lib.dgl_gemm_batch(desc_arr, len(desc_arr), s)
            if st != 0:
                raise RuntimeError(f"batch failed: {dgl.status_string(st)}")
    else:
        def step_call(s=s_handle):
            for f in calls:
                f(s)
    plans = [dgl.dgl_plan_linear(dtype_ids[c.dtype], c.m, c.n, c.K,
                                 dgl.OUT_F32 if c.out == "f32" else dgl.OUT_BF16, int(c.gated)) if c.linear else
             dgl.dgl_plan(dtype_ids[c.dtype], c.m, c.n, c.K,
                          dgl.OUT_F32 if c.out == "f32" else dgl.OUT_BF16) for c in cases]
    if forced is not None:
        plans = [forced for _ in cases]

    def kernel_name(c, p):
        """Kernel variant as ncu lists it: tile and C-store path (C is a contiguous
        torch tensor, so its pitch alone decides the path)."""
        if p.path == dgl.PATH_DECODE:
            return f"decode_gemm_kernel<{c.dtype}>"
        out_bytes = 4 if c.out == "f32" else 2
        if (c.n * out_bytes) % 16 == 0:
            store = "tma-store"
        else:
            store = "predicated" if c.out == "f32" else "row-staging"
        epi = ", linear" if c.linear else ""
        if c.a_major or c.b_major:
            epi = f", {'mn' if c.a_major else 'k'}-{'mn' if c.b_major else 'k'} major"
        return f"tc_gemm_kernel<{c.dtype}, {p.tile_m}x{p.tile_n}, {store}{epi}>"

    knames = [kernel_name(c, p) for c, p in zip(cases, plans)]
    flops = [float(c.flops) for c in cases]
    nbytes = []
    for c in cases:
        o = 4 if c.out == "f32" else 2
        if c.dtype == "mxfp4":
            # the GEMM guide's MXFP4 formula (section 8.2), with C at its own element size
            nbytes.append((c.m + c.n) * c.K // 2 + c.m * c.n * o + (c.m + c.n) * (c.K // 32))
            continue
        if c.dtype == "w4a8":
            # the guide's 4-bit weight formula (section 8.2): A one byte, B half a byte per element
            nbytes.append(c.m * c.K + c.n * c.K // 2 + c.m * c.n * o + 4 * (c.m + c.n))
            continue
        e = 2 if c.dtype == "bf16" else 1
        nbytes.append(c.m * c.K * e + c.b_rows * c.K * e + c.m * c.n * o +
                      (4 * (c.m + c.b_rows) if c.dtype == "fp8" else 0) + (4 * c.b_rows if c.bias is not None else 0))

    # warm-up
    for _ in range(args.warmup):
        step_call()
    torch.cuda.synchronize()
    st = lib.dgl_device_status(s_handle)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {dgl.status_string(st)}")

    # One step captured as a CUDA graph: the ten calls' host work (argument
    # checks, plan and tensor-map cache look-ups, launch) then leaves the timed
    # loop, which replays the same launches back to back.  Capture needs a
    # stream of its own; one step on it first gives a split schedule its
    # workspace there.  The graph is replayed on the timing stream.
    cap_stream = torch.cuda.Stream(device=dev)
    step_call(cap_stream.cuda_stream)
    torch.cuda.synchronize()
    step_graph = capture_graph(torch, step_call, cap_stream)
    launch_mode = ("cuda graph of one step" if step_graph is not None else "stream launches") + \
        (", one dgl_gemm_batch" if batched else ", one call per GEMM")

    # ---------------------------------------------------------- device-timed region
    # Pass 1 times whole steps (the reported value): the calls go back to back,
    # so each kernel's launch and set-up can overlap the previous kernel's end
    # (programmatic dependent launch).  Pass 2 replays the same steps as a graph
    # with an event node between calls, which serialises them: each call's
    # duration with its own launch and ramp-up (reported as "serialised"); the
    # events sit in the graph, so the host's launch gaps stay out.
    K_steps = args.steps
    ncall = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ncall + 1)] for _ in range(K_steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(K_steps):
        if step_graph is not None:
            step_graph.replay()
        else:
            step_call()
    t_end.record(stream)
    barrier()
    # the same step as one call per GEMM, for comparison (not the reported value)
    ms_single_calls = None
    if batched:
        single_graph = capture_graph(torch, lambda s: [f(s) for f in calls], cap_stream)
        if single_graph is not None:
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for s in range(K_steps):
                single_graph.replay()
            u1.record(stream)
            torch.cuda.synchronize()
            ms_single_calls = u0.elapsed_time(u1) / K_steps
            del single_graph
    timing_graph = timed_calls_graph(torch, calls, cap_stream, K_steps)
    if timing_graph is not None:
        evs, tg = timing_graph
        tg.replay()
    else:
        for s in range(K_steps):
            ev = evs[s]
            ev[0].record(stream)
            for i, f in enumerate(calls):
                f()
                ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    st = lib.dgl_device_status(s_handle)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {dgl.status_string(st)}")
    total_ms = t_start.elapsed_time(t_end)
    ms_per_step = total_ms / K_steps
    per_call_ms = [0.0] * ncall
    for s in range(K_steps):
        for i in range(ncall):
            per_call_ms[i] += evs[s][i].elapsed_time(evs[s][i + 1])
    per_call_ms = [v / K_steps for v in per_call_ms]
    ms_per_step_events = sum(per_call_ms)
    call_timing = "graph with an event node between calls" if timing_graph is not None else \
        "stream launches with an event between calls"

    step_flops = sum(flops)
    ms_max, value = over_ranks(ms_per_step, step_flops, dist, dev)

    # ---------------------------------------------------------- headline shapes, each on its own
    pk, pk_src = peaks()
    headline = None
    if not args.no_headline and args.shape is None:
        headline = headline_run(torch, dgl, lib, dev, pk)

    # ---------------------------------------------------------- each GEMM of the step, back to back
    # Every GEMM is also timed on its own as back-to-back launches, the way it
    # runs inside the step, where each launch's set-up overlaps its
    # predecessor's end.  These durations add up to about the step time; the
    # serialised per-call durations above add up to more (each carries its
    # launch and ramp-up), so the per-kernel figures and the roofline use the
    # back-to-back ones and report the serialised ones beside them.
    b2b_ms = [back_to_back_us(torch, make_call, op, dev, make_desc=make_desc if batched else None, lib=lib) * 1e-3
              for op in ops]
    clocks = sampler.stop()
    by_kernel = {}
    for i, kn in enumerate(knames):
        d = by_kernel.setdefault(kn, {"ms": 0.0, "ms_serial": 0.0, "flops": 0.0, "bytes": 0.0, "launches": 0})
        d["ms"] += b2b_ms[i]
        d["ms_serial"] += per_call_ms[i]
        d["flops"] += flops[i]
        d["bytes"] += nbytes[i]
        d["launches"] += 1
    dominant = max(by_kernel, key=lambda k: by_kernel[k]["ms"])
    dk = by_kernel[dominant]

    # ---------------------------------------------------------- context: torch.matmul (cuBLAS), off the measured path
    # Each plain bf16 GEMM of the step is timed once more through torch.matmul
    # on the same device buffers (C = A B^T), back to back with events around
    # 20 calls; E4M3, fused-epilogue and MN-major cases have no such column.
    cublas_us = [None] * ncall
    if not args.no_context:
        for i, (c, A, B, sa, sb, C, _o, bias) in enumerate(ops):
            if c.dtype != "bf16" or c.linear or c.a_major or c.b_major or c.out != "bf16":
                continue
            a_t = A.view(torch.bfloat16)
            b_t = B.view(torch.bfloat16)
            c_t = C
            for _ in range(3):
                torch.matmul(a_t, b_t.t(), out=c_t)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(20):
                torch.matmul(a_t, b_t.t(), out=c_t)
            e1.record(stream)
            torch.cuda.synchronize()
            cublas_us[i] = e0.elapsed_time(e1) / 20 * 1e3

    # ---------------------------------------------------------- roofline of the dominant kernel
    serial = {"timing": "the step replayed with an event between calls: each launch serialised after its "
                        "predecessor, its launch and ramp-up included",
              "avg_launch_us": dk["ms_serial"] * 1e3 / dk["launches"]}
    if dominant.startswith("tc_gemm"):
        # a contraction's peak: the measured bf16 figure times the nominal dense
        # ratio of its own type (E4M3 4.5 / 2.25 PFLOP/s, FP4 13.5 / 2.25)
        ratio, ratio_txt = (6.0, " x6 (fp4 nominal ratio)") if "mxfp4" in dominant else \
            ((2.0, " x2 (fp8 nominal ratio)") if ("fp8" in dominant or "w4a8" in dominant) else (1.0, ""))
        peak_tf = pk["bf16_tflops"] * ratio
        achieved = dk["flops"] / (dk["ms"] * 1e-3) / 1e12
        roofline = {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peak_tf,
                    "unit": "TFLOP/s", "frac": achieved / peak_tf,
                    "traffic": recorded_traffic(args.workload, dominant) if args.shape is None and forced is None
                    else None,
                    "peak_source": f"{pk_src} bf16 burst" + ratio_txt,
                    "launches_per_step": dk["launches"], "avg_launch_us": dk["ms"] * 1e3 / dk["launches"],
                    "algorithmic_flops_per_launch": dk["flops"] / dk["launches"]}
        serial["achieved"] = dk["flops"] / (dk["ms_serial"] * 1e-3) / 1e12
        serial["frac"] = serial["achieved"] / peak_tf
    else:
        achieved = dk["bytes"] / (dk["ms"] * 1e-3) / 1e9
        roofline = {"kernel": dominant, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / pk["hbm_gbs"],
                    "traffic": recorded_traffic(args.workload, dominant) if args.shape is None and forced is None
                    else None,
                    "peak_source": f"{pk_src} hbm copy",
                    "launches_per_step": dk["launches"], "avg_launch_us": dk["ms"] * 1e3 / dk["launches"],
                    "algorithmic_bytes_per_launch": dk["bytes"] / dk["launches"]}
        serial["achieved"] = dk["bytes"] / (dk["ms_serial"] * 1e-3) / 1e9
        serial["frac"] = serial["achieved"] / pk["hbm_gbs"]
    roofline["timing"] = ("each of the kernel's GEMMs alone: 48 back-to-back launches over operand copies rotated "
                          "through more than L2" + (", issued as one dgl_gemm_batch as in the step" if batched else "") +
                          ", replayed as one CUDA graph (CUDA events); the per-GEMM "
                          f"durations of the step add up to {sum(b2b_ms) * 1e3:.1f} us against the "
                          f"{ms_per_step * 1e3:.1f} us step")
    roofline["serialised"] = serial
    kernels = {k: {"launches_per_step": v["launches"], "us_per_step": v["ms"] * 1e3,
                   "share": v["ms"] / sum(x["ms"] for x in by_kernel.values()),
                   "us_per_step_serialised": v["ms_serial"] * 1e3,
                   "share_serialised": v["ms_serial"] / sum(x["ms_serial"] for x in by_kernel.values())}
               for k, v in by_kernel.items()}
    dec = {k: v for k, v in by_kernel.items() if k.startswith("decode")}
    roofline_decode = None
    if dec:
        db = sum(v["bytes"] for v in dec.values())
        dm = sum(v["ms"] for v in dec.values())
        roofline_decode = {"bound": "hbm", "achieved": db / (dm * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                           "unit": "GB/s", "frac": db / (dm * 1e-3) / 1e9 / pk["hbm_gbs"],
                           "peak_source": f"{pk_src} hbm copy"}
    per_shape = []
    for i, c in enumerate(cases):
        t = b2b_ms[i] * 1e-3
        per_shape.append({"shape": [c.m, c.n, c.K], "dtype": c.dtype, "out": c.out, "kernel": knames[i],
                          "epilogue": ({"act": ["none", "gelu", "silu"][c.act], "bias": c.bias is not None,
                                        "gated": c.gated} if c.linear else None),
                          "us": b2b_ms[i] * 1e3, "us_serialised": per_call_ms[i] * 1e3, "tflops": flops[i] / t / 1e12,
                          "gbs": nbytes[i] / t / 1e9, "tile_eff": round(plans[i].tile_eff, 4),
                          "wq_eff": round(plans[i].wq_eff, 4), "grid": plans[i].grid,
                          "torch_matmul_us": cublas_us[i]})

    # ---------------------------------------------------------- end to end through host buffers
    e2e = None
    if args.e2e_steps > 0:
        host = []
        h2d = d2h = 0
        for (c, A, B, sa, sb, C, _o, bias) in ops:
            hA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True).copy_(A.cpu())
            hB = torch.empty(B.shape, dtype=B.dtype, pin_memory=True).copy_(B.cpu())
            hsa = sa.cpu().pin_memory() if sa is not None else None
            hsb = sb.cpu().pin_memory() if sb is not None else None
            hC = torch.empty(C.shape, dtype=C.dtype, pin_memory=True)
            hbias = bias.cpu().pin_memory() if bias is not None else None
            host.append((hA, hB, hsa, hsb, hC, hbias))
            h2d += hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
            if hbias is not None:
                h2d += 4 * hbias.numel()
            if hsa is not None:
                h2d += hsa.element_size() * (hsa.numel() + hsb.numel())
            d2h += hC.numel() * hC.element_size()

        # Pipelined as a caller would: inputs go up on a copy stream, the GEMMs
        # run on the compute stream, results come down on a second copy
        # stream, so one GEMM's copies overlap another's kernel.  Events keep
        # each buffer's reuse in order across steps.
        h2d_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        done = [torch.cuda.Event() for _ in ops]      # compute of op i finished (its inputs free)
        drained = [torch.cuda.Event() for _ in ops]   # D2H of op i's C finished (C free)

        def e2e_step():
            for i, ((c, A, B, sa, sb, C, _o, bias), (hA, hB, hsa, hsb, hC, hbias), f) in enumerate(
                    zip(ops, host, calls)):
                with torch.cuda.stream(h2d_s):
                    h2d_s.wait_event(done[i])
                    A.copy_(hA, non_blocking=True)
                    B.copy_(hB, non_blocking=True)
                    if bias is not None:
                        bias.copy_(hbias, non_blocking=True)
                    if sa is not None:
                        sa.copy_(hsa, non_blocking=True)
                        sb.copy_(hsb, non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(h2d_s)
                stream.wait_event(ready)
                stream.wait_event(drained[i])
                f()
                done[i].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(done[i])
                    hC.copy_(C, non_blocking=True)
                    drained[i].record(d2h_s)

        e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        for _ in range(args.e2e_steps):
            e2e_step()
        for ev in drained:
            stream.wait_event(ev)
        e1.record(stream)
        barrier()
        e2e_ms, e2e_value = over_ranks(e0.elapsed_time(e1) / args.e2e_steps, step_flops, dist, dev)
        e2e = {"value": e2e_value, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": args.e2e_steps}

    # ---------------------------------------------------------- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f_, s_, cores, text = oracle_sample_run(cases, args.cpu_macs)
        cpu = {"value": f_ / s_ / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": text, "seconds": s_}

    if rank == 0:
        l2_mb = torch.cuda.get_device_properties(dev).L2_cache_size / 2**20
        ws = sum(nbytes) / 2**20
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K_steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "+".join(sorted({{"bf16": "bf16", "fp8": "e4m3", "mxfp4": "e2m1", "w4a8": "e4m3xe2m1"}[c.dtype]
                                      for c in cases})),
            "data": "synthetic (seeded SplitMix64 draws)",
            "config": {"workload": workload_text(args), "gemms_per_step": ncall, "launch": launch_mode,
                       "per_call_timing": call_timing,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": (f"inputs larger than L2: {ws:.0f} MiB per step vs {l2_mb:.0f} MiB")
                             if ws > l2_mb else
                             (f"inputs fit in L2 ({ws:.0f} MiB vs {l2_mb:.0f} MiB): a profiling run, "
                              f"not a bench line")},
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": K_steps * ncall, "clocks": clocks,
            "roofline": roofline,
        }
        if ms_single_calls is not None:
            # the same step issued as one call per GEMM (each kernel waits for its
            # predecessor before loading operands), measured right after it
            line["ms_per_step_single_calls"] = ms_single_calls
        detail = dict(line)
        detail.update({"roofline_decode": roofline_decode, "kernels": kernels, "per_shape": per_shape,
                       "ms_per_step_with_call_events": ms_per_step_events, "headline": headline})
        # the full record on stderr; stdout carries one compact line whose
        # tail holds the per-shape times and the headline shapes
        print(json.dumps(detail), file=sys.stderr, flush=True)
        line["cpu_baseline"] = cpu and {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        if cpu:
            line["cpu_baseline"]["sample"] = "first rows of each GEMM of the step"
        line["roofline"] = {k: roofline[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                      "traffic", "peak_source", "avg_launch_us")}
        for k in ("achieved", "frac", "avg_launch_us"):
            line["roofline"][k] = round(line["roofline"][k], 4)
        line["roofline"]["serialised"] = {k: round(roofline["serialised"][k], 4)
                                          for k in ("achieved", "frac", "avg_launch_us")}
        if roofline_decode:
            line["roofline_decode"] = {"achieved": round(roofline_decode["achieved"], 1),
                                       "frac": round(roofline_decode["frac"], 4)}
        line["per_shape_us"] = {f"{c.m}x{c.n}x{c.K}": round(b2b_ms[i] * 1e3, 2) for i, c in enumerate(cases)}
        line["headline"] = compact_headline(headline)
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def compact_headline(headline):
    """The headline block as the stdout line carries it: per shape its time, the
    single-call time, the rate and its fractions of the nominal and measured
    peaks (the full record on stderr keeps every field)."""
    if not headline:
        return headline
    keep = ("us", "us_single_calls", "TFLOP/s", "GB/s", "of_nominal", "of_measured")
    return {shape: {k: rec[k] for k in keep if k in rec} for shape, rec in headline.items()}


def back_to_back_us(torch, make_call, op, dev, launches=48, reps=7, make_desc=None, lib=None):
    """One GEMM of the step on its own: `launches` back-to-back launches over
    ceil(3 L2 / (|A| + |B|)) copies of its operands (each with its own C), so
    every launch reads them from HBM, replayed as one CUDA graph: one
    dgl_gemm_batch of `launches` items when make_desc is given (as the step
    runs), else single calls.  Returns the per-launch time of the median
    replay, in us."""
    import math
    c, A, B, sa, sb, C, o, bias = op
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ab = A.numel() * A.element_size() + B.numel() * B.element_size()
    copies = max(2, math.ceil(3 * l2 / ab))
    # the copies stay referenced here: a call holds raw device pointers only
    bufs = [op] + [(c, A.clone(), B.clone(), sa, sb, torch.empty_like(C), o, bias) for _ in range(copies - 1)]
    calls = [make_call(*x) for x in bufs]
    stream = torch.cuda.Stream(device=dev)
    for f in calls:
        f(stream.cuda_stream)
    torch.cuda.synchronize()
    L = copies * max(1, math.ceil(launches / copies))
    if make_desc is not None:
        import dense_gemm_linear_gb300 as dgl
        arr = dgl.gemm_descs([make_desc(*bufs[t % copies]) for t in range(L)])

        def body(s):
            st = lib.dgl_gemm_batch(arr, L, s)
            if st != 0:
                raise RuntimeError(f"batch failed: {dgl.status_string(st)}")
    else:
        def body(s):
            for t in range(L):
                calls[t % copies](s)
    g = capture_graph(torch, body, stream)
    times = []
    for i in range(reps + 2):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if g is not None:
            with torch.cuda.stream(stream):
                g.replay()
        else:
            body(stream.cuda_stream)
        e1.record(stream)
        e1.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1) * 1e3 / L)
    torch.cuda.synchronize()
    del g, calls, bufs
    torch.cuda.empty_cache()
    return statistics.median(times)


def timed_calls_graph(torch, calls, stream, steps):
    """K steps captured as one CUDA graph with a timing event recorded between
    consecutive calls (event record nodes), so that each call's duration is
    read on the device without the host's launch gaps.  Returns (events, graph),
    or None where events cannot be recorded as graph nodes (the caller then
    times eager launches)."""
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
               for _ in range(steps)]
    except TypeError:
        return None

    def body(handle):
        for ev in evs:
            ev[0].record()
            for i, f in enumerate(calls):
                f(handle)
                ev[i + 1].record()
    g = capture_graph(torch, body, stream)
    return None if g is None else (evs, g)


def capture_graph(torch, body, stream=None):
    """Capture body(stream_handle) into a CUDA graph on `stream` (default: the
    current stream); None if capture fails."""
    stream = stream or torch.cuda.current_stream()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(stream.cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        return g
    except Exception as exc:  # noqa: BLE001 -- any capture failure falls back to stream launches
        print(f"graph capture failed, timing stream launches: {exc}", file=sys.stderr)
        torch.cuda.synchronize()
        return None


# The shapes the targets are stated on, each timed on its own: 4096^3 in bf16
# and E4M3 against the dense tensor peak, and the decode shapes (the LLaMA-2 7B
# up/gate projection at 1 and 16 tokens, 16 x 4096 x 4096) against HBM.
HEADLINE = [("bf16", 4096, 4096, 4096, "bf16", "square_normal"),
            ("fp8", 4096, 4096, 4096, "bf16", "fp8"),
            ("bf16", 1, 11008, 4096, "bf16", "normal"),
            ("bf16", 16, 11008, 4096, "bf16", "normal"),
            ("bf16", 16, 4096, 4096, "bf16", "normal")]
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0}
NOMINAL_HBM_GBS = 8000.0


def headline_run(torch, dgl, lib, dev, pk, launches=48, reps=7):
    """Time each HEADLINE shape alone: its operands rotate through
    ceil(3 L2 / (|A| + |B|)) copies, so every launch reads them from HBM, and
    `launches` back-to-back GEMMs, issued as one dgl_gemm_batch, are replayed
    as one CUDA graph; the same launches as single calls are timed beside them
    (us_single_calls).  Returns {shape: {us, rate, fractions of the nominal and
    measured peaks}}."""
    import math

    from synthetic import make_workload_case
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for entry in HEADLINE:
        c = make_workload_case(entry)
        if c.dtype == "bf16":
            A = torch.from_numpy(c.A.view("int16")).to(dev)
            B = torch.from_numpy(c.B.view("int16")).to(dev)
            sa = sb = None
            e = 2
        else:
            A = torch.from_numpy(c.A).to(dev)
            B = torch.from_numpy(c.B).to(dev)
            sa = torch.from_numpy(c.sa).to(dev)
            sb = torch.from_numpy(c.sb).to(dev)
            e = 1
        ab = (c.m + c.n) * c.K * e
        copies = max(2, math.ceil(3 * l2 / ab))
        As = [A] + [A.clone() for _ in range(copies - 1)]
        Bs = [B] + [B.clone() for _ in range(copies - 1)]
        Cs = [torch.empty((c.m, c.n), dtype=torch.bfloat16, device=dev) for _ in range(copies)]

        def launch(r, s):
            if c.dtype == "bf16":
                st = lib.dgl_gemm_bf16(As[r].data_ptr(), Bs[r].data_ptr(), Cs[r].data_ptr(), c.m, c.n, c.K, c.m, c.n,
                                       dgl.OUT_BF16, s)
            else:
                st = lib.dgl_gemm_fp8(As[r].data_ptr(), Bs[r].data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                      Cs[r].data_ptr(), c.m, c.n, c.K, c.m, c.n, dgl.OUT_BF16, s)
            if st != 0:
                raise RuntimeError(f"headline {c.name}: {dgl.status_string(st)}")

        # one stream for the warm-up, the capture and the timing events, so a
        # split schedule's workspace exists before the capture
        stream = torch.cuda.Stream(device=dev)
        cur = stream.cuda_stream
        for r in range(copies):
            launch(r, cur)
        torch.cuda.synchronize()
        L = copies * max(1, math.ceil(launches / copies))
        # the same L GEMMs as one dgl_gemm_batch: independent, so each kernel
        # loads its operands while the previous one finishes
        arr = dgl.gemm_descs([dict(dtype=dgl.DTYPE_BF16 if c.dtype == "bf16" else dgl.DTYPE_E4M3,
                                   out_dtype=dgl.OUT_BF16, A=As[t % copies].data_ptr(), B=Bs[t % copies].data_ptr(),
                                   scale_a=sa.data_ptr() if sa is not None else None,
                                   scale_b=sb.data_ptr() if sb is not None else None, C=Cs[t % copies].data_ptr(),
                                   M=c.m, N=c.n, K=c.K, m_valid=c.m, n_valid=c.n) for t in range(L)])

        def batch(s):
            st = lib.dgl_gemm_batch(arr, L, s)
            if st != 0:
                raise RuntimeError(f"headline {c.name}: {dgl.status_string(st)}")

        def timed(body):
            g = capture_graph(torch, body, stream)
            times = []
            for i in range(reps + 2):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if g is not None:
                    with torch.cuda.stream(stream):
                        g.replay()
                else:
                    body(cur)
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    times.append(e0.elapsed_time(e1) * 1e3 / L)
            return statistics.median(times)

        us = timed(batch)
        us_single = timed(lambda s: [launch(t % copies, s) for t in range(L)])
        key = f"{c.m}x{c.n}x{c.K} {'e4m3' if c.dtype == 'fp8' else 'bf16'}"
        plan = dgl.dgl_plan(dgl.DTYPE_BF16 if c.dtype == "bf16" else dgl.DTYPE_E4M3, c.m, c.n, c.K)
        rec = {"us": round(us, 2), "us_single_calls": round(us_single, 2), "copies": copies,
               "tile": "decode" if plan.path == dgl.PATH_DECODE else f"{plan.tile_m}x{plan.tile_n}"}
        if c.m > 16:
            tf = 2.0 * c.m * c.n * c.K / (us * 1e-6) / 1e12
            meas = pk["bf16_tflops"] * (2.0 if c.dtype == "fp8" else 1.0)
            rec.update({"TFLOP/s": round(tf, 1), "of_nominal": round(tf / NOMINAL_TFLOPS[c.dtype], 4),
                        "of_measured": round(tf / meas, 4), "target_of_nominal": 0.70})
        else:
            nb = (c.m * c.K + c.n * c.K) * e + c.m * c.n * 2 + (4 * (c.m + c.n) if c.dtype == "fp8" else 0)
            gbs = nb / (us * 1e-6) / 1e9
            rec.update({"GB/s": round(gbs, 1), "of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                        "of_measured": round(gbs / pk["hbm_gbs"], 4), "target_of_nominal": 0.60})
        out[key] = rec
        del arr, As, Bs, Cs, A, B
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    sys.exit(main())
