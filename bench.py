#!/usr/bin/env python
"""Benchmark of the tiled FP32 matrix multiply C = A.B on GB300.

One step = one sgemm_f32_ws call over the workload (the whole path: argument
checks, the schedule choice, the operand copies that pay -- at 4096^3 the
transpose of A into its k-major copy --, the product kernels with their copy
pipelines, FMA main loops, split fix-up where used, and epilogues; the
workspace is allocated once, outside the timed region).
Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME | --shape M,N,K]
                  [--impl ours|reference]
  python bench.py --op transpose [--rows R --cols C] [--layout fast|padded|unpadded|swizzled]

Timing: inputs resident in HBM; before every timed step the L2 is flushed by
writing a 256 MiB buffer (outside the step's events); each step is bracketed
by CUDA events on the launching stream.  ms_per_step is the mean over the K
steps, max over ranks.  N > 1 runs independent replicas (one full product per
GPU, no collective on the data path): value = total FLOP / max time.

--impl reference times the FP64 CPU oracle (the only baseline this path has)
on the host cores, each step a bounded row-block sample of the same product.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP32 GEMM TFLOP/s at M=N=K=4096 and % of GB300 FP32 CUDA-core peak"
FMA_PER_CLK_PER_SM = 128  # FP32 CUDA-core lanes per SM (4 partitions x 32)


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--shape", default=None,
                    help="M,N,K: a dense product with uniform[-1,1] inputs from seed 0 instead of a named workload "
                         "(for profiling other shapes)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-tc", action="store_true", help="skip the tensor-core 3xTF32 variant")
    ap.add_argument("--clocks-csv", default=None, help="keep the raw nvidia-smi samples in this file")
    ap.add_argument("--op", choices=["gemm", "transpose"], default="gemm",
                    help="gemm: the FP32 product (default); transpose: the FP32 transpose workload")
    ap.add_argument("--rows", type=int, default=8192, help="transpose: input rows")
    ap.add_argument("--cols", type=int, default=8192, help="transpose: input cols")
    ap.add_argument("--layout", choices=["fast", "padded", "unpadded", "swizzled"], default="fast",
                    help="transpose: kernel (fast = transpose_f32, else the 32x32 tile kernel's layout)")
    return ap.parse_args()


def _measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def _workload(name, shape=None):
    from dense_fp32_tiled_gb300 import synth
    if shape:
        M, N, K = (int(x) for x in shape.split(","))
        return synth.Workload(f"sgemm_{M}x{N}x{K}_uniform", M, N, K, K, N, N, "uniform", 1.0, 0, (0, 1), "full")
    return synth.WORKLOADS[name or synth.HEADLINE]


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""
    Q = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, path: str | None = None):
        self.uuid = uuid
        self.proc = None
        self.t0 = self.t1 = None  # wall-clock bounds of the timed region
        self.path = path or os.path.join(tempfile.gettempdir(), f"sgemm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows, inside = [], []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                rows.append(parts)
                try:
                    t = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    t += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                except (ValueError, IndexError):
                    t = None
                if t is not None and self.t0 is not None and self.t0 - 0.15 <= t <= self.t1 + 0.15:
                    inside.append(parts)
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[2]) for r in use) if v is not None]
        mx = [v for v in (num(r[3]) for r in use) if v is not None]
        pw = [v for v in (num(r[4]) for r in use) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "power_w_max": max(pw) if pw else None,
                "samples": len(use), "samples_in_timed_region": len(inside)}


def _traffic(key: str):
    """DRAM bytes per launch recorded in profiles/dram_traffic.json for one
    benchmarked kernel, if it was captured on the kernel as built now (same
    source stamp); else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get("entries", {}).get(key)
    if not e:
        return None
    from dense_fp32_tiled_gb300 import build as lib_build
    if lib_build.kernel_stamp(e["sources"]) != e.get("source_stamp"):
        return None
    return int(e["dram_bytes_per_launch"])


def cpu_baseline(w, seconds: float):
    """Time the FP64 oracle as it stands on a row-block sample of the product."""
    import numpy as np
    import oracle
    from dense_fp32_tiled_gb300 import synth
    oracle.build()
    A = synth.matrix(w.M, w.K, w.seed, w.ids[0], w.kind, w.sigma)
    B = synth.matrix(w.K, w.N, w.seed, w.ids[1], w.kind, w.sigma)
    probe = max(1, min(w.M, 8))
    t0 = time.perf_counter()
    oracle.gemm(A[:probe], B, with_abs=False)
    t_probe = time.perf_counter() - t0
    rows = int(max(1, min(w.M, probe * seconds / max(t_probe, 1e-6))))
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, with_abs=False)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product (all N, all K), FP64 "
                      f"i-k-j loops, {dt:.1f} s"}, rows


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from dense_fp32_tiled_gb300 import synth
    w = _workload(a.workload, a.shape)
    oracle.build()
    A = synth.matrix(w.M, w.K, w.seed, w.ids[0], w.kind, w.sigma)
    B = synth.matrix(w.K, w.N, w.seed, w.ids[1], w.kind, w.sigma)
    total_budget = 150.0
    per_step = total_budget / max(1, a.steps + a.warmup)
    probe = max(1, min(w.M, 4))
    t0 = time.perf_counter()
    oracle.gemm(A[:probe], B, with_abs=False)
    t_probe = time.perf_counter() - t0
    rows = int(max(1, min(w.M, probe * per_step / max(t_probe, 1e-6))))
    for _ in range(a.warmup):
        oracle.gemm(A[:rows], B, with_abs=False)
    times = []
    for _ in range(a.steps):
        t0 = time.perf_counter()
        oracle.gemm(A[:rows], B, with_abs=False)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    flops = 2.0 * rows * w.N * w.K
    value = flops / (ms / 1e3) / 1e12
    sample = f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product per step (all N, all K)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, a.gpus, "host cores, no L2 flush"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def combine_ranks(ms: float, flops: float, world: int, device=None):
    """Replica timing across ranks: the slowest rank's ms per step, and the
    whole-job throughput (world x FLOP per step / that time) in TFLOP/s.

    Each rank runs the full product on its own GPU; the only cross-rank
    operation is this max-reduction of a scalar (no data-path collective).
    """
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * flops / (ms / 1e3) / 1e12


def _config(w, n, l2):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "lda": w.lda, "ldb": w.ldb, "ldc": w.ldc,
            "inputs": f"{w.kind}{'' if w.kind != 'normal' else f'(0,{w.sigma})'} seed {w.seed}",
            "l2": l2, "parallelism": "replicas" if n > 1 else "single GPU"}


def run_transpose(a):
    """FP32 transpose out = in^T: bytes moved (read + write) per second."""
    import torch
    import dense_fp32_tiled_gb300 as sg
    from dense_fp32_tiled_gb300 import build as lib_build
    from dense_fp32_tiled_gb300 import synth
    lib_build.build()
    sg.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    rows, cols = a.rows, a.cols
    x_h = synth.matrix(rows, cols, 61, 0)
    x = torch.from_numpy(x_h).to(dev)
    y = torch.empty((cols, rows), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    layout = None if a.layout == "fast" else a.layout

    def step():
        st = sg.transpose_f32(rows, cols, x.data_ptr(), cols, y.data_ptr(), rows, stream.cuda_stream, layout=layout)
        if st != 0:
            raise RuntimeError(sg.transpose_status_string(st))
    for _ in range(a.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    with ClockSampler(uuid, a.clocks_csv) as clk:
        torch.cuda.synchronize(dev)
        clk.t0 = time.time()
        for i in range(a.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        clk.t1 = time.time()
    ms = statistics.mean(st.elapsed_time(en) for st, en in zip(starts, ends))
    nbytes = 2.0 * 4 * rows * cols
    gbs = nbytes / (ms / 1e3) / 1e9
    peak = float(_measured_peaks().get("hbm_gbs") or 6800.0)
    # DRAM bytes per launch from the committed ncu summary (taken on the 8192 x 8192 vector path)
    traffic = _traffic("transpose_f32_8192") if a.layout == "fast" and (rows, cols) == (8192, 8192) else None
    line = {"metric": "FP32 transpose GB/s (bytes read + written)", "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"transpose_{rows}x{cols}", "rows": rows, "cols": cols, "kernel": a.layout,
                       "inputs": "uniform seed 61", "l2": "flushed before every timed step"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": traffic, "peak_basis": "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"},
            "gpu_launches": a.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    a = _args()
    if a.impl == "reference":
        run_reference(a)
        return
    if a.op == "transpose":
        run_transpose(a)
        return
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from dense_fp32_tiled_gb300 import build as lib_build
    if rank == 0:
        lib_build.build()
    if world > 1:
        dist.barrier()
    import dense_fp32_tiled_gb300 as sg
    from dense_fp32_tiled_gb300 import synth
    sg.load_library()

    w = _workload(a.workload, a.shape)
    dev = torch.device("cuda", local)
    A_h, B_h = w.inputs(ld_buffers=True)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    c_elems = (w.M - 1) * w.ldc + w.N
    C = torch.empty(c_elems, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    # the library's balanced entry point, with the workspace it asks for
    # (for these operands: room for the copies that pay -- the k-major copy of
    # A at large N, repacked rows where they are not 16-byte aligned)
    ws_bytes = sg.workspace_size_for(w.M, w.N, w.K, A.data_ptr(), w.lda, B.data_ptr(), w.ldb)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step():
        st = sg.sgemm_f32_ws(w.M, w.N, w.K, A.data_ptr(), w.lda, B.data_ptr(), w.ldb, C.data_ptr(), w.ldc,
                             ws.data_ptr(), ws_bytes, s)
        if st != 0:
            raise sg.SgemmError(st)
    # kernels of ours per step: schedule 3 runs a one-CTA-per-tile grid and a
    # split-tail grid, the others (bit 32, the cluster split of K, included)
    # one grid; each copied operand (bits 4, 8: rows repacked; 16: A
    # transposed into its k-major copy) adds its copy kernel
    _, sched_kind, _ = sg.ws_schedule(w.M, w.N, w.K, A.data_ptr(), w.lda, B.data_ptr(), w.ldb, C.data_ptr(), w.ldc,
                                      ws_bytes)
    kernels_per_step = ((2 if sched_kind & 3 == 3 else 1) + bool(sched_kind & 4) + bool(sched_kind & 8)
                        + bool(sched_kind & 16))

    for _ in range(a.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    with ClockSampler(uuid, a.clocks_csv) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        clk.t0 = time.time()
        t_wall = time.perf_counter()
        torch.cuda.nvtx.range_push("bench: timed steps (sgemm_f32_ws)")
        for i in range(a.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall
        clk.t1 = time.time()
    times = [st.elapsed_time(en) for st, en in zip(starts, ends)]
    flops = float(w.flops)
    ms, value = combine_ranks(statistics.mean(times), flops, world, dev)
    clocks = clk.summary()

    # ---- end to end through the host-buffer entry point: pinned host A, B ->
    # device -> product -> pinned host C, every step (sgemm_f32_host overlaps
    # the row-panel copies of one call with its products)
    e2e = None
    if not a.no_e2e:
        hA = torch.from_numpy(A_h).pin_memory()
        hB = torch.from_numpy(B_h).pin_memory()
        hC = torch.empty(c_elems, dtype=torch.float32).pin_memory()
        h_bytes = sg.host_workspace_size(w.M, w.N, w.K)
        h_ws = torch.empty(h_bytes, dtype=torch.uint8, device=dev)

        def host_step():
            st = sg.sgemm_f32_host(w.M, w.N, w.K, hA.data_ptr(), w.lda, hB.data_ptr(), w.ldb, hC.data_ptr(), w.ldc,
                                   h_ws.data_ptr(), h_bytes, s)
            if st != 0:
                raise sg.SgemmError(st, "sgemm_f32_host")
        e_steps = max(3, min(50, a.steps // 2))
        for _ in range(2):
            host_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        torch.cuda.nvtx.range_push("bench: end-to-end steps (sgemm_f32_host)")
        for _ in range(e_steps):
            host_step()
        torch.cuda.nvtx.range_pop()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms, e_value = combine_ranks(e0.elapsed_time(e1) / e_steps, flops, world, dev)
        e2e = {"value": e_value, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(A_h.nbytes + B_h.nbytes), "d2h_bytes_per_step": int(c_elems * 4),
               "ms_per_step": e_ms, "entry_point": "sgemm_f32_host (pinned host buffers)"}

    # ---- roofline: FP32 FMA pipe of all SMs
    peaks = _measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2070.0)
    sms = props.multi_processor_count
    peak = sms * FMA_PER_CLK_PER_SM * 2 * sm_max * 1e6 / 1e12
    achieved = flops / (ms / 1e3) / 1e12 if world == 1 else value / world
    # the committed DRAM counters were captured on the 4096^3 product only
    headline = w.name == synth.HEADLINE
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": _traffic("sgemm_f32_4096") if headline else None,
                "peak_basis": f"{sms} SMs x 128 FP32 FMA/clk x 2 FLOP x {sm_max:.0f} MHz (max SM clock)"}
    if sched_kind & 3 == 3:
        dp, tail = (("sgemm_f32_kmajor_kernel", "sgemm_f32_kmajor_tail_kernel") if sched_kind & 16 else
                    ("sgemm_f32_tiled_kernel", "sgemm_f32_tail_kernel"))
        roofline["kernels"] = (f"{dp} (whole waves) + {tail} (leftover tiles in K parts), overlapped; achieved and "
                               "traffic cover the whole step")
    if sched_kind & 32:
        roofline["kernels"] = ("sgemm_f32_clusterk_kernel: clusters of CTAs split each tile's K, partial sums added "
                               "through distributed shared memory; achieved covers the whole step")
    if sched_kind & 12:
        roofline["repack"] = ("repack_rows_kernel copies " + " and ".join(
            n for n, bit in (("A", 4), ("B", 8)) if sched_kind & bit) +
            " into 16-byte aligned rows first, inside the timed step")
    if sched_kind & 16:
        roofline["kmajor_copy"] = ("transpose_f32 writes A^T into the workspace first, inside the timed step "
                                   "(achieved counts the step's whole time); the product kernels then load "
                                   "k-major A tiles and store nothing to shared memory")
    if clocks.get("sm_mhz"):
        roofline["frac_at_sampled_clock"] = achieved / (peak * clocks["sm_mhz"] / sm_max)

    # ---- the tensor-core 3xTF32 variant of the same product (same inputs,
    # same timing protocol); reported beside the CUDA-core path
    tc = None
    if not a.no_tc:
        tc_bytes = sg.tc_workspace_size(w.M, w.N, w.K)
        tc_ws = torch.empty(max(tc_bytes, 256), dtype=torch.uint8, device=dev)

        def tc_step():
            st = sg.sgemm_f32_3xtf32(w.M, w.N, w.K, A.data_ptr(), w.lda, B.data_ptr(), w.ldb, C.data_ptr(),
                                     w.ldc, tc_ws.data_ptr(), tc_bytes, s)
            if st != 0:
                raise sg.SgemmError(st, "sgemm_f32_3xtf32")
        for _ in range(a.warmup):
            flush.zero_()
            tc_step()
        tc_steps = max(3, min(a.steps, 200))
        t_starts = [torch.cuda.Event(enable_timing=True) for _ in range(tc_steps)]
        t_ends = [torch.cuda.Event(enable_timing=True) for _ in range(tc_steps)]
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_push("bench: tensor-core variant steps (sgemm_f32_3xtf32)")
        for i in range(tc_steps):
            flush.zero_()
            t_starts[i].record(stream)
            tc_step()
            t_ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        tc_ms, tc_value = combine_ranks(statistics.mean(x.elapsed_time(y) for x, y in zip(t_starts, t_ends)),
                                        flops, world, dev)
        tf32_peak = float(peaks.get("bf16_tflops") or 1895.4) * 1.1 / 2.25
        tc_achieved = 3.0 * flops / (tc_ms / 1e3) / 1e12
        tc = {"value": tc_value, "unit": "TFLOP/s", "ms_per_step": tc_ms, "steps": tc_steps,
              "entry_point": "sgemm_f32_3xtf32 (split pre-pass + tcgen05 kind::tf32 MMA kernel; timed together)",
              "gpu_launches": 2 * tc_steps,
              "roofline": {"bound": "tensor", "achieved": tc_achieved, "peak": tf32_peak, "unit": "TFLOP/s",
                           "frac": tc_achieved / tf32_peak,
                           "traffic": _traffic("sgemm_3xtf32_4096") if headline else None,
                           "peak_basis": "TF32 dense = measured bf16 burst x 1.1/2.25 (nominal ratio); "
                                         "achieved counts the 3 TF32 products per FP32 product"}}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu, _ = cpu_baseline(w, a.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": _config(w, world, "flushed before every timed step (256 MiB write, outside the events)"),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": kernels_per_step * a.steps,
                "clocks": clocks, "pct_of_fp32_peak": 100.0 * achieved / peak, "tensor_core_variant": tc,
                "ms_min": min(times), "ms_max": max(times), "wall_s_timed_region": t_wall}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
