"""Benchmark of the SpGEMM library: C = A * A on a seeded R-MAT matrix (scale 18, edge factor
16, Graph500 quadrant probabilities, fp64 values U[0,1)), one GPU per process.

One step = one whole product through the library (create: planner, IP count and binning;
symbolic; caller allocation of C; numeric; destroy), inputs resident in HBM.  The metric is
GFLOP/s = 2 x intermediate products / time, plus the fraction of the HBM roofline of the
compulsory bytes (A, the rows of B that are touched, and C).  L2 is flushed between timed steps
by writing a 512 MiB buffer outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1..5]

`--impl reference` times the CPU oracle (ordered-map Gustavson) on the host cores on a bounded
sample of the same rows.  Under torchrun each rank runs its own replica (the product does not
need a second GPU); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SpGEMM GFLOP/s (2 x intermediate products / s), 1 x GB300"
UNIT = "GFLOP/s"


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest value over the ranks (the slowest replica's time); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ip_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job GFLOP/s: every rank's replica does 2 * IP flops per step."""
    return 2.0 * ip_per_step * steps * world / seconds / 1e9


def compulsory_bytes(A, B, c_nnz: int) -> int:
    """bytes(A) + bytes(rows of B that A touches) + bytes(C); bytes(X) = (rows+1)*8 + 12*nnz."""
    touched = np.zeros(B.rows, dtype=bool)
    touched[A.col] = True
    b_nnz = int(np.diff(B.row_ptr)[touched].sum())
    return (A.rows + 1) * 8 + 12 * A.nnz + (B.rows + 1) * 8 + 12 * b_nnz + (A.rows + 1) * 8 + 12 * c_nnz


KERNEL_OF = {"outer_product": "k_outer_product", "histogram": "k_histogram", "multisplit": "k_multisplit",
             "chunk_symbolic": "k_chunk", "chunk_dense": "k_chunk_dense"}


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of this workload, or None
    when there is none or the kernel's source file changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_%s.md" % workload.replace("rmat_s18_ef16", "rmat_s18"))
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) == 5 and parts[0] == "traffic" and parts[1] == kernel:
            kv = dict(x.split("=", 1) for x in parts[2:])
            src = os.path.join(ROOT, "sparse_gemm_irregular_gb300", "csrc", kv["source"])
            if not os.path.exists(src):
                return None
            if hashlib.sha1(open(src, "rb").read()).hexdigest()[:12] != kv["sha1"]:
                return None
            return int(kv["bytes"])
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def sample_rows_by_ip(A, B, ip_budget: float, seed: int = 0):
    """Seeded uniform row sample whose intermediate products add up to about ip_budget."""
    import oracle
    ip = oracle.row_ip(A, B)
    order = np.argsort(synth.draws(seed, synth.STREAM_SAMPLE, 0, A.rows), kind="stable")
    cum = np.cumsum(ip[order])
    k = int(np.searchsorted(cum, ip_budget)) + 1
    rows = np.sort(order[:max(1, min(k, A.rows))])
    return rows, int(ip[rows].sum())


def oracle_rate(A, B, seconds: float, threads: int):
    """Time the oracle (as it stands) on a row sample sized to about `seconds` of work."""
    import oracle
    rows, ipn = sample_rows_by_ip(A, B, 2e6)
    t0 = time.perf_counter()
    oracle.spgemm_rows(A, B, rows, threads=threads)
    dt = time.perf_counter() - t0
    rate = ipn / max(dt, 1e-6)
    for attempt in range(2):
        rows, ipn = sample_rows_by_ip(A, B, rate * seconds, seed=1 + attempt)
        t0 = time.perf_counter()
        oracle.spgemm_rows(A, B, rows, threads=threads)
        dt = time.perf_counter() - t0
        if dt >= 0.6 * seconds:
            break
        rate = ipn / max(dt, 1e-6)
    return 2.0 * ipn / dt / 1e9, len(rows), ipn, dt


def run_reference(args, A, cfg_name, rank):
    """CPU oracle on the host cores: each step is a bounded row sample of the workload."""
    if rank != 0:
        return
    import oracle
    threads = os.cpu_count() or 1
    _, _, ipn0, _ = None, None, None, None
    # size each step to about 4 s of oracle work on all cores
    rows, ipn = sample_rows_by_ip(A, A, 2e6)
    t0 = time.perf_counter()
    oracle.spgemm_rows(A, A, rows, threads=threads)
    rate = ipn / max(time.perf_counter() - t0, 1e-6)
    rows, ipn = sample_rows_by_ip(A, A, rate * 4.0, seed=1)
    for _ in range(args.warmup):
        oracle.spgemm_rows(A, A, rows[: max(1, len(rows) // 8)], threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.spgemm_rows(A, A, rows, threads=threads)
    dt = time.perf_counter() - t0
    value = 2.0 * ipn * args.steps / dt / 1e9
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg_name, "rows_per_step": len(rows),
                                        "ip_per_step": ipn},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "%d seeded uniform rows (%d intermediate products) per step"
                                   % (len(rows), ipn)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# Algorithmic bytes per element of the kernels that can dominate (the speed-of-light volume,
# gMAGNUS page, section IV-C, Eq. (8) for the histogram).
def kernel_bytes(name, st, elems_heavy, nnz_c_heavy, final_chunks, heavy_rows):
    if name == "outer_product":
        return 12 * elems_heavy                       # write C^ (col + val)
    if name == "histogram":
        return 4 * elems_heavy + 8 * (heavy_rows + 1) + 8 * final_chunks   # Eq. (8)
    if name == "multisplit":
        return 24 * elems_heavy                       # read + write C^ (col + val)
    if name == "chunk_symbolic":
        return 4 * elems_heavy                        # read C^_reord columns
    if name == "chunk_numeric":
        return 12 * elems_heavy + 12 * nnz_c_heavy    # read C^_reord, write the heavy rows of C
    if name == "chunk_dense":
        return 12 * st.dense_elems + 12 * st.dense_nnz  # its share of the same
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--flags", type=int, default=0, help="extra SPGEMM_FLAG_* bits for A/B runs")
    ap.add_argument("--chunk-width", type=int, default=0, help="planner override W (A/B runs)")
    ap.add_argument("--tau", type=int, default=0, help="planner override tau (A/B runs)")
    ap.add_argument("--rmat-scale", type=int, default=0,
                    help="replace the workload by a seeded R-MAT of this scale (small cases for profiling)")
    ap.add_argument("--edge-factor", type=int, default=16)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the variant measurements (direct split, upper-bound and estimated light rows)")
    ap.add_argument("--workflow", type=int, default=0,
                    help="light-row sizing: 0 exact symbolic, 1 IP upper bound, 2 HyperLogLog, 3 automatic")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.rmat_scale:
        cfg_name = "rmat_s%d_ef%d" % (args.rmat_scale, args.edge_factor)
        A = synth.rmat(args.rmat_scale, args.edge_factor, seed=0)
    else:
        cfg_name = synth.CONFIGS[args.config][0]
        A = synth.config(args.config)

    if args.impl == "reference":
        run_reference(args, A, cfg_name, rank)
        return

    import torch
    import torch.distributed as dist
    import sparse_gemm_irregular_gb300 as sg

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sg.load()
    dA = sg.DeviceCSR.from_host(A)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    timing = sg.options(flags=sg.binding.FLAG_TIMING | args.flags, chunk_width=args.chunk_width, tau=args.tau,
                        workflow=args.workflow)
    plain = (sg.options(flags=args.flags, chunk_width=args.chunk_width, tau=args.tau, workflow=args.workflow)
             if (args.flags or args.chunk_width or args.tau or args.workflow) else None)

    def step(opts=None, keep=False):
        p = sg.Product(dA, dA, stream=stream, opts=opts)
        rp, nnz = p.symbolic()
        col, val = p.numeric()
        out = (p.stats(), p.phase_times() if opts is not None else None)
        p.close()
        if keep:
            return out, (rp, col, val)
        return out

    for _ in range(args.warmup):
        (st, _), _c = step(plain, keep=True)
        del _c
    torch.cuda.synchronize()

    # timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    phase_tot = {}
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = sg.spgemm_kernel_launches()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.fill_(float(i))        # L2 flush, outside the step's events
            ev[i][0].record(stream)
            st, ph = step(timing)
            ev[i][1].record(stream)
            for k_, (ms, n_) in ph.items():
                a = phase_tot.setdefault(k_, [0.0, 0])
                a[0] += ms
                a[1] += n_
        torch.cuda.synchronize()
    launches = sg.spgemm_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_total = max_over_ranks(sum(step_ms) / 1e3, world)

    ip = st.ip_total
    c_nnz = st.c_nnz
    value = job_rate(ip, args.steps, world, t_total)
    ms_per_step = t_total / args.steps * 1e3
    peak, peak_src = load_peaks()
    comp = compulsory_bytes(A, A, c_nnz)
    hbm_frac = comp / (t_total / args.steps) / 1e9 / peak

    # dominant kernel of the step and its roofline
    kern = ["outer_product", "histogram", "multisplit", "chunk_symbolic", "chunk_dense"]
    dom = max(kern, key=lambda k_: phase_tot.get(k_, [0, 0])[0])
    dom_ms, dom_n = phase_tot[dom]
    roofline = None
    byt = kernel_bytes(dom, st, st.ip_heavy, st.c_nnz_heavy, st.final_chunks, st.rows_heavy)
    if dom_n and byt:
        achieved = byt * args.steps / (dom_ms / 1e3) / 1e9   # algorithmic bytes / device time
        traffic = measured_traffic(KERNEL_OF.get(dom, ""), cfg_name)
        roofline = {"kernel": KERNEL_OF.get(dom, dom), "bound": "hbm", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                    "algorithmic_bytes_per_launch": byt,
                    "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)",
                    "timed_regions_per_step": dom_n / args.steps,
                    "ms_per_step": dom_ms / args.steps}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg_name, "m": A.rows, "nnz_A": A.nnz, "ip_total": ip, "nnz_C": c_nnz,
                   "rows_heavy": st.rows_heavy, "ip_heavy": st.ip_heavy,
                   "light_rows": ("exact symbolic", "IP upper bound", "HyperLogLog estimate")[st.workflow],
                   "l2": "512 MiB buffer written between timed steps (outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_roofline": {"compulsory_bytes": comp, "frac": hbm_frac, "peak_gbs": peak,
                         "peak_source": peak_src},
        "phases_ms_per_step": {k_: v[0] / args.steps for k_, v in phase_tot.items() if v[1]},
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "step_ms": step_ms,
    }

    # the same product on other paths, measured the same way: the direct split of level 0
    # (SPGEMM_FLAG_DIRECT_SPLIT) and the light rows sized by their IP bound or by HyperLogLog
    # estimates instead of the exact symbolic pass (SPGEMM_WORKFLOW_UPPER_BOUND / _ESTIMATE)
    if not args.no_variants:
        result["variants"] = {}
        for name, vflags, vwf in (("direct_split", sg.binding.FLAG_DIRECT_SPLIT, args.workflow),
                                  ("upper_bound", 0, sg.binding.WORKFLOW_UPPER_BOUND),
                                  ("estimate", 0, sg.binding.WORKFLOW_ESTIMATE)):
            vopt = sg.options(flags=sg.binding.FLAG_TIMING | vflags | args.flags, chunk_width=args.chunk_width,
                              tau=args.tau, workflow=vwf)
            for _ in range(2):
                step(vopt)
            torch.cuda.synchronize()
            vms, vph = [], {}
            for i in range(args.steps):
                flush.fill_(float(i))
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                _, ph = step(vopt)
                b_.record(stream)
                torch.cuda.synchronize()
                vms.append(a_.elapsed_time(b_))
                for k_, (ms, n_) in ph.items():
                    vph[k_] = vph.get(k_, 0.0) + ms
            vt = max_over_ranks(sum(vms) / 1e3, world)
            result["variants"][name] = {
                "value": job_rate(ip, args.steps, world, vt), "unit": UNIT,
                "ms_per_step": vt * 1e3 / args.steps,
                "phases_ms_per_step": {k_: v / args.steps for k_, v in vph.items() if v > 0}}

    # end to end through the public API with host buffers
    if not args.no_e2e:
        result["e2e"] = e2e(args, A, sg, torch, stream, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gf, nrows, ipn, dt = oracle_rate(A, A, 12.0, threads)
        result["cpu_baseline"] = {"value": gf, "unit": UNIT, "cores": threads, "kind": "oracle",
                                  "sample": "%d seeded uniform rows, %d intermediate products, %.1f s"
                                            % (nrows, ipn, dt)}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def e2e(args, A, sg, torch, stream, world):
    """Same metric through the public API with host inputs and outputs: every step copies A from
    pinned host memory, runs the product, and receives C in pinned host memory through
    spgemm_numeric_host (C is computed in row windows and each finished window is copied out
    while the next one is computed).  Warm-up steps as for the device-resident metric."""
    hp = [torch.from_numpy(a).pin_memory() for a in (A.row_ptr, A.col, A.val)]
    dev = [torch.empty_like(x, device="cuda") for x in hp]
    h2d = sum(x.numel() * x.element_size() for x in hp)
    host_c = None
    times = []
    warm = max(3, args.warmup)
    steps = max(1, min(args.steps, 3))
    d2h = 0
    st = None
    for i in range(warm + steps):
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for x, y in zip(dev, hp):
            x.copy_(y, non_blocking=True)
        dA = sg.DeviceCSR(A.rows, A.cols, dev[0], dev[1], dev[2])
        p = sg.Product(dA, dA, stream=stream)
        _, nnz = p.symbolic()
        if host_c is None:  # first (warm-up) pass: pin the host arrays of C once
            host_c = [torch.empty(A.rows + 1, dtype=torch.int64).pin_memory(),
                      torch.empty(max(nnz, 1), dtype=torch.int32).pin_memory(),
                      torch.empty(max(nnz, 1), dtype=torch.float64).pin_memory()]
        p.numeric_host(host_c[1], host_c[2], host_c[0])
        t1.record(stream)
        st = p.stats()
        p.close()
        torch.cuda.synchronize()
        d2h = (A.rows + 1) * 8 + nnz * 12
        if i >= warm:
            times.append(t0.elapsed_time(t1) / 1e3)
    t = max_over_ranks(sum(times), world)
    return {"value": job_rate(st.ip_total, len(times), world, t), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": len(times), "warmup": warm}


if __name__ == "__main__":
    main()
