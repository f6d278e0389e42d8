"""Benchmark of the SpGEMM library: C = A * A on the seeded synthetic workloads, one GPU per
process.

Headline workload: R-MAT scale 21, edge factor 32 (Graph500 quadrant probabilities, fp64
values U[0,1)), the largest of the five.  Its C (about 6e10 entries, 0.7 TB) fits neither the
device nor the host, so the numeric phase runs in row windows (spgemm_row_windows cuts them
between heavy batches) into one reused device buffer; every window is computed inside the
timed step.  The other four workloads (uniform 8 per row, band 7, R-MAT scale 18, the
Markov-clustering expansion) are measured the same way in the same run and reported under
"workloads".

One step = one whole product through the library (create: planner, IP count and binning;
symbolic; caller allocation of C or reuse of the window buffer; numeric; destroy), inputs
resident in HBM.  The metric is GFLOP/s = 2 x intermediate products / time, plus the fraction
of the HBM roofline of the compulsory bytes (A, the rows of B that are touched, and C).  L2 is
flushed between timed steps by writing a 512 MiB buffer outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1..5]

`--impl reference` times the CPU oracle (ordered-map Gustavson) on the host cores on a bounded
sample of the same rows.  Under torchrun each rank runs its own replica (the product does not
need a second GPU); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
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
# A C larger than this share of the device memory is produced window by window into a reused
# device buffer; a C larger than HOST_C_BYTES comes back to the host window by window as well
WINDOWED_SHARE = 0.5
HOST_C_BYTES = 32e9
WINDOW_TARGET = 1_000_000_000      # entries of C per numeric window (windows hold whole heavy batches)


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


def cpu_model() -> str:
    """The host CPU's model name (lscpu on Arm hosts, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


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
    rows, ipn = sample_rows_by_ip(A, B, 2e6 * threads / 16)
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
                         "cpu": cpu_model(),
                         "sample": "%d seeded uniform rows (%d intermediate products) per step"
                                   % (len(rows), ipn)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def kernel_bytes(name, st):
    """Algorithmic bytes per product of a kernel that can dominate (the speed-of-light volume of
    the gMAGNUS page, section IV-C).  When C^_reord is kept from the symbolic to the numeric
    phase (stats.resident) the heavy rows are expanded once, with values; otherwise the symbolic
    phase expands columns only and the numeric phase expands again with values -- unless the
    symbolic phase counted the heavy chunks from generated products (stats.gen_symbolic), which
    leaves one expansion, in the numeric phase."""
    e = st.ip_heavy
    res = bool(st.resident)
    once = res or bool(st.gen_symbolic)   # one expansion per product, with values
    if name == "outer_product":
        return 12 * e if once else (4 + 12) * e         # write C^ / C^_reord (col [+ val])
    if name == "multisplit":
        return 24 * e if res else (8 + 24) * e          # read + write C^ (col [+ val])
    if name == "chunk_symbolic":
        return 4 * e                                     # read C^_reord columns
    if name == "chunk_dense":
        return 12 * st.dense_elems + 12 * st.dense_nnz  # read its C^_reord elements, write its C entries
    return None


class Workload:
    """One input on the device plus how its C is produced (whole, or window by window)."""

    def __init__(self, name, A, sg, torch):
        self.name, self.A = name, A
        self.dA = sg.DeviceCSR.from_host(A)
        self.sg, self.torch = sg, torch
        self.col = self.val = None   # reused device window buffers (windowed products)
        self.windowed = None

    def ensure_buffers(self, n):
        torch = self.torch
        if self.col is None or self.col.numel() < n:
            self.col = self.val = None
            torch.cuda.empty_cache()
            self.col = torch.empty(max(n, 1), dtype=torch.int32, device="cuda")
            self.val = torch.empty(max(n, 1), dtype=torch.float64, device="cuda")

    def step(self, stream, opts=None, dA=None):
        """One whole product; returns (stats, phase times or None, number of numeric windows)."""
        sg = self.sg
        dA = dA if dA is not None else self.dA
        p = sg.Product(dA, dA, stream=stream, opts=opts)
        try:
            _, nnz = p.symbolic()
            if self.windowed is None:
                total = self.torch.cuda.get_device_properties(0).total_memory
                self.windowed = nnz * 12 > WINDOWED_SHARE * total
            if self.windowed:
                cuts, wmax = p.row_windows(WINDOW_TARGET)
                self.ensure_buffers(wmax)
                p.numeric_windows(self.col, self.val, cuts=cuts)
                nwin = len(cuts) - 1
            else:
                p.numeric()
                nwin = 1
            out = (p.stats(), p.phase_times() if opts is not None else None, nwin)
        finally:
            p.close()
        return out


def timed_steps(w, stream, flush, steps, warmup, opts_timed, opts_plain, world, clocks=None):
    """warmup untimed steps, then `steps` timed ones (CUDA events on the product's stream, L2
    flushed before each outside the events).  Returns (seconds over ranks, stats, phase sums,
    per-step ms, windows per step, kernel launches in the timed steps)."""
    import torch
    sg = w.sg
    st = None
    for _ in range(warmup):
        st, _, _ = w.step(stream, opts_plain)
    torch.cuda.synchronize()
    phase_tot = {}
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = sg.spgemm_kernel_launches()
    nwin = 1
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        for i in range(steps):
            flush.fill_(float(i))        # L2 flush, outside the step's events
            ev[i][0].record(stream)
            st, ph, nwin = w.step(stream, opts_timed)
            ev[i][1].record(stream)
            for k_, (ms, n_) in ph.items():
                a = phase_tot.setdefault(k_, [0.0, 0])
                a[0] += ms
                a[1] += n_
        torch.cuda.synchronize()
    launches = sg.spgemm_kernel_launches() - launches0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_total = max_over_ranks(sum(step_ms) / 1e3, world)
    return t_total, st, phase_tot, step_ms, nwin, launches


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def phase_table(phase_tot, steps):
    """Device milliseconds per step and phase.  The light rows run on their own stream next to
    the heavy pipeline, so their numeric region is the wall time of that stream, overlapped."""
    out = {}
    for k_, v in phase_tot.items():
        if not v[1]:
            continue
        key = "light_numeric_overlapped_wall" if k_ == "light_numeric" else k_
        out[key] = v[0] / steps
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, help="headline workload (1..5); default R-MAT scale 21")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the other four workloads")
    ap.add_argument("--flags", type=int, default=0, help="extra SPGEMM_FLAG_* bits for A/B runs")
    ap.add_argument("--chunk-width", type=int, default=0, help="planner override W (A/B runs)")
    ap.add_argument("--tau", type=int, default=0, help="planner override tau (A/B runs)")
    ap.add_argument("--rmat-scale", type=int, default=0,
                    help="replace the workload by a seeded R-MAT of this scale (small cases for profiling)")
    ap.add_argument("--edge-factor", type=int, default=16)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the variants of the headline product (the separate level-0 multisplit pass, "
                         "chunks generated from the column-split B)")
    ap.add_argument("--all-variants", action="store_true",
                    help="also the light rows sized by their IP bound or by HyperLogLog estimates")
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
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    extra = dict(chunk_width=args.chunk_width, tau=args.tau, workflow=args.workflow)
    timing = sg.options(flags=sg.binding.FLAG_TIMING | args.flags, **extra)
    plain = sg.options(flags=args.flags, **extra) if (args.flags or args.chunk_width or args.tau or args.workflow) \
        else None

    w = Workload(cfg_name, A, sg, torch)
    clk = ClockSampler(local)
    t_total, st, phase_tot, step_ms, nwin, launches = timed_steps(
        w, stream, flush, args.steps, args.warmup, timing, plain, world, clocks=clk)

    ip = st.ip_total
    c_nnz = st.c_nnz
    value = job_rate(ip, args.steps, world, t_total)
    ms_per_step = t_total / args.steps * 1e3
    peak, peak_src = load_peaks()
    comp = compulsory_bytes(A, A, c_nnz)
    hbm_frac = comp / (t_total / args.steps) / 1e9 / peak

    # dominant kernel of the step and its roofline
    kern = ["outer_product", "multisplit", "chunk_symbolic", "chunk_dense"]
    dom = max(kern, key=lambda k_: phase_tot.get(k_, [0, 0])[0])
    dom_ms, dom_n = phase_tot.get(dom, [0.0, 0])
    roofline = None
    byt = kernel_bytes(dom, st)
    kname = "k_outer_direct" if (dom == "outer_product" and st.direct_split) else KERNEL_OF.get(dom, dom)
    if dom_n and byt:
        achieved = byt * args.steps / (dom_ms / 1e3) / 1e9   # algorithmic bytes / device time
        traffic = measured_traffic(kname, cfg_name)
        roofline = {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                    "algorithmic_bytes_per_step": byt,
                    "algorithmic_bytes_per_launch": byt * args.steps / dom_n,
                    "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)",
                    "timed_regions_per_step": dom_n / args.steps,
                    "ms_per_step": dom_ms / args.steps}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg_name, "m": A.rows, "nnz_A": A.nnz, "ip_total": ip, "nnz_C": c_nnz,
                   "rows_heavy": st.rows_heavy, "ip_heavy": st.ip_heavy,
                   "heavy_batches": st.heavy_batches, "resident": st.resident,
                   "symbolic_heavy": "generated products" if st.gen_symbolic else "expansion",
                   "level0_split": "inside the outer product" if st.direct_split else "separate multisplit pass",
                   "numeric_windows": nwin,
                   "light_rows": ("exact symbolic", "IP upper bound", "HyperLogLog estimate")[st.workflow],
                   "l2": "512 MiB buffer written between timed steps (outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_roofline": {"compulsory_bytes": comp, "frac": hbm_frac, "peak_gbs": peak,
                         "peak_source": peak_src},
        "phases_ms_per_step": phase_table(phase_tot, args.steps),
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "step_ms": step_ms,
    }

    # the same product on other paths, measured the same way (fewer steps): the paper's flow of
    # a separate outer product and level-0 multisplit pass (SPGEMM_FLAG_EXPAND_SPLIT), the heavy
    # chunks generated from the column-split B (SPGEMM_FLAG_FUSED), and on request the light rows
    # sized by their IP bound or by HyperLogLog estimates (SPGEMM_WORKFLOW_UPPER_BOUND / _ESTIMATE)
    if not args.no_variants:
        result["variants"] = {}
        todo = [("expanded_multisplit", sg.binding.FLAG_EXPAND_SPLIT, args.workflow),
                ("generated_chunks", sg.binding.FLAG_FUSED, args.workflow)]
        if args.all_variants:
            todo += [("upper_bound", 0, sg.binding.WORKFLOW_UPPER_BOUND),
                     ("estimate", 0, sg.binding.WORKFLOW_ESTIMATE)]
        vsteps = min(args.steps, 5)
        for name, vflags, vwf in todo:
            vopt = sg.options(flags=sg.binding.FLAG_TIMING | vflags | args.flags, chunk_width=args.chunk_width,
                              tau=args.tau, workflow=vwf)
            vt, vst, vph, _, _, _ = timed_steps(w, stream, flush, vsteps, 2, vopt, vopt, world)
            result["variants"][name] = {
                "value": job_rate(ip, vsteps, world, vt), "unit": UNIT, "steps": vsteps,
                "ms_per_step": vt * 1e3 / vsteps, "phases_ms_per_step": phase_table(vph, vsteps)}

    # end to end through the public API with host buffers
    if not args.no_e2e:
        result["e2e"] = e2e(args, w, sg, torch, stream, world)

    # the other workloads, measured the same way (device-resident inputs; the L2 flush between
    # steps; max over ranks), each with its end-to-end figure
    if not args.no_others and not args.rmat_scale:
        result["workloads"] = {}
        for cid in sorted(synth.CONFIGS):
            if cid == args.config:
                continue
            name = synth.CONFIGS[cid][0]
            Ao = synth.config(cid)
            wo = Workload(name, Ao, sg, torch)
            ot, ost, oph, oms, onw, _ = timed_steps(wo, stream, flush, args.steps, args.warmup, timing, plain, world)
            ocomp = compulsory_bytes(Ao, Ao, ost.c_nnz)
            entry = {"value": job_rate(ost.ip_total, args.steps, world, ot), "unit": UNIT,
                     "ms_per_step": ot * 1e3 / args.steps, "steps": args.steps,
                     "ip_total": ost.ip_total, "nnz_C": ost.c_nnz, "rows_heavy": ost.rows_heavy,
                     "resident": ost.resident, "numeric_windows": onw,
                     "hbm_roofline": {"compulsory_bytes": ocomp,
                                      "frac": ocomp / (ot / args.steps) / 1e9 / peak},
                     "phases_ms_per_step": phase_table(oph, args.steps)}
            if not args.no_e2e:
                entry["e2e"] = e2e(args, wo, sg, torch, stream, world)
            result["workloads"][name] = entry
            del wo
            torch.cuda.synchronize()
            sg.spgemm_release_memory()
            torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gf, nrows, ipn, dt = oracle_rate(A, A, 10.0, threads)
        gf1, nrows1, ipn1, dt1 = oracle_rate(A, A, 6.0, 1)
        result["cpu_baseline"] = {"value": gf, "unit": UNIT, "cores": threads, "kind": "oracle",
                                  "cpu": cpu_model(),
                                  "sample": "%d seeded uniform rows, %d intermediate products, %.1f s"
                                            % (nrows, ipn, dt),
                                  "one_core": {"value": gf1, "unit": UNIT, "cores": 1,
                                               "sample": "%d seeded uniform rows, %d intermediate products, "
                                                         "%.1f s" % (nrows1, ipn1, dt1)}}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def e2e(args, w, sg, torch, stream, world):
    """Same metric through the public API with host inputs and outputs, over the same number of
    steps as the device-resident metric: every step copies A from pinned host memory and the
    product's C comes back to pinned host memory.  A C that fits the host goes through
    spgemm_numeric_host (row windows computed on the device, each finished window copied out
    while the next is computed).  A C larger than the host (the R-MAT scale 21 product) is
    computed window by window with spgemm_numeric_rows into two device buffers, and each window
    is copied, piece by piece, into a reused pinned host buffer on a second stream while the next
    window is computed: every entry of C crosses to the host, one piece at a time."""
    A = w.A
    torch.cuda.synchronize()
    sg.spgemm_release_memory()
    torch.cuda.empty_cache()
    host_windowed = None
    hp = [torch.from_numpy(a).pin_memory() for a in (A.row_ptr, A.col, A.val)]
    dev = [torch.empty_like(x, device="cuda") for x in hp]
    h2d = sum(x.numel() * x.element_size() for x in hp)
    times = []
    warm = max(3, args.warmup)
    steps = args.steps
    d2h = 0
    st = None
    copy_stream = torch.cuda.Stream()
    host_c = None
    win = None   # windowed: two device buffers, two pinned host pieces
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
        if host_windowed is None:
            host_windowed = w.windowed or nnz * 12 > HOST_C_BYTES
        if not host_windowed:
            if host_c is None:  # first (warm-up) pass: pin the host arrays of C once
                host_c = [torch.empty(A.rows + 1, dtype=torch.int64).pin_memory(),
                          torch.empty(max(nnz, 1), dtype=torch.int32).pin_memory(),
                          torch.empty(max(nnz, 1), dtype=torch.float64).pin_memory()]
            p.numeric_host(host_c[1], host_c[2], host_c[0])
        else:
            cuts, wmax = p.row_windows(WINDOW_TARGET)
            if win is None or win["dev"][0][0].numel() < wmax:
                win = None
                torch.cuda.empty_cache()
                piece = 1 << 27  # entries per host copy piece (1.5 GB of col + val)
                win = {"dev": [(torch.empty(wmax, dtype=torch.int32, device="cuda"),
                                torch.empty(wmax, dtype=torch.float64, device="cuda")) for _ in range(2)],
                       "host": (torch.empty(piece, dtype=torch.int32).pin_memory(),
                                torch.empty(piece, dtype=torch.float64).pin_memory()),
                       "piece": piece, "done": [torch.cuda.Event() for _ in range(2)]}
            rp_host = p.row_ptr.cpu().numpy()
            for wi, (rb, re) in enumerate(zip(cuts[:-1], cuts[1:])):
                b = wi % 2
                dcol, dval = win["dev"][b]
                if wi >= 2:
                    stream.wait_event(win["done"][b])      # its previous window copied out
                sg.spgemm_numeric_rows(p.h, rb, re, dcol.data_ptr(), dval.data_ptr())
                ev = torch.cuda.Event()
                ev.record(stream)
                copy_stream.wait_event(ev)
                n = int(rp_host[re] - rp_host[rb])
                # the window goes to the host piece by piece, in stream order on the copy stream
                # (each piece lands before the next overwrites it), while the next window computes
                with torch.cuda.stream(copy_stream):
                    hc, hv = win["host"]
                    for o in range(0, n, win["piece"]):
                        e_ = min(n, o + win["piece"])
                        hc[:e_ - o].copy_(dcol[o:e_], non_blocking=True)
                        hv[:e_ - o].copy_(dval[o:e_], non_blocking=True)
                win["done"][b].record(copy_stream)
            stream.wait_stream(copy_stream)
        t1.record(stream)
        st = p.stats()
        p.close()
        torch.cuda.synchronize()
        d2h = (A.rows + 1) * 8 + nnz * 12
        if i >= warm:
            times.append(t0.elapsed_time(t1) / 1e3)
    t = max_over_ranks(sum(times), world)
    out = {"value": job_rate(st.ip_total, len(times), world, t), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": len(times), "warmup": warm}
    if host_windowed:
        out["host_output"] = "row windows copied into a reused pinned host buffer (C beyond the host budget)"
    del win, host_c
    torch.cuda.synchronize()
    sg.spgemm_release_memory()
    torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
