#!/usr/bin/env python3
"""Benchmark of the GB300 generalized GEMM with fused epilogues.

Default run (the contract line): one step is the whole hot path over one batch
of synthetic input -- the M = N = K = 8192 fp16 GEMM with fp32 C and D,
alpha = 1.5, beta = 0.5, in all four operand layouts (NN, NT, TN, TT), each a
separate library call.  `value` is TFLOP/s over the timed steps with inputs
resident in HBM (inputs are larger than L2, no flush needed); `e2e` is the same
metric through gemm_run_host (host buffers, copies inside the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--suite]

--impl reference times the CPU oracle (fp64, all host cores) on bounded samples
of the same workload.  --suite prints one extra JSON line per workload of the
parity suite (256^3, FC layer, int8, SGEMM, square sweep, skinny).
Multi-GPU: replicas only (each rank runs the full workload on its own GPU; no
data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "GEMM TFLOP/s (TOP/s int8) at 1 GB300 and % of dense tensor-core peak"
LAYOUTS = ["NN", "NT", "TN", "TT"]
MAIN_N = 8192
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DOMINANT_KERNEL_SOURCES = ["dense_gemm_epilogues_gb300/csrc/tc2_kernel.cu",
                           "dense_gemm_epilogues_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "tc_pair_gemm_f16_8192_traffic.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--suite", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload measurements of the other benchmark workloads")
    ap.add_argument("--case", default=None,
                    help="run one named workload --iters times (profiling driver); see CASES")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--vs-cublas", action="store_true",
                    help="time the library against torch.matmul / F.linear (cuBLAS) on the square "
                         "sweep, a short-K shape and the FC layer; a comparison, not a contract line")
    return ap.parse_args()


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def choose_tensor_peak(peaks: dict, clocks: dict, timed_s: float):
    """The tensor-core denominator of a timed region: the burst peak, unless the
    region lasted at least a second and the chip sat at its power cap in most of
    the samples taken under load -- the condition of the sustained peak.
    Returns (peak, source text)."""
    under_load = clocks.get("samples_under_load") or 0
    capped = clocks.get("power_cap_samples_under_load") or 0
    src = peaks.get("source", "measured")
    if timed_s >= 1.0 and under_load > 0 and 2 * capped > under_load:
        return peaks["bf16_tflops_sustained"], (
            f"{src} bf16 dense sustained: the {timed_s:.2f} s timed region ran at the power cap in "
            f"{capped} of {under_load} samples under load (fp16 has the same dense rate)")
    return peaks["bf16_tflops"], (
        f"{src} bf16 dense burst: the {timed_s:.3f} s timed region ran at the power cap in {capped} of "
        f"{under_load} samples under load (fp16 has the same dense rate)")


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of the ranks' values of x (each rank's elapsed time -> the
    job's); x itself when there is one rank (dist None)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return flops_per_rank * world / seconds / 1e12


def workload_config(world: int) -> dict:
    return {"workload": "gemm_f16_8192x8192x8192_alpha1.5_beta0.5_fp32_C_D_layouts_NN_NT_TN_TT",
            "M": MAIN_N, "N": MAIN_N, "K": MAIN_N, "layouts": LAYOUTS, "ab": "f16",
            "accumulate": "f32", "c": "f32", "d": "f32", "alpha": 1.5, "beta": 0.5,
            "gemms_per_step": len(LAYOUTS),
            "l2": "inputs larger than L2 (A, B 134 MB per layout, C and D 268 MB); no flush",
            "parallelism": f"replicas{world}"}


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        top = max(mx) if mx else None
        loaded_rows = [r for r in rows if num(r[1]) is not None and top and num(r[1]) > 0.5 * top] or rows
        loaded = [num(r[1]) for r in loaded_rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        cap = sum(1 for r in loaded_rows if r[8].lower() == "active")
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": top, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_cap_samples_under_load": cap,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# --------------------------------------------------------------- traffic ----

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in DOMINANT_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_counters() -> dict:
    """DRAM bytes and tensor-pipe activity per launch of the dominant kernel from
    the committed ncu summary; empty when the kernel sources changed since the
    capture (the figures would describe another kernel)."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_source_hash():
            return {}
        out = {"traffic": float(kv["dram_bytes_per_launch"])}
        if "tensor_pipe_active_pct" in kv:
            out["tensor_pipe_active_pct"] = float(kv["tensor_pipe_active_pct"])
        for k in ("sm_cycles_active", "sm_clock_hz_under_ncu", "launch_us_under_ncu"):
            if k in kv:
                out[k] = float(kv[k])
        return out
    except (OSError, KeyError, ValueError):
        return {}


def theoretical_at_clock(counters: dict, flops_per_launch: float, sms: int) -> dict:
    """The second denominator: SMs x per-SM dense rate x the clock ncu saw.  The
    per-SM rate is measured from the committed counters (flops per tensor-active
    cycle per SM), the SM count read from the device.  None when the counters
    are stale or absent."""
    need = ("sm_cycles_active", "sm_clock_hz_under_ncu", "launch_us_under_ncu", "tensor_pipe_active_pct")
    if not all(k in counters for k in need):
        return None
    busy = counters["sm_cycles_active"] * counters["tensor_pipe_active_pct"] / 100.0
    per_sm_rate = flops_per_launch / sms / busy
    peak = sms * per_sm_rate * counters["sm_clock_hz_under_ncu"] / 1e12
    achieved = flops_per_launch / (counters["launch_us_under_ncu"] * 1e-6) / 1e12
    return {"sms": sms, "flops_per_tensor_cycle_per_sm": round(per_sm_rate, 1),
            "clock_ghz": round(counters["sm_clock_hz_under_ncu"] / 1e9, 4), "peak": round(peak, 1),
            "achieved_under_ncu": round(achieved, 1), "frac": round(achieved / peak, 4), "unit": "TFLOP/s"}


def measured_traffic():
    """DRAM bytes per launch of the dominant kernel (None when stale)."""
    return measured_counters().get("traffic")


# ------------------------------------------------------------ our kernels ---

def kernel_label(cfg: dict) -> str:
    if cfg.get("kernel_name") == "tc_pair":
        return (f"tc_pair_gemm_kernel (tcgen05 cta_group::2, {cfg['bm']}x{cfg['bn']} tiles per CTA pair, "
                f"{cfg['stages']} stages)")
    return f"tc_gemm_kernel (tcgen05, {cfg.get('bm')}x{cfg.get('bn')} tiles, {cfg.get('stages')} stages)"


def make_main_problems():
    from dense_gemm_epilogues_gb300 import inputs as I
    return [I.square_fp16_8192(l) for l in LAYOUTS]


def device_inputs(problems, device):
    """Generate each layout's inputs (same seed => same logical matrices) and
    copy them to the device; C is shared, D is one output buffer."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    out = []
    C = None
    for p in problems:
        inp = I.generate(p, I.BASE_SEED + 1)
        if C is None:
            C = inp.C.to(device)
        out.append({"p": p, "A": inp.A.to(device), "B": inp.B.to(device), "host": inp})
    D = torch.empty((MAIN_N, MAIN_N), dtype=torch.float32, device=device)
    return out, C, D


def run_gemm(G, plan, p, A, B, C, D, stream, epi):
    G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N, p.K,
               p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(), p.ldc,
               D.data_ptr(), p.ldd, epi, stream)


def bench_ours(args, rank, world, local_rank):
    import torch
    import dense_gemm_epilogues_gb300 as G

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    G.load_library()
    problems = make_main_problems()
    ins, C, D = device_inputs(problems, device)
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, local_rank)
    epi = G.make_epilogue(G.GEMM_F32)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream

    def step(ev=None):
        for li, x in enumerate(ins):
            if ev is not None:
                ev[li][0].record(stream)
            run_gemm(G, plan, x["p"], x["A"], x["B"], C, D, sh, epi)
            if ev is not None:
                ev[li][1].record(stream)

    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    gpu_id = cvd.split(",")[local_rank] if cvd else str(local_rank)
    sampler = ClockSampler(gpu_id)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler.start()
    cfg_used = plan.last_config()
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in ins] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    launch_ms = [e[0].elapsed_time(e[1]) for st in evs for e in st]
    status = plan.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = max_over_ranks(total_ms, dist, device)

    flops_per_gemm = 2.0 * MAIN_N ** 3
    flops_step = flops_per_gemm * len(ins)
    value = job_tflops(flops_step * args.steps, world, total_ms / 1e3)
    peaks = load_peaks()
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    per_layout_ms = {l: round(statistics.mean(st[li][0].elapsed_time(st[li][1]) for st in evs), 4)
                     for li, l in enumerate(LAYOUTS)}
    achieved = flops_per_gemm / avg_launch_s / 1e12
    peak, peak_source = choose_tensor_peak(peaks, clocks, total_ms / 1e3)
    counters = measured_counters()
    roofline = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": counters.get("traffic"),
                "tensor_pipe_active_pct": counters.get("tensor_pipe_active_pct"),
                "theoretical_at_ncu_clock": theoretical_at_clock(
                    counters, flops_per_gemm, torch.cuda.get_device_properties(device).multi_processor_count),
                "counters_source": "profiles/tc_pair_gemm_f16_8192_traffic.txt (ncu, TN launch; null once "
                                   "the kernel sources change)",
                "peak_source": peak_source,
                "frac_of_burst_peak": round(achieved / peaks["bf16_tflops"], 4),
                "burst_peak": peaks["bf16_tflops"],
                "sustained_peak": peaks["bf16_tflops_sustained"],
                "kernel": kernel_label(cfg_used),
                "algorithmic_flops_per_launch": flops_per_gemm,
                "avg_launch_ms": round(avg_launch_s * 1e3, 4), "per_layout_ms": per_layout_ms}

    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(G, plan, ins, device, min(args.steps, 20), dist)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic", "config": workload_config(world), "roofline": roofline,
            "clocks": clocks, "e2e": e2e, "gpu_launches": len(ins) * args.steps,
            "kernel_config": cfg_used}
    if rank == 0 and not args.no_configs:
        line["configs"] = measure_configs(G, device, gpu_id)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(budget_s=15.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.suite and rank == 0:
        run_suite(G, device)
        run_batched_suite(G, device)
        run_diag_suite(G, device)
        run_pair_suite(G, device)
        run_transform_suite(G, device)
    plan.close()
    if dist:
        dist.destroy_process_group()


def bench_e2e(G, plan, ins, device, steps, dist):
    """Same metric through gemm_run_host: per step and layout, the H2D copy of A,
    B and C from pinned host memory, the GEMM, and the D2H copy of D."""
    import torch
    hosts = []
    for x in ins:
        h = x["host"]
        hosts.append((x["p"], h.A.pin_memory(), h.B.pin_memory()))
    Ch = ins[0]["host"].C.pin_memory()
    Dh = torch.empty((MAIN_N, MAIN_N), dtype=torch.float32).pin_memory()
    epi = G.make_epilogue(G.GEMM_F32)
    stream = torch.cuda.current_stream(device).cuda_stream

    def step():
        for p, A, B in hosts:
            G.gemm_run_host(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b],
                            p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                            p.beta, Ch.data_ptr(), p.ldc, Dh.data_ptr(), p.ldd, epi, stream)

    step()   # sizes the plan's staging buffers
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t, dist, device)
    world = dist.get_world_size() if dist else 1
    flops = 2.0 * MAIN_N ** 3 * len(hosts) * steps * world
    h2d = sum(A.numel() * A.element_size() + B.numel() * B.element_size() for _, A, B in hosts)
    h2d += len(hosts) * Ch.numel() * Ch.element_size()
    d2h = len(hosts) * Dh.numel() * Dh.element_size()
    return {"value": round(flops / el / 1e12, 1), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "api": "gemm_run_host (C ABI, host buffers)"}


# ------------------------------------------------------------- CPU oracle ---

def _oracle_rows(O, inp, rows, nthreads=None):
    import numpy as np
    p = inp.problem
    rr = np.repeat(np.asarray(rows, dtype=np.int64), p.N)
    cc = np.tile(np.arange(p.N, dtype=np.int64), len(rows))
    t = time.perf_counter()
    O.gemm_entries(O.F16, O.LAYOUT_N if p.layout_a == "N" else O.LAYOUT_T,
                   O.LAYOUT_N if p.layout_b == "N" else O.LAYOUT_T, p.M, p.N, p.K, p.alpha,
                   inp.A, p.lda, inp.B, p.ldb, rr, cc, beta=p.beta, c_dtype=O.F32, C=inp.C,
                   ldc=p.ldc, d_dtype=O.F32, nthreads=nthreads)
    return time.perf_counter() - t


def cpu_baseline_sample(budget_s: float = 15.0, problem=None, inp=None) -> dict:
    """The oracle, as it stands, on whole rows of the TN 8192^3 GEMM."""
    import oracle as O
    from dense_gemm_epilogues_gb300 import inputs as I
    O.build()
    if inp is None:
        problem = problem or I.square_fp16_8192("TN")
        inp = I.generate(problem, I.BASE_SEED + 1)
    p = inp.problem
    t1 = _oracle_rows(O, inp, [0])
    rows = max(1, int(budget_s / max(t1, 1e-6)))
    rows = min(rows, p.M)
    el = _oracle_rows(O, inp, list(range(rows)))
    flops = 2.0 * rows * p.N * p.K
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": O.max_threads(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": f"{rows} full rows ({rows}x{p.N} outputs, K={p.K}) of the {p.layout_a}{p.layout_b} "
                      f"8192^3 fp16 GEMM with alpha/beta epilogue, fp64 accumulation"}


def bench_reference(args, rank, world):
    """The reference arm: the CPU oracle timed on bounded samples of the same
    workload (rows of each layout's GEMM in turn)."""
    if rank != 0:
        return
    import oracle as O
    from dense_gemm_epilogues_gb300 import inputs as I
    O.build()
    problems = make_main_problems()
    inps = [I.generate(p, I.BASE_SEED + 1) for p in problems]
    total_steps = args.steps + args.warmup
    per_step = min(6.0, 150.0 / max(total_steps, 1))
    # Rows per step, per layout: the oracle's speed per row depends on the layout
    # (a column-major A is walked with a stride), so each is calibrated apart.
    rows = []
    for inp in inps:
        t_row = _oracle_rows(O, inp, [0])
        rows.append(max(1, int(per_step / max(t_row, 1e-6))))
    for s in range(args.warmup):
        _oracle_rows(O, inps[s % 4], list(range(rows[s % 4])))
    el, flops = 0.0, 0.0
    for s in range(args.steps):
        el += _oracle_rows(O, inps[s % 4], list(range(rows[s % 4])))
        flops += 2.0 * rows[s % 4] * MAIN_N * MAIN_N
    value = flops / el / 1e12
    sample = (f"per step {'/'.join(map(str, rows))} full rows (x{MAIN_N} outputs, K={MAIN_N}) of the "
              f"NN/NT/TN/TT GEMMs in turn, fp64 oracle, about {per_step:.1f} s each")
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(world), "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": O.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ suite ---

def run_suite(G, device, warmup=3, iters=20):
    """One JSON line per workload of the parity suite (not the contract line)."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    peaks = load_peaks()
    cases = [(I.square_fp16_256(), 0), (I.fc_bf16_8192x4096x11008(), 2), (I.int8_8192(), 3),
             (I.sgemm_4096_bias_relu(), 4)]
    cases += [(I.square_fp16(n), 5) for n in (512, 1024, 2048, 4096, 16384)]
    cases += [(I.skinny_fp16_16384x64x16384(), 6)]
    stream = torch.cuda.current_stream(device)
    for p, k in cases:
        inp = I.generate(p, I.BASE_SEED + k)
        A, B = inp.A.to(device), inp.B.to(device)
        C = inp.C.to(device) if inp.C is not None else None
        bias = inp.bias.to(device) if inp.bias is not None else None
        D = torch.empty((p.M, p.ldd), dtype=I.TORCH_DTYPES[p.d], device=device)
        cc = p.c or ("s32" if p.ab == "s8" else "f32")
        plan = G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[cc], device.index or 0)
        bm = {"none": G.GEMM_BIAS_NONE, "col": G.GEMM_BIAS_COL, "row": G.GEMM_BIAS_ROW}[p.bias_mode]
        epi = G.make_epilogue(G.DTYPE_CODES[p.d], bias.data_ptr() if bias is not None else 0,
                              G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32, bm,
                              G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE)

        def call_on(st):
            G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M,
                       p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                       C.data_ptr() if C is not None else None, p.ldc if C is not None else 0,
                       D.data_ptr(), p.ldd, epi, st.cuda_stream)

        def call():
            call_on(stream)
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
        for _ in range(warmup):
            call()
        # (1) back to back: `iters` calls between two events, so the host-side
        # work of each call overlaps the previous kernel; per call = total / iters.
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        t_b2b = e0.elapsed_time(e1) / 1e3 / iters
        # (2) cold: L2 flushed before each single call; includes the host-side
        # work between the start event and the launch.
        times = []
        for _ in range(5):
            flush.zero_()
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            call()
            c1.record(stream)
            torch.cuda.synchronize()
            times.append(c0.elapsed_time(c1) / 1e3)
        t_cold = statistics.median(times)
        t = t_b2b
        # (3) GPU time alone: the same calls replayed from a CUDA graph on a side
        # stream (no host work between launches).
        t_graph = None
        try:
            side = torch.cuda.Stream(device)
            side.wait_stream(torch.cuda.current_stream(device))
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                gr.capture_begin()
                for _ in range(iters):
                    call_on(side)
                gr.capture_end()
            side.synchronize()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(side):    # replay() launches on the current stream
                gr.replay()
                side.synchronize()
                g0.record(side)
                gr.replay()
                g1.record(side)
            side.synchronize()
            t_graph = g0.elapsed_time(g1) / 1e3 / iters
            del gr
        except RuntimeError:
            t_graph = None
        status = plan.device_status()
        cfg = plan.last_config()
        eb = I.ELEM_BYTES
        algo_bytes = (inp.A.numel() * eb[p.ab] + inp.B.numel() * eb[p.ab] + p.M * p.N * eb[p.d]
                      + (p.M * p.N * eb[p.c] if p.c else 0))
        tflops = p.flops / t / 1e12
        rec = {"suite": p.name, "M": p.M, "N": p.N, "K": p.K, "kernel": cfg["kernel_name"],
               "tile": f"{cfg['bm']}x{cfg['bn']}x{cfg['bk']}", "grid": cfg["grid"],
               "median_us": round(t * 1e6, 2), "cold_us": round(t_cold * 1e6, 2),
               "graph_us": round(t_graph * 1e6, 2) if t_graph else None,
               "tflops_graph": round(p.flops / t_graph / 1e12, 2) if t_graph else None,
               "inputs_fit_l2": algo_bytes < 126e6, "tflops": round(tflops, 2),
               "gbs": round(algo_bytes / t / 1e9, 1), "algo_bytes": algo_bytes,
               "frac_tensor_peak": round(tflops / peaks["bf16_tflops"], 4),
               "frac_hbm": round(algo_bytes / t / 1e9 / peaks["hbm_gbs"], 4), "status": status}
        print(json.dumps(rec), flush=True)
        plan.close()
        del A, B, C, D, bias, flush
        torch.cuda.empty_cache()


def run_transform_suite(G, device, iters=10):
    """Operand transforms after load (t(x) = act(scale * x) on A and/or B): each
    workload graph-timed without transforms, with them on the selector's path,
    and forced inside the kernel / staged (GEMM_XF_STAGE=0 / 1).  One JSON line
    per workload."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    cases = [("fc_relu_x", I.fc_bf16_8192x4096x11008(), dict(a_act=G.GEMM_ACT_RELU)),
             ("gemm8192_tn_relu_a_scale_b", I.square_fp16_8192("TN").with_(beta=0.0, c=None),
              dict(a_act=G.GEMM_ACT_RELU, b_scale=0.5)),
             ("gemm2048_relu_a", I.square_fp16(2048), dict(a_act=G.GEMM_ACT_RELU)),
             ("skinny_relu_a", I.skinny_fp16_16384x64x16384(), dict(a_act=G.GEMM_ACT_RELU))]
    for name, p, xf in cases:
        inp = I.generate(p, I.BASE_SEED + 30)
        A, B = inp.A.to(device), inp.B.to(device)
        C = inp.C.to(device) if inp.C is not None else None
        bias = inp.bias.to(device) if inp.bias is not None else None
        D = torch.empty((p.M, p.ldd), dtype=I.TORCH_DTYPES[p.d], device=device)
        plan = G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[p.c or "f32"], device.index or 0)
        bm = {"none": G.GEMM_BIAS_NONE, "col": G.GEMM_BIAS_COL, "row": G.GEMM_BIAS_ROW}[p.bias_mode]

        def graph_us(epi):
            side = torch.cuda.Stream(device)
            side.wait_stream(torch.cuda.current_stream(device))   # the inputs were copied on the current stream

            def call():
                G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N, p.K,
                           p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                           C.data_ptr() if C is not None else None, p.ldc if C is not None else 0,
                           D.data_ptr(), p.ldd, epi, side.cuda_stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    call()
                side.synchronize()
                gr = torch.cuda.CUDAGraph()
                gr.capture_begin()
                for _ in range(iters):
                    call()
                gr.capture_end()
                gr.replay()
                side.synchronize()
                g0 = torch.cuda.Event(enable_timing=True)
                g1 = torch.cuda.Event(enable_timing=True)
                g0.record(side)
                gr.replay()
                g1.record(side)
            side.synchronize()
            return round(g0.elapsed_time(g1) * 1e3 / iters, 2), plan.last_config()

        def epi_of(**kw):
            return G.make_epilogue(G.DTYPE_CODES[p.d], bias.data_ptr() if bias is not None else 0,
                                   G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32, bm,
                                   G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE, **kw)
        rec = {"transform_suite": name, "M": p.M, "N": p.N, "K": p.K, "transform": {
            k: v for k, v in xf.items()}}
        rec["plain_us"], _ = graph_us(epi_of())
        old_env = os.environ.pop("GEMM_XF_STAGE", None)
        rec["default_us"], cfg = graph_us(epi_of(**xf))
        rec["default_path"] = "staged" if cfg["xf_staged"] else "in_kernel"
        for v, key in (("0", "in_kernel_us"), ("1", "staged_us")):
            os.environ["GEMM_XF_STAGE"] = v
            rec[key], _ = graph_us(epi_of(**xf))
        os.environ.pop("GEMM_XF_STAGE", None)
        if old_env is not None:
            os.environ["GEMM_XF_STAGE"] = old_env
        rec["kernel"] = cfg["kernel_name"]
        rec["status"] = plan.device_status()
        print(json.dumps(rec), flush=True)
        plan.close()
        del A, B, C, D, bias
        torch.cuda.empty_cache()


# Every benchmark workload beside the contract's (the FC layer, int8, SGEMM, the
# square sweep and the skinny GEMM), measured in the default
# run: (problem constructor, seed offset, bound of its roofline).
def config_workloads():
    from dense_gemm_epilogues_gb300 import inputs as I
    out = [("gemm_f16_tn_256", I.square_fp16_256(), 0, "tensor"),
           ("fc_bf16_8192x4096x11008_bias_relu", I.fc_bf16_8192x4096x11008(), 2, "tensor"),
           ("gemm_s8_tn_8192", I.int8_8192(), 3, "tensor"),
           ("sgemm_f32_tn_4096_bias_relu", I.sgemm_4096_bias_relu(), 4, "alu")]
    out += [(f"sweep_gemm_f16_tn_{n}", I.square_fp16(n), 5, "tensor") for n in (512, 1024, 2048, 4096, 16384)]
    out += [("skinny_gemm_f16_tn_16384x64x16384", I.skinny_fp16_16384x64x16384(), 6, "hbm")]
    return out


def algorithmic_bytes(p, eb) -> int:
    """Bytes a GEMM must move at least once: A, B, C (when read), bias, D."""
    n = p.M * p.K * eb[p.ab] + p.K * p.N * eb[p.ab] + p.M * p.N * eb[p.d]
    if p.c:
        n += p.M * p.N * eb[p.c]
    if p.bias:
        n += (p.N if p.bias_mode == "col" else p.M) * eb[p.bias]
    return n


def ffma_peak_tflops(sm_count: int, sm_mhz: float) -> float:
    """FP32 FFMA issue peak: 128 FP32 lanes per SM, 2 flops per FMA."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


def measure_configs(G, device, gpu_id, min_region_s=0.4, max_iters=3000):
    """One record per benchmark workload: mean device time per call from CUDA
    events on the launching stream around `iters` back-to-back calls, with its
    own clock record and roofline.  A workload whose inputs and output fit in L2 rotates over enough
    copies of them (different addresses, same values) that the copies together
    exceed L2 three times over, so no call finds its data in L2."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    peaks = load_peaks()
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    stream = torch.cuda.current_stream(device)
    eb = I.ELEM_BYTES
    l2_bytes = 129e6
    records = []
    for name, p, k, bound in config_workloads():
        inp = I.generate(p, I.BASE_SEED + k)
        abytes = algorithmic_bytes(p, eb)
        nsets = 1 if abytes >= 2 * l2_bytes else int(min(1024, -(-3 * l2_bytes // abytes)))
        sets = []
        for _ in range(nsets):
            sets.append({"A": inp.A.to(device), "B": inp.B.to(device),
                         "C": inp.C.to(device) if inp.C is not None else None,
                         "bias": inp.bias.to(device) if inp.bias is not None else None,
                         "D": torch.empty((p.M, p.ldd), dtype=I.TORCH_DTYPES[p.d], device=device)})
        cc = p.c or ("s32" if p.ab == "s8" else "f32")
        plan = G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[cc], device.index or 0)
        bm = {"none": G.GEMM_BIAS_NONE, "col": G.GEMM_BIAS_COL, "row": G.GEMM_BIAS_ROW}[p.bias_mode]
        epis = [G.make_epilogue(G.DTYPE_CODES[p.d], x["bias"].data_ptr() if x["bias"] is not None else 0,
                                G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32, bm,
                                G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE) for x in sets]

        def call(i):
            x = sets[i % nsets]
            G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M,
                       p.N, p.K, p.alpha, x["A"].data_ptr(), p.lda, x["B"].data_ptr(), p.ldb, p.beta,
                       x["C"].data_ptr() if x["C"] is not None else None,
                       p.ldc if x["C"] is not None else 0, x["D"].data_ptr(), p.ldd, epis[i % nsets],
                       stream.cuda_stream)
        for i in range(max(3, min(nsets, 50))):
            call(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(5):
            call(i)
        torch.cuda.synchronize()
        est = max((time.perf_counter() - t0) / 5, 1e-6)
        iters = int(min(max_iters, max(10, min_region_s / est)))
        # Back to back between two events (no event between calls, so each launch
        # may start its prologue while the previous call finishes, as in use).
        sampler = ClockSampler(gpu_id)
        sampler.start()
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for i in range(iters):
            call(i)
        r1.record(stream)
        torch.cuda.synchronize()
        clocks = sampler.stop()
        region_s = r0.elapsed_time(r1) / 1e3
        t_mean = region_s / iters
        cfg = plan.last_config()
        status = plan.device_status()
        flops = p.flops
        rec = {"name": name, "M": p.M, "N": p.N, "K": p.K, "layout": p.layout_a + p.layout_b,
               "ab": p.ab, "d": p.d, "alpha": p.alpha, "beta": p.beta,
               "epilogue": (f"bias[{p.bias_mode}] " if p.bias else "") + (p.act if p.act != "none" else ""),
               "kernel": cfg["kernel_name"], "tile": f"{cfg['bm']}x{cfg['bn']}", "grid": cfg["grid"],
               "stream_k_tiles": cfg["sk_tiles"], "half_tiles": cfg["half_tiles"],
               "iters": iters, "mean_us": round(t_mean * 1e6, 2),
               "timing": "CUDA events around the back-to-back calls on the launching stream",
               "l2": (f"rotates over {nsets} copies of the inputs and output "
                      f"({nsets * abytes / 1e6:.0f} MB > 3 x L2); no flush") if nsets > 1
                     else "inputs and output exceed L2; no flush",
               "algorithmic_bytes": abytes, "flops": flops, "status": status, "clocks": clocks}
        if bound == "hbm":
            ach = abytes / t_mean / 1e9
            rec.update(value=round(ach, 1), unit="GB/s",
                       roofline={"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                                 "peak_source": f"{peaks['source']} HBM copy bandwidth"},
                       tflops=round(flops / t_mean / 1e12, 2))
        elif bound == "alu":
            mhz = clocks.get("sm_max_mhz") or 2070.0
            pk = ffma_peak_tflops(sm_count, mhz)
            ach = flops / t_mean / 1e12
            rec.update(value=round(ach, 2), unit="TFLOP/s",
                       roofline={"bound": "alu", "achieved": round(ach, 2), "peak": round(pk, 2),
                                 "unit": "TFLOP/s", "frac": round(ach / pk, 4),
                                 "peak_source": f"FFMA issue rate: {sm_count} SMs x 128 FP32 lanes x 2 flops "
                                                f"x {mhz:.0f} MHz (maximum SM clock)"})
            med = clocks.get("sm_mhz")
            if med:
                rec["roofline"]["frac_at_median_clock"] = round(ach / ffma_peak_tflops(sm_count, med), 4)
        else:
            pk, src = choose_tensor_peak(peaks, clocks, region_s)
            ach = flops / t_mean / 1e12
            unit = "TOP/s" if p.ab == "s8" else "TFLOP/s"
            if p.ab == "s8":
                src += "; int8 runs on the fp16 tensor-core kind (exact chunks), so its unit's peak is fp16's"
            rec.update(value=round(ach, 2), unit=unit,
                       roofline={"bound": "tensor", "achieved": round(ach, 2), "peak": pk, "unit": unit,
                                 "frac": round(ach / pk, 4), "peak_source": src},
                       gbs=round(abytes / t_mean / 1e9, 1))
        records.append(rec)
        plan.close()
        del sets, inp
        torch.cuda.empty_cache()
    return records


def run_batched_suite(G, device, warmup=3, iters=20):
    """Strided-batched workloads (one JSON line each): back-to-back calls and
    CUDA-graph replay, as run_suite."""
    import torch
    peaks = load_peaks()
    cases = [("batched_f16_tn_64x1024x1024x1024", 64, 1024, 1024, 1024, "f16", "f32"),
             ("batched_bf16_tn_256x512x512x128", 256, 512, 512, 128, "bf16", "bf16")]
    for name, batch, M, N, K, ab, d in cases:
        td = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
        gen = torch.Generator().manual_seed(20261202 + 11)
        A = (torch.rand((batch, M, K), generator=gen) * 2 - 1).to(td[ab]).to(device)
        B = (torch.rand((batch, N, K), generator=gen) * 2 - 1).to(td[ab]).to(device)
        D = torch.empty((batch, M, N), dtype=td[d], device=device)
        plan = G.Plan(G.DTYPE_CODES[ab], G.GEMM_F32, device.index or 0)
        epi = G.make_epilogue(G.DTYPE_CODES[d])

        def call_on(st):
            G.gemm_run_strided_batched(plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, M, N, K, 1.0,
                                       A.data_ptr(), K, M * K, B.data_ptr(), K, N * K, 0.0, None,
                                       0, 0, D.data_ptr(), N, M * N, batch, epi, 0, st.cuda_stream)
        stream = torch.cuda.current_stream(device)
        for _ in range(warmup):
            call_on(stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            call_on(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / iters
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            gr.capture_begin()
            for _ in range(iters):
                call_on(side)
            gr.capture_end()
            gr.replay()
            side.synchronize()
            e0.record(side)
            gr.replay()
            e1.record(side)
        side.synchronize()
        tg = e0.elapsed_time(e1) / 1e3 / iters
        flops = 2.0 * batch * M * N * K
        eb = {"f16": 2, "bf16": 2, "f32": 4}
        algo_bytes = batch * (M * K + N * K) * eb[ab] + batch * M * N * eb[d]
        cfg = plan.last_config()
        print(json.dumps({"suite": name, "batch": batch, "M": M, "N": N, "K": K,
                          "kernel": cfg["kernel_name"], "tiles": cfg["tiles"],
                          "median_us": round(t * 1e6, 2), "graph_us": round(tg * 1e6, 2),
                          "tflops": round(flops / t / 1e12, 2), "tflops_graph": round(flops / tg / 1e12, 2),
                          "gbs_graph": round(algo_bytes / tg / 1e9, 1), "algo_bytes": algo_bytes,
                          "frac_tensor_peak": round(flops / tg / 1e12 / peaks["bf16_tflops"], 4),
                          "frac_hbm": round(algo_bytes / tg / 1e9 / peaks["hbm_gbs"], 4),
                          "status": plan.device_status()}), flush=True)
        plan.close()
        del A, B, D, gr
        torch.cuda.empty_cache()


def run_diag_suite(G, device, warmup=3, iters=20, sets=4):
    """Diagonal-operand workloads (one JSON line each).  Calls rotate over
    `sets` copies of the inputs and outputs (each copy larger than L2), so every
    call reads its operands from HBM.  The same GEMM with the diagonal written
    out as a dense matrix (gemm_run, tensor cores) is timed beside it."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    peaks = load_peaks()
    for layout in ("N", "T"):
        p = I.diag_fp16_4096(layout)
        dinp = I.generate_diag(p, I.BASE_SEED + 20)
        dg = dinp.diag.to(device)
        Xs = [dinp.X.to(device) for _ in range(sets)]
        Cs = [dinp.C.to(device) for _ in range(sets)]
        Ds = [torch.empty((p.M, p.ldd), dtype=torch.float32, device=device) for _ in range(sets)]
        plan = G.Plan(G.GEMM_F16, G.GEMM_F32, device.index or 0)
        epi = G.make_epilogue(G.GEMM_F32)
        side_code = G.GEMM_SIDE_LEFT if p.side == "left" else G.GEMM_SIDE_RIGHT

        def diag_call(k, st):
            G.gemm_run_diag(plan.handle, side_code, G.LAYOUT_CODES[p.layout_x], p.M, p.N, p.alpha,
                            dg.data_ptr(), Xs[k].data_ptr(), p.ldx, p.beta, Cs[k].data_ptr(), p.ldc,
                            Ds[k].data_ptr(), p.ldd, epi, st.cuda_stream)

        sq = torch.zeros((p.M, p.M), dtype=torch.float16, device=device)
        sq.diagonal().copy_(dg)            # symmetric, so its storage serves either layout
        dp = p.dense()

        def dense_call(k, st):
            G.gemm_run(plan.handle, G.LAYOUT_CODES[dp.layout_a], G.LAYOUT_CODES[dp.layout_b], dp.M,
                       dp.N, dp.K, dp.alpha, sq.data_ptr(), dp.lda, Xs[k].data_ptr(), dp.ldb,
                       dp.beta, Cs[k].data_ptr(), dp.ldc, Ds[k].data_ptr(), dp.ldd, epi,
                       st.cuda_stream)

        def timed(call):
            stream = torch.cuda.current_stream(device)
            for w in range(warmup):
                call(w % sets, stream)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for it in range(iters):
                call(it % sets, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1e3 / iters
            side = torch.cuda.Stream(device)
            side.wait_stream(torch.cuda.current_stream(device))
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                gr.capture_begin()
                for it in range(iters):
                    call(it % sets, side)
                gr.capture_end()
                gr.replay()
                side.synchronize()
                e0.record(side)
                gr.replay()
                e1.record(side)
            side.synchronize()
            return t, e0.elapsed_time(e1) / 1e3 / iters

        t, tg = timed(diag_call)
        cfg = plan.last_config()
        td, tdg = timed(dense_call)
        dense_cfg = plan.last_config()
        algo_bytes = p.n_diag * 2 + p.M * p.N * (2 + 4 + 4)
        print(json.dumps({"suite": p.name, "M": p.M, "N": p.N, "side": p.side, "layout_x": p.layout_x,
                          "kernel": cfg["kernel_name"], "grid": cfg["grid"], "tiles": cfg["tiles"],
                          "median_us": round(t * 1e6, 2), "graph_us": round(tg * 1e6, 2),
                          "gbs_graph": round(algo_bytes / tg / 1e9, 1), "algo_bytes": algo_bytes,
                          "frac_hbm": round(algo_bytes / tg / 1e9 / peaks["hbm_gbs"], 4),
                          "dense_kernel": dense_cfg["kernel_name"], "dense_graph_us": round(tdg * 1e6, 2),
                          "dense_median_us": round(td * 1e6, 2),
                          "speedup_vs_dense": round(tdg / tg, 2), "rotating_sets": sets,
                          "status": plan.device_status()}), flush=True)
        plan.close()
        del Xs, Cs, Ds, sq, dg
        torch.cuda.empty_cache()


def run_pair_suite(G, device, warmup=3, iters=20):
    """Complex and dual-number GEMM workloads (one JSON line each): the whole
    gemm_run_complex call (staging pass + tensor-core GEMM), back to back and
    from a CUDA graph.  TFLOP/s count the definition's real operations (8 per
    complex multiply-add, 6 per dual one)."""
    import torch
    from dense_gemm_epilogues_gb300 import inputs as I
    peaks = load_peaks()
    for unit in ("complex", "dual"):
        p = I.pair_fp16_4096(unit)
        inp = I.generate_pairs(p, I.BASE_SEED + 30)
        A, B, C = inp.A.to(device), inp.B.to(device), inp.C.to(device)
        D = torch.empty((p.M, p.ldd, 2), dtype=torch.float32, device=device)
        plan = G.Plan(G.GEMM_F16, G.GEMM_F32, device.index or 0)
        epi = G.make_epilogue(G.GEMM_F32)
        code = G.GEMM_UNIT_IMAGINARY if unit == "complex" else G.GEMM_UNIT_DUAL

        def call_on(st):
            G.gemm_run_complex(plan.handle, code, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b],
                               p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                               p.beta, C.data_ptr(), p.ldc, D.data_ptr(), p.ldd, epi, st.cuda_stream)
        stream = torch.cuda.current_stream(device)
        for _ in range(warmup):
            call_on(stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            call_on(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / iters
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            gr.capture_begin()
            for _ in range(iters):
                call_on(side)
            gr.capture_end()
            gr.replay()
            side.synchronize()
            e0.record(side)
            gr.replay()
            e1.record(side)
        side.synchronize()
        tg = e0.elapsed_time(e1) / 1e3 / iters
        cfg = plan.last_config()
        real_flops = 2.0 * p.M * (2 * p.N) * (2 * p.K)
        print(json.dumps({"suite": p.name, "unit": unit, "M": p.M, "N": p.N, "K": p.K,
                          "kernel": cfg["kernel_name"], "real_gemm": f"{p.M}x{2 * p.N}x{2 * p.K}",
                          "median_us": round(t * 1e6, 2), "graph_us": round(tg * 1e6, 2),
                          "tflops_graph": round(p.flops / tg / 1e12, 2),
                          "tensor_tflops_graph": round(real_flops / tg / 1e12, 2),
                          "frac_tensor_peak": round(real_flops / tg / 1e12 / peaks["bf16_tflops"], 4),
                          "status": plan.device_status()}), flush=True)
        plan.close()
        del A, B, C, D, gr
        torch.cuda.empty_cache()


def _cases():
    from dense_gemm_epilogues_gb300 import inputs as I
    return {
        "square4096_tn_ab": I.square_fp16_8192("TN").with_(name="gemm_f16_tn_4096_ab", M=4096,
                                                          N=4096, K=4096),
        "square4096_nt_ab": I.square_fp16_8192("NT").with_(name="gemm_f16_nt_4096_ab", M=4096,
                                                          N=4096, K=4096),
        "square8192_tn_ab": I.square_fp16_8192("TN"),
        "square8192_nt_ab": I.square_fp16_8192("NT"),
        "square8192_nn_ab": I.square_fp16_8192("NN"),
        "square8192_tt_ab": I.square_fp16_8192("TT"),
        "fc": I.fc_bf16_8192x4096x11008(),
        "int8_4096": I.int8_8192().with_(name="gemm_s8_tn_4096", M=4096, N=4096, K=4096),
        "int8_8192": I.int8_8192(),
        "square2048": I.square_fp16(2048),
        "square4096_k1024": I.square_fp16(4096).with_(name="gemm_f16_tn_4096x4096x1024", K=1024, d="f16"),
        "sgemm4096": I.sgemm_4096_bias_relu(),
        "skinny": I.skinny_fp16_16384x64x16384(),
    }


def run_diag_case(layout: str, iters: int):
    """The 4096 x 4096 diagonal-operand workload `iters` times (profiling driver)."""
    import torch
    import dense_gemm_epilogues_gb300 as G
    from dense_gemm_epilogues_gb300 import inputs as I
    p = I.diag_fp16_4096(layout)
    dinp = I.generate_diag(p, I.BASE_SEED + 20)
    dev = torch.device("cuda", 0)
    dg, X, C = dinp.diag.to(dev), dinp.X.to(dev), dinp.C.to(dev)
    D = torch.empty((p.M, p.ldd), dtype=torch.float32, device=dev)
    plan = G.Plan(G.GEMM_F16, G.GEMM_F32, 0)
    stream = torch.cuda.current_stream(dev)
    for i in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        G.gemm_run_diag(plan.handle, G.GEMM_SIDE_LEFT, G.LAYOUT_CODES[layout], p.M, p.N, p.alpha,
                        dg.data_ptr(), X.data_ptr(), p.ldx, p.beta, C.data_ptr(), p.ldc, D.data_ptr(),
                        p.ldd, G.make_epilogue(G.GEMM_F32), stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        print(json.dumps({"case": p.name, "iter": i, "ms": round(e0.elapsed_time(e1), 4),
                          "config": plan.last_config()}), flush=True)
    if plan.device_status() != 0:
        raise RuntimeError("device status non-zero")
    plan.close()


def run_case(name: str, iters: int):
    """Run one workload `iters` times on cuda:0 and print per-call times
    (a driver for profilers; its numbers are not benchmark results)."""
    import torch
    import dense_gemm_epilogues_gb300 as G
    from dense_gemm_epilogues_gb300 import inputs as I
    if name in ("diag_n", "diag_t"):
        run_diag_case(name[-1].upper(), iters)
        return
    p = _cases()[name]
    inp = I.generate(p, I.BASE_SEED + 7)
    dev = torch.device("cuda", 0)
    A, B = inp.A.to(dev), inp.B.to(dev)
    C = inp.C.to(dev) if inp.C is not None else None
    bias = inp.bias.to(dev) if inp.bias is not None else None
    D = torch.empty((p.M, p.ldd), dtype=I.TORCH_DTYPES[p.d], device=dev)
    cc = p.c or ("s32" if p.ab == "s8" else "f32")
    plan = G.Plan(G.DTYPE_CODES[p.ab], G.DTYPE_CODES[cc], 0)
    bm = {"none": G.GEMM_BIAS_NONE, "col": G.GEMM_BIAS_COL, "row": G.GEMM_BIAS_ROW}[p.bias_mode]
    epi = G.make_epilogue(G.DTYPE_CODES[p.d], bias.data_ptr() if bias is not None else 0,
                          G.DTYPE_CODES[p.bias] if p.bias else G.GEMM_F32, bm,
                          G.GEMM_ACT_RELU if p.act == "relu" else G.GEMM_ACT_NONE)
    stream = torch.cuda.current_stream(dev)
    for i in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        G.gemm_run(plan.handle, G.LAYOUT_CODES[p.layout_a], G.LAYOUT_CODES[p.layout_b], p.M, p.N,
                   p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                   C.data_ptr() if C is not None else None, p.ldc if C is not None else 0,
                   D.data_ptr(), p.ldd, epi, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        print(json.dumps({"case": name, "iter": i, "ms": round(e0.elapsed_time(e1), 4),
                          "config": plan.last_config()}), flush=True)
    if plan.device_status() != 0:
        raise RuntimeError("device status non-zero")
    plan.close()


def _graph_us(device, call, iters=20, replays=5):
    """GPU time per call: `iters` calls captured in one CUDA graph on a side
    stream, the best of `replays` replays timed with CUDA events."""
    import torch
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))   # the inputs were written on the current stream
    with torch.cuda.stream(side):
        for _ in range(3):
            call(side)
    side.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        gr.capture_begin()
        for _ in range(iters):
            call(side)
        gr.capture_end()
    side.synchronize()
    best = float("inf")
    for _ in range(replays):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record(side)
            gr.replay()
            e1.record(side)
        side.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1000.0 / iters)
    del gr
    return best


def run_vs_cublas():
    """The library against cuBLAS (torch.matmul; F.linear + relu_ for the FC
    layer) on the same inputs, both graph-timed, one JSON line per shape, in
    increasing size with the short-K shape before the long ones (a long shape
    changes the clock state the next one starts in).  fp16 in and out, TN;
    every library result is checked against the fp32 product."""
    import torch
    import torch.nn.functional as F
    import dense_gemm_epilogues_gb300 as G
    G.load_library()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    for (M, N, K) in [(256,) * 3, (512,) * 3, (1024,) * 3, (2048,) * 3, (4096, 4096, 1024), (3072,) * 3,
                      (4096,) * 3, (8192,) * 3]:
        A = (torch.rand(M, K, device=dev, generator=g) * 2 - 1).half()
        B = (torch.rand(N, K, device=dev, generator=g) * 2 - 1).half()
        D = torch.empty(M, N, device=dev, dtype=torch.float16)
        plan = G.Plan(G.GEMM_F16, G.GEMM_F32, 0)
        epi = G.make_epilogue(G.GEMM_F16)

        def lib(st):
            G.gemm_run(plan.handle, G.GEMM_OP_T, G.GEMM_OP_N, M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), K,
                       0.0, None, 0, D.data_ptr(), N, epi, st.cuda_stream)
        Bt = B.t()

        def cub(st):
            torch.matmul(A, Bt)
        t_lib = _graph_us(dev, lib)
        torch.cuda.synchronize()
        nonfinite = int((~torch.isfinite(D)).sum())
        ref = torch.matmul(A.float(), B.float().t())
        err = ((D.float() - ref).abs() / (ref.abs() + 1)).max().item()
        del ref
        t_cub = _graph_us(dev, cub)
        print(json.dumps({"vs_cublas": f"{M}x{N}x{K}", "lib_us": round(t_lib, 2), "cublas_us": round(t_cub, 2),
                          "lib_tflops": round(2 * M * N * K / t_lib / 1e6, 1),
                          "cublas_tflops": round(2 * M * N * K / t_cub / 1e6, 1),
                          "kernel": plan.last_config()["kernel_name"], "max_rel_err": err,
                          "nonfinite": nonfinite, "status": plan.device_status()}), flush=True)
        plan.close()
    M, K, N = 8192, 4096, 11008
    X = torch.randn(M, K, device=dev, generator=g).bfloat16()
    W = (torch.randn(K, N, device=dev, generator=g) * 0.02).bfloat16()
    bias = torch.randn(N, device=dev, generator=g) * 0.1
    bias16 = bias.bfloat16()
    D = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
    plan = G.Plan(G.GEMM_BF16, G.GEMM_F32, 0)
    epi = G.make_epilogue(G.GEMM_BF16, bias.data_ptr(), G.GEMM_F32, G.GEMM_BIAS_COL, G.GEMM_ACT_RELU)

    def lib_fc(st):
        G.gemm_run(plan.handle, G.GEMM_OP_T, G.GEMM_OP_T, M, N, K, 1.0, X.data_ptr(), K, W.data_ptr(), N, 0.0,
                   None, 0, D.data_ptr(), N, epi, st.cuda_stream)
    Wt = W.t().contiguous()

    def cub_fc(st):
        torch.relu_(F.linear(X, Wt, bias16))
    t_lib, t_cub = _graph_us(dev, lib_fc), _graph_us(dev, cub_fc)
    print(json.dumps({"vs_cublas": "fc_8192x11008x4096_bias_relu", "lib_us": round(t_lib, 2),
                      "cublas_us": round(t_cub, 2), "lib_tflops": round(2 * M * N * K / t_lib / 1e6, 1),
                      "cublas_tflops": round(2 * M * N * K / t_cub / 1e6, 1),
                      "kernel": plan.last_config()["kernel_name"], "status": plan.device_status()}), flush=True)
    plan.close()


def main():
    args = parse_args()
    rank, world, local_rank = dist_info()
    if args.case:
        run_case(args.case, args.iters)
        return
    if args.vs_cublas:
        run_vs_cublas()
        return
    if args.impl == "reference":
        bench_reference(args, rank, world)
        return
    bench_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
