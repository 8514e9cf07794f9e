#!/usr/bin/env python
"""Benchmark of the conditional-simulation hot path on GB300.

One step = one pass of the whole path over the headline workload (n = 32768 uniform sites,
exponential Matern range 0.03, nugget 1e-4, tile 512, M = 2048 simulations, fixedacc 1e-4):
covariance tiles + statistics, precision map + scale, adaptive Cholesky, normal draws fused
with the mixed-precision TRMM, calibration scan + quantiles + regions.  Inputs (locations,
zhat, v) are resident in HBM before the timed region; the tile matrix (>1 GB) is far larger
than L2, so no flush is needed between steps.

Metric (per the paper's own TRMM measure extended to the factorisation): Cholesky+TRMM
TFLOP/s = (n^3/3 + n^2/2 + n/6 + n^2 M) / time; `value` divides by the whole step time.
The JSON line also reports the Cholesky+TRMM-only rate, its multiple of the measured FP64
peak, the fraction of the precision-weighted peak, and simulations per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 (torchrun) each rank runs an independent replica (the path is single-GPU).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputgen  # noqa: E402

TIMED_KERNELS = ["k_diag_chol", "k_diag_chol_df", "k_split_diag_df", "k_tc_old", "k_tc_new", "k_tc_trsm", "k_tc_trmm",
                 "k_cov_stats", "k_cov_stats_refine", "k_generate", "k_scan"]
WORKLOAD = inputgen.WORKLOADS["c"]
SEED_Z = 12345


def flops(n, M):
    return n ** 3 / 3.0 + n ** 2 / 2.0 + n / 6.0, float(n) ** 2 * M


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sus": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


def attributed_flops(pmap: np.ndarray, nb: int, n: int, M: int):
    """Algorithmic flops by the arithmetic that executes them (FP64 units, FP16 tensor
    MMAs, FP32-class 3-MMA FP16 splits) for the left-looking schedule of the library."""
    nt = pmap.shape[0]
    f = {"fp64": 0.0, "fp32": 0.0, "fp16": 0.0}
    name = {0: "fp64", 1: "fp32", 2: "fp16"}
    b3 = float(nb) ** 3
    for j in range(nt):
        f["fp64"] += b3 / 3.0                       # diagonal factor
        for i in range(j, nt):
            for k in range(j):
                pc = max(pmap[i, j], pmap[i, k], pmap[j, k])
                f[name[pc]] += b3 if i == j else 2.0 * b3   # SYRK / GEMM
            if i > j:
                f[name[pmap[i, j]]] += b3           # triangular solve at the tile's class
    trmm = {"fp16": float(n) ** 2 * M - n * nb * M, "fp32": float(n) * nb * M}   # off-diagonal / diagonal
    return f, trmm


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for k, nm in enumerate(names):
                if len(r) > 4 + k and r[4 + k].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(n_s: int, M_s: int):
    """The oracle as it stands on the leading n_s sites of the workload: covariance,
    unblocked Cholesky, simulation, calibration.  Returns (seconds, flops)."""
    import oracle
    w = WORKLOAD
    xy = inputgen.workload_locations(w)[:n_s]
    Z = inputgen.standard_normals(n_s, M_s, SEED_Z)
    t0 = time.perf_counter()
    V = oracle.covariance_matrix(xy, w.family, w.sigma2, w.beta, w.nu, w.nugget)
    L = oracle.cholesky_lower(V)
    Y = oracle.simulate(L, Z)
    oracle.calibrate(Y, np.zeros(n_s), np.diag(V).copy(), w.u, w.level)
    dt = time.perf_counter() - t0
    fc, ft = flops(n_s, M_s)
    return dt, fc + ft


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        nums = [d.get("num_threads", 1) for d in threadpool_info()]
        if nums:
            return int(max(nums))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, world, rank):
    if rank != 0:
        return
    n_s, M_s = 2048, 2048
    for _ in range(args.warmup):
        oracle_sample(n_s, M_s)
    times, fl = [], 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample(n_s, M_s)
        times.append(dt)
    ms = 1e3 * float(np.mean(times))
    val = fl / (ms / 1e3) / 1e12
    unit = "TFLOP/s"
    line = {"metric": "Cholesky+TRMM TFLOP/s", "value": val, "unit": unit, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"oracle on the leading {n_s} sites of {WORKLOAD.name}", "n": n_s, "M": M_s},
            "cpu_baseline": {"value": val, "unit": unit, "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"leading {n_s} of {WORKLOAD.n} sites, M={M_s}, one full oracle pass per step"},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU path
def run_peaks(local):
    """Measured peaks of the arithmetic units the path runs on (cr_peak_probe), best of 3."""
    import torch
    import mixed_precision_dense_mat_gb300 as cr
    torch.cuda.set_device(local)
    cr.load()
    out = {}
    for name, kind in (("fp64_dfma", cr.CR_PEAK_DFMA), ("fp64_dmma", cr.CR_PEAK_DMMA), ("fp32_ffma", cr.CR_PEAK_FFMA),
                       ("df_mac", cr.CR_PEAK_DF_MAC)):
        out[name] = max(cr.peak_probe(kind, 4096) for _ in range(3))
    print(json.dumps({"peaks_tflops": out, "device": torch.cuda.get_device_name(local)}), flush=True)



def run_ours(args, world, rank, local):
    import torch
    import mixed_precision_dense_mat_gb300 as cr
    torch.cuda.set_device(local)
    cr.load()
    w = WORKLOAD
    n, nb, M = w.n, w.nb, w.M
    dev = torch.device("cuda", local)
    xy_h = inputgen.workload_locations(w)
    xy = torch.from_numpy(xy_h).to(dev)
    V = cr.TileMat(n, nb)
    Y = cr.colmajor_empty(n, M, torch.float64)
    zhat = torch.zeros(n, dtype=torch.float64, device=dev)              # no observations: zhat = 0
    vvec = torch.full((n,), w.sigma2 + w.nugget, dtype=torch.float64, device=dev)   # v_i = V_ii
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    info_box = {}

    def step(seed, e):
        e[0].record(stream)
        cr.cov_build(V, xy, w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget)
        e[1].record(stream)
        pmap, info = cr.precision_map(V, amp=True, fixedacc=w.fixedacc)
        e[2].record(stream)
        info_box["map"], info_box["info"] = pmap, info
        assert cr.potrf_adaptive(V) == 0
        e[3].record(stream)
        cr.trmm_sim(V, None, M, seed=seed, out=Y, flags=cr.CR_TRMM_GENERATE)
        e[4].record(stream)
        out = cr.calibrate(Y, zhat, vvec, w.u, w.level)
        e[5].record(stream)
        return out

    for q in range(args.warmup):
        step(SEED_Z + q, [ev() for _ in range(6)])
    torch.cuda.synchronize()

    # peaks of the units without a measured figure, measured here on this GPU: the FP64
    # FMA (the tile precision's own peak) and the double-float accumulate the diagonal
    # executor runs on (its ALU roofline)
    unit_peaks = {"fp64_dfma": cr.peak_probe(cr.CR_PEAK_DFMA, 2048), "df_mac": cr.peak_probe(cr.CR_PEAK_DF_MAC, 2048)}

    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if "CUDA_VISIBLE_DEVICES" in os.environ else str(local)
    clocks = ClockSampler(gpu_id)
    barrier(world)
    torch.cuda.synchronize()
    l0 = cr.kernel_launches()
    # the timed steps run without per-kernel timing (no events around the library's launches)
    cr.timing_enable(False)
    evs = [[ev() for _ in range(6)] for _ in range(args.steps)]
    t_start, t_end = ev(), ev()
    wall0 = time.perf_counter()
    t_start.record(stream)
    for q in range(args.steps):
        step(SEED_Z + 100 + q, evs[q])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    launches = cr.kernel_launches() - l0
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world)
    stages = ["cov_build", "precision_map", "potrf", "rng_trmm", "calibrate"]
    st = {s: float(np.mean([evs[q][k].elapsed_time(evs[q][k + 1]) for q in range(args.steps)])) for k, s in enumerate(stages)}
    per_step = [evs[q][0].elapsed_time(evs[q][5]) for q in range(args.steps)]
    ms = total_ms / args.steps
    fc, ft = flops(n, M)
    value = world * (fc + ft) / (ms / 1e3) / 1e12
    ct_ms = st["potrf"] + st["rng_trmm"]
    ct_tflops = (fc + ft) / (ct_ms / 1e3) / 1e12

    # a separate pass with per-kernel timing (CUDA events on each kernel's own stream) for the
    # kernel table and the roofline; its steps are not part of the timed result
    n_inst = 0 if args.no_kernel_timing else max(1, min(args.steps, 3))
    ktime = {k: (0.0, 0) for k in TIMED_KERNELS}
    inst_ms = None
    if n_inst:
        cr.timing_reset()
        cr.timing_enable(True)
        a, b = ev(), ev()
        a.record(stream)
        for q in range(n_inst):
            step(SEED_Z + 300 + q, [ev() for _ in range(6)])
        b.record(stream)
        torch.cuda.synchronize()
        cr.timing_enable(False)
        inst_ms = a.elapsed_time(b) / n_inst
        ktime = {k: cr.timing_read(k) for k in TIMED_KERNELS}

    pk = peaks()
    pmap, info = info_box["map"], info_box["info"]
    fch, ftr = attributed_flops(pmap.copy(), nb, n, M)
    p16 = pk["bf16_sus"] * 1e12
    peak_of = {"fp64": unit_peaks["fp64_dfma"] * 1e12, "fp16": p16, "fp32": p16 / 3.0}
    t_star = sum(fch[k] / peak_of[k] for k in fch) + sum(ftr[k] / peak_of[k] for k in ftr)
    frac_weighted = t_star / (ct_ms / 1e3)

    # per-kernel device time per step (instrumented pass) and the roofline of each against its
    # algorithmic work per launch
    kern = {}
    meas = "measured" if pk["src"] == "measured" else "fallback"
    def entry(name, bound, work_per_launch, unit, peak, peak_note):
        k_ms, cnt = ktime[name]
        if cnt == 0:
            return None
        per = k_ms / cnt
        ach = work_per_launch / (per / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
        return {"kernel": name, "bound": bound, "launches_per_step": cnt / n_inst, "ms_per_launch": per,
                "ms_per_step": k_ms / n_inst, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                "traffic": None, "peak_source": peak_note}
    kern["k_diag_chol_df"] = entry("k_diag_chol_df", "alu", 2.0 * nb ** 3 / 3.0, "TFLOP/s", unit_peaks["df_mac"],
                                   "double-float accumulate rate measured in this run (cr_peak_probe CR_PEAK_DF_MAC); "
                                   "work: nb^3/3 factor + nb^3/3 triangular inverse per launch")
    kern["k_diag_chol"] = entry("k_diag_chol", "alu", 2.0 * nb ** 3 / 3.0, "TFLOP/s", unit_peaks["fp64_dfma"],
                                "FP64 FMA rate measured in this run (cr_peak_probe CR_PEAK_DFMA); "
                                "work: nb^3/3 factor + nb^3/3 triangular inverse per launch")
    kern["k_tc_trmm"] = entry("k_tc_trmm", "tensor", float(n) ** 2 * M, "TFLOP/s", pk["bf16"],
                              f"{meas} bf16 burst (FP16 MMA runs at the bf16 rate); work: n^2 M per launch")
    kern["k_scan"] = entry("k_scan", "hbm", 8.0 * n * M + 16.0 * n, "GB/s", pk["hbm"],
                           f"{meas} HBM copy bandwidth; work: 8 n M + 16 n bytes per launch")
    # the Cholesky's tensor-core work, over the Cholesky stage's wall time (its launches run on
    # three concurrent streams, so their summed device time exceeds the stage)
    tc_ms = sum(ktime[k][0] for k in ("k_tc_old", "k_tc_new", "k_tc_trsm"))
    if tc_ms > 0:
        ach = (fch["fp16"] + fch["fp32"]) / (st["potrf"] / 1e3) / 1e12
        kern["k_tc_cholesky"] = {"kernel": "k_tc (update and solve modes)", "bound": "tensor",
                                 "ms_per_step_device_sum": tc_ms / n_inst, "stage_ms": st["potrf"], "achieved": ach,
                                 "peak": pk["bf16_sus"], "unit": "TFLOP/s", "frac": ach / pk["bf16_sus"], "traffic": None,
                                 "peak_source": f"{meas} bf16 sustained; work: FP16- and FP32-class Cholesky products "
                                                "(one per product, however many MMAs it takes) over the Cholesky "
                                                "stage's wall time"}
    for k in ("k_tc_old", "k_tc_new", "k_tc_trsm", "k_split_diag_df", "k_cov_stats", "k_cov_stats_refine", "k_generate"):
        k_ms, cnt = ktime[k]
        if cnt:
            kern[k] = {"kernel": k, "ms_per_step": k_ms / n_inst, "launches_per_step": cnt / n_inst}
    # the roofline line: the kernel with the largest device time per step among single kernels
    # with a stated work per launch (each is at most the step time)
    timed = {k: v for k, v in kern.items() if v and "ms_per_launch" in v}
    roof = None
    if timed:
        dominant = max(timed.values(), key=lambda e: e["ms_per_step"])
        roof = {key: dominant[key] for key in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        roof["kernel"] = dominant["kernel"]
        roof["ms_per_step"] = dominant["ms_per_step"]
        roof["peak_source"] = dominant["peak_source"]

    # end to end through the public API with host buffers: H2D of the locations, D2H of
    # the regions and counts, every step
    xy_pin = torch.from_numpy(xy_h).pin_memory()
    cin_h = torch.empty(n, dtype=torch.uint8).pin_memory()
    cout_h = torch.empty(n, dtype=torch.uint8).pin_memory()
    cnt_h = torch.empty(n, dtype=torch.int32).pin_memory()
    e2e_steps = max(1, min(args.steps, 3))
    barrier(world)
    torch.cuda.synchronize()
    a, b = ev(), ev()
    a.record(stream)
    for q in range(e2e_steps):
        xy.copy_(xy_pin, non_blocking=True)
        out = step(SEED_Z + 200 + q, [ev() for _ in range(6)])
        cin_h.copy_(out["c_in"], non_blocking=True)
        cout_h.copy_(out["c_out"], non_blocking=True)
        cnt_h.copy_(out["count"], non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, world)
    e2e_val = world * (fc + ft) / (e2e_ms / 1e3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_s, M_s = 8192, 2048     # about 10-20 s of host work
        dt, fl = oracle_sample(n_s, M_s)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"one oracle pass (covariance, unblocked Cholesky, simulation, calibration) on the leading "
                         f"{n_s} of {n} sites with M={M_s}: {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": "Cholesky+TRMM TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16/f32/f64 adaptive", "data": "synthetic",
            "config": {"workload": w.name, "n": n, "nb": nb, "M": M, "fixedacc": w.fixedacc, "range": w.beta,
                       "nu": w.nu, "nugget": w.nugget, "l2": "working set (tiles > 1 GB) larger than L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "ms_per_step_median": float(np.median(per_step)), "ms_per_step_min": float(np.min(per_step)),
            "ms_per_step_max": float(np.max(per_step)),
            "chol_trmm": {"tflops": ct_tflops, "ms": ct_ms, "x_fp64_peak": ct_tflops / unit_peaks["fp64_dfma"],
                          "frac_weighted_peak": frac_weighted, "weighted_peak_ms": t_star * 1e3,
                          "flops_by_precision": {k: fch[k] + ftr.get(k, 0.0) for k in fch}},
            "sims_per_s": world * M / (st["rng_trmm"] / 1e3),
            "stages_ms": st,
            "precision_map": {"n_fp64": info["n_fp64"], "n_fp32": info["n_fp32"], "n_fp16": info["n_fp16"],
                              "s": info["s"], "check1": info["check1"], "check2": info["check2"]},
            "roofline": roof,
            "kernels": kern,
            "unit_peaks_tflops": unit_peaks,
            "kernel_timing_pass": {"steps": n_inst, "ms_per_step": inst_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": int(xy_h.nbytes),
                    "d2h_bytes_per_step": int(n * (1 + 1 + 4))},
            "gpu_launches": launches,
            "clocks": clk,
            "wall_s_timed": wall,
        }
        print(json.dumps(line), flush=True)
    V.close()


def run_krige(args, world, rank, local):
    """The universal-kriging workload (16384 noisy observations and a 128 x 128 prediction grid,
    Matern nu = 1, range 0.1, tau^2 = 0.01, tile 512, M = 1024, fixedacc 1e-6, u = 1.6, level
    0.90).  Kriging (W, zhat, v), the map and the factorisation are set up once (their times are
    reported, not in the metric); one step is one batch of M conditional simulations: normal
    draws fused with the mixed-precision TRMM, then the correction with the calibration
    (cr_correct_calibrate: with the double-float product S is never written; with the Ozaki
    product on the tensor cores, --fp64-gemm ozaki, S goes through scratch and W's slices are
    cut once at setup, cr_weights_prepare, as W itself is computed once).  Metric:
    simulations per second, M / (t_rng + t_trmm + t_correct + t_calibrate).  The separate
    correction + calibration calls are timed beside it."""
    import torch
    import mixed_precision_dense_mat_gb300 as cr
    torch.cuda.set_device(local)
    cr.load()
    ozaki = args.fp64_gemm == "ozaki"
    cr.set_option(cr.CR_OPT_FP64_GEMM, cr.CR_GEMM_OZAKI if ozaki else cr.CR_GEMM_DF)
    w = inputgen.WORKLOADS["k"]
    n, n_p, n_o, nb, M = w.n, w.n_pred, w.n_obs, w.nb, w.M
    dev = torch.device("cuda", local)
    xy_h = inputgen.workload_locations(w)
    xy = torch.from_numpy(xy_h).to(dev)
    X = np.column_stack([np.ones(n), xy_h[:, 0], xy_h[:, 1]])
    y_h = inputgen.observation_values(xy_h[n_p:], (1.0, 0.5, -0.3), 0.1, 3)
    yo = torch.from_numpy(y_h).to(dev)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    V = cr.TileMat(n, nb)
    e = [ev() for _ in range(4)]
    e[0].record(stream)
    cr.cov_build(V, xy, w.family, w.sigma2, w.beta, w.nu, nugget=w.nugget, n_pred=n_p, tau2=w.tau2)
    W, zhat, v = cr.krige(V, cr.as_colmajor(torch.from_numpy(X[n_p:]).to(dev))[0],
                          cr.as_colmajor(torch.from_numpy(X[:n_p]).to(dev))[0], yo)
    e[1].record(stream)
    pmap, info = cr.precision_map(V, amp=True, fixedacc=w.fixedacc)
    assert cr.potrf_adaptive(V) == 0
    e[2].record(stream)
    torch.cuda.synchronize()
    t_krige, t_chol = e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])
    Y = cr.colmajor_empty(n, M, torch.float64)

    # the Ozaki product cuts the fixed kriging weights into slices once (cr_weights_prepare),
    # part of the setup like W itself
    Wp, t_prep = None, 0.0
    if ozaki:
        e[2].record(stream)
        Wp = cr.Weights(W)
        e[3].record(stream)
        torch.cuda.synchronize()
        t_prep = e[2].elapsed_time(e[3])

    def correct_calibrate():
        if Wp is not None:
            return cr.correct_calibrate_prepared(Wp, yo, Y, zhat, v, w.u, w.level)
        return cr.correct_calibrate(W, yo, Y, n_p, n_o, zhat, v, w.u, w.level)

    def step(seed, fused=True):
        cr.trmm_sim(V, None, M, seed=seed, out=Y, flags=cr.CR_TRMM_GENERATE)
        if fused:
            return correct_calibrate()
        S = cr.krige_correct(W, yo, Y, n_p, n_o)
        return cr.calibrate(S, zhat, v, w.u, w.level)

    for q in range(args.warmup):
        step(SEED_Z + q)
    torch.cuda.synchronize()
    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if "CUDA_VISIBLE_DEVICES" in os.environ else str(local)
    clocks = ClockSampler(gpu_id)
    barrier(world)
    torch.cuda.synchronize()
    l0 = cr.kernel_launches()
    a, b = ev(), ev()
    a.record(stream)
    for q in range(args.steps):
        out = step(SEED_Z + 100 + q)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = cr.kernel_launches() - l0
    clk = clocks.stop()
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world)
    # the parts of one step, and the unfused path, in a separate pass
    parts = {}
    pe = [ev() for _ in range(3)]
    pe[0].record(stream)
    cr.trmm_sim(V, None, M, seed=SEED_Z + 500, out=Y, flags=cr.CR_TRMM_GENERATE)
    pe[1].record(stream)
    correct_calibrate()
    pe[2].record(stream)
    torch.cuda.synchronize()
    parts["rng_trmm"] = pe[0].elapsed_time(pe[1])
    parts["correct_calibrate"] = pe[1].elapsed_time(pe[2])
    ue = [ev() for _ in range(5)]
    ue[0].record(stream)
    S = cr.krige_correct_prepared(Wp, yo, Y) if Wp is not None else cr.krige_correct(W, yo, Y, n_p, n_o)
    ue[1].record(stream)
    cr.calibrate(S, zhat, v, w.u, w.level)
    ue[2].record(stream)
    if Wp is not None:
        # the same correction cutting W again (cr_krige_correct), for comparison
        cr.krige_correct(W, yo, Y, n_p, n_o, out=S)
    ue[3].record(stream)
    torch.cuda.synchronize()
    parts["correct"] = ue[0].elapsed_time(ue[1])
    parts["calibrate"] = ue[1].elapsed_time(ue[2])
    if Wp is not None:
        parts["correct_without_prepared_weights"] = ue[2].elapsed_time(ue[3])
    corr_flops = 2.0 * n_p * n_o * M
    oz = None
    if ozaki:
        # one more Ozaki correction with per-part device timing: slicing (of R: W's slices are
        # prepared), the slice GEMMs
        # (FP16 tensor-core flops: sum over levels L = 2..9 of (L - 1) 2 n_p M n_o', n_o' = c kc
        # with c = ceil(n_o / 4096) chunks of kc = ceil(n_o / c) rounded up to 128 rows) and the
        # exact accumulation (its algorithmic bytes: the chunk products read once, the
        # double-float accumulator written, read and rewritten per level, Y_p read and S written
        # by the last level)
        cr.timing_reset()
        cr.timing_enable(True)
        cr.krige_correct_prepared(Wp, yo, Y, out=S)
        t = {k: cr.timing_read(k)[0] for k in ("k_oz_slice", "oz_gemm", "k_oz_accum")}
        cr.timing_enable(False)
        cpk = -(-n_o // 4096)
        kc = -(-(-(-n_o // cpk)) // 128) * 128
        kpad = cpk * kc
        gemm_flops = 36 * 2.0 * n_p * M * kpad
        accum_bytes = (36 * (kpad // kc) * 4 + 128) * n_p * M
        oz = {"slice_ms": t["k_oz_slice"], "gemm_ms": t["oz_gemm"], "accum_ms": t["k_oz_accum"],
              "gemm_fp16_tflops": gemm_flops / (t["oz_gemm"] / 1e3) / 1e12,
              "accum_gbs": accum_bytes / (t["k_oz_accum"] / 1e3) / 1e9}
    if rank == 0:
        line = {"metric": "conditional simulations/s (kriging workload)", "value": world * M / (ms / 1e3),
                "unit": "simulations/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16/f32/f64 adaptive; " + ("Ozaki FP16 tensor-core correction" if ozaki else "df correction"),
                "data": "synthetic",
                "config": {"workload": w.name, "n_pred": n_p, "n_obs": n_o, "nb": nb, "M": M, "fixedacc": w.fixedacc,
                           "u": w.u, "level": w.level, "parallelism": f"replicas x{world}"},
                "setup_ms": {"covariance_and_kriging": t_krige, "map_and_cholesky": t_chol,
                             "weights_prepare": t_prep},
                "parts_ms": parts,
                "correction_tflops": corr_flops / (parts["correct"] / 1e3) / 1e12,
                "fp64_gemm": args.fp64_gemm,
                "ozaki_parts": oz,
                "precision_map": {"n_fp64": info["n_fp64"], "n_fp32": info["n_fp32"], "n_fp16": info["n_fp16"], "s": info["s"]},
                "regions": {"q_in": out["q_in"], "q_out": out["q_out"], "inner": int(out["c_in"].sum().item()),
                            "outer": int(out["c_out"].sum().item())},
                "gpu_launches": launches, "clocks": clk}
        print(json.dumps(line), flush=True)
    V.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true", help="skip the per-kernel device timing (no roofline)")
    ap.add_argument("--n", type=int, default=0, help="profiling only: smaller n of the same workload family")
    ap.add_argument("--peaks", action="store_true", help="print the arithmetic units' measured peaks and exit")
    ap.add_argument("--fp64-gemm", default="ozaki", choices=["df", "ozaki"],
                    help="kriging workload: the correction's FP64 product in double-float on the FP32 units, or by "
                         "the Ozaki scheme on the FP16 tensor cores")
    ap.add_argument("--workload", default="headline", choices=["headline", "krige"],
                    help="headline: the Cholesky+TRMM step of the n = 32768 workload (default); krige: conditional "
                         "simulations per second on the kriging workload")
    args = ap.parse_args()
    global WORKLOAD
    if args.n:
        import dataclasses
        WORKLOAD = dataclasses.replace(WORKLOAD, n_pred=args.n, name=WORKLOAD.name.replace("n=32768", f"n={args.n}"))
    world, rank, local = dist_setup()
    if args.peaks:
        run_peaks(local)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.workload == "krige":
            run_krige(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
