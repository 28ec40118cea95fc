"""Benchmark of the batched Dion / Orth-Dion optimizer step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--variant orth|dion|mixed]
    python bench.py --configs all|models|sweep  # one line per workload configuration, then the
                                                # memory -> compute crossover of the rank sweep
    python bench.py --impl reference ...      # the float64 CPU oracle, timed on host cores

One "step" is the whole hot path -- phases (a)-(e) of every matrix of the
workload -- through the C ABI.  The default workload is every weight matrix
of a 28-layer Llama-3B (196 matrices, rank = min(m, n)/16, fp32 state, bf16
gradients), synthetic seeded inputs.  The state X, G, R (28 GB) is far larger than
L2, so no L2 flush is needed between steps.

Prints ONE JSON line on rank 0.  With --gpus N > 1 (launched by torchrun)
every rank runs its own full replica of the workload (weak scaling, no data
collective); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
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

METRIC = "Dion/Orth-Dion step ms & effective GB/s, 3B shapes; % of HBM/TC roofline"
PHASES = "abcde"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--configs", default=None, choices=["all", "models", "sweep"],
                    help="measure every configuration (one JSON line each) instead of the headline")
    ap.add_argument("--workload", default="llama3b_28L_rdiv16")
    ap.add_argument("--variant", default="orth", choices=["orth", "dion", "mixed"])
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=14,
                    help="matrix groups of the host-fed end-to-end step (copy/compute overlap)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-muon", action="store_true", help="skip the Muon comparator line on the same matrices")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


NOMINAL_HBM_GBS = 8000.0        # the spec-sheet figure, reported beside the measured copy rate
TF32_PER_BF16 = 1.1 / 2.25      # nominal dense tf32 / bf16 ratio (context only)


def measure_tf32_tflops(dev, size=8192, reps=10):
    """Dense TF32 tensor-core throughput on this GPU: cuBLAS fp32 matmul with
    TF32 enabled, size^3, best of ``reps`` (a burst, like the bf16 peak it sits
    beside).  The contractions here are 3xTF32 (three tf32 products per
    fp32-accurate product), so their peak in fp32-equivalent flops is this / 3."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(size, size, device=dev)
        b = torch.randn(size, size, device=dev)
        c = torch.empty(size, size, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * size ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def tensor_peak(peaks):
    """3xTF32 peak in fp32-equivalent TFLOP/s and where it comes from."""
    if peaks.get("tf32_tflops"):
        return peaks["tf32_tflops"] / 3.0, "measured here: cuBLAS TF32 8192^3 burst / 3 (3xTF32)"
    return peaks["bf16_tflops"] * TF32_PER_BF16 / 3.0, \
        peaks["source"] + " bf16 burst x 1.1/2.25 (tf32) / 3 (3xTF32)"


# DRAM traffic of one k_epi launch per element of X, from the ncu capture of the
# GPT-160M case on the current kernel (three streamed-state slots: 1.2320 GB read +
# 0.6347 GB written for 8.49e7 elements); the traffic of a launch is this times the
# launch's elements.  Set EPI_TRAFFIC_CURRENT to False when k_epi changes, until it
# is captured again.
EPI_TRAFFIC_BYTES_PER_ELEM = (1231990784 + 634691328) / 84934656
EPI_TRAFFIC_CURRENT = True


def variant_of(args):
    return lambda i: ("orth", "dion")[i % 2] if args.variant == "mixed" else args.variant


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            t0 = time.perf_counter()
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.rows.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(max(0.0, 0.1 - (time.perf_counter() - t0)))

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4)
                          if len(r) > 5 + k and r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- multi-rank
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank steps its own full copy of the workload
    (weak scaling), and the job is done when the last rank is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(step_bytes: float, ms_per_step: float, world: int) -> float:
    """Whole-job algorithmic GB/s: all ranks' bytes over the slowest rank's time."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------- CUDA arm
def build_state(wl, dev, args, variant):
    import torch
    from rank_orthonormalized_optimizer_03_b300 import synth
    mats = []
    for k, spec in enumerate(wl.mats):
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=args.seed, device=dev)
        # warm start: the raw Gaussian draw scaled by 1/sqrt(n); the first step
        # orthonormalises through orth(M V) itself.
        V0 = (V0_raw / math.sqrt(spec.n)).contiguous()
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=V0, eta=spec.eta, beta=spec.beta,
                         variant=variant(k), scale=spec.scale))
    torch.cuda.synchronize()
    return mats


def bench_config(wl, variant_name, world):
    """The workload the line is quoted on (the same for both arms)."""
    state_gb = sum(s.m * s.n for s in wl.mats) * (8 + (2 if wl.g_dtype == "bf16" else 4)) / 1e9
    ranks = sorted({s.r for s in wl.mats})
    return {"workload": wl.name, "matrices": len(wl.mats), "elements": wl.elems, "g_dtype": wl.g_dtype,
            "ranks": ranks, "variant": variant_name, "parallelism": f"replica{world}",
            "l2": f"inputs {state_gb:.2f} GB >> 126 MB L2, no flush"}


def roofline_entry(bound, achieved, peak, unit, source):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "peak_source": source}


def measure(wl, args, dev, world, variant_name, peaks, min_timed_s=1.0):
    """Time K steps of one workload through the C ABI (CUDA events on the launching
    stream, phase boundaries marked by events) and build its JSON fields."""
    import torch
    import torch.distributed as dist
    from rank_orthonormalized_optimizer_03_b300 import accounting, dion

    vof = (lambda i: ("orth", "dion")[i % 2]) if variant_name == "mixed" else (lambda i: variant_name)
    mats = build_state(wl, dev, args, vof)
    plan = dion.Plan(mats)
    stream = torch.cuda.current_stream()
    cost = accounting.step_cost(wl.mats, wl.g_dtype, vof)
    plan.upload()
    t0 = time.perf_counter()
    for _ in range(args.warmup):
        plan.step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / max(1, args.warmup)
    steps = args.steps
    if min_timed_s and est * steps < min_timed_s:
        steps = min(2000, int(math.ceil(min_timed_s / max(est, 1e-5))))

    def barrier():
        if world > 1:
            dist.barrier()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(steps):
            ev[s][0].record(stream)
            for ph in range(5):
                plan.phases(ph, ph)
                ev[s][ph + 1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    phase_ms = {PHASES[p]: statistics.mean(ev[s][p].elapsed_time(ev[s][p + 1]) for s in range(steps))
                for p in range(5)}
    ms_per_step = total_ms / steps
    status = plan.status()
    bad = sum(1 for v in status if v & dion.FATAL)
    shifted = sum(1 for v in status if v & dion.DION_MAT_SHIFTED)

    step = cost["step"]
    value = job_throughput_gbs(step.bytes, ms_per_step, world)
    tpeak, tsrc = tensor_peak(peaks)
    hbm = peaks["hbm_gbs"]
    hsrc = peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"

    # the whole step against max(algorithmic bytes / HBM, algorithmic flops / 3xTF32 peak)
    t_mem = step.bytes / (hbm * 1e9) * 1e3
    t_ten = step.flops / (tpeak * 1e12) * 1e3
    step_roof = {"bound": "hbm" if t_mem >= t_ten else "tensor", "ideal_ms": round(max(t_mem, t_ten), 4),
                 "hbm_ms": round(t_mem, 4), "tensor_ms": round(t_ten, 4),
                 "frac": round(max(t_mem, t_ten) / ms_per_step, 4),
                 "frac_vs_nominal_8tbs": round(max(step.bytes / (NOMINAL_HBM_GBS * 1e9) * 1e3, t_ten) / ms_per_step, 4),
                 "algorithmic_bytes": step.bytes, "algorithmic_flops": step.flops,
                 "impl_extra_bytes": round(cost["impl_extra_bytes"])}

    # the dominant phase's kernel against its own schedule's bytes and flops
    dom = max(phase_ms, key=phase_ms.get)
    dom_kernel = {"a": "k_stream<0> (P = M V)", "b": "orth(P) chain", "c": "k_stream<1> (W = M^T U)",
                  "d": "orth(W) chain", "e": "k_epi"}[dom]
    c = cost[dom]
    secs = phase_ms[dom] * 1e-3
    gbs, tfl = c.bytes / secs / 1e9, c.flops / secs / 1e12
    hbm_roof = roofline_entry("hbm", gbs, hbm, "GB/s", hsrc)
    hbm_roof["frac_vs_nominal_8tbs"] = round(gbs / NOMINAL_HBM_GBS, 4)
    ten_roof = roofline_entry("tensor", tfl, tpeak, "TFLOP/s", tsrc)
    if c.bytes / (hbm * 1e9) >= c.flops / (tpeak * 1e12):
        roof, other = hbm_roof, ten_roof
    else:
        roof, other = ten_roof, hbm_roof
    traffic = EPI_TRAFFIC_BYTES_PER_ELEM * wl.elems if dom == "e" and EPI_TRAFFIC_CURRENT else None
    roof.update({"traffic": round(traffic) if traffic else None, "kernel": dom_kernel, "phase": dom,
                 "per_launch_ms": round(phase_ms[dom], 4),
                 "algorithmic_per_launch": {"bytes": c.bytes, "flops": c.flops}, "other_roofline": other})
    if traffic:
        roof["traffic_note"] = "ncu dram bytes of the GPT-160M k_epi capture, scaled by elements"
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "precision": "fp32 state; contractions as 3xTF32 tensor-core products with fp32 accumulation",
        "config": bench_config(wl, variant_name, world),
        "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
        "tflops": round(world * step.flops / (ms_per_step * 1e-3) / 1e12, 3),
        "step_roofline": step_roof,
        "roofline": roof,
        "peaks": {"hbm_gbs": hbm, "tensor_3xtf32_tflops": round(tpeak, 1),
                  "tf32_tflops_measured": round(peaks["tf32_tflops"], 1) if peaks.get("tf32_tflops") else None,
                  "bf16_tflops_burst": peaks["bf16_tflops"]},
        "clocks": clk.summary(),
        "gpu_launches": plan.launches_per_step * steps,
        "status_failed": bad, "status_shifted": shifted,
    }
    return out, plan, mats, cost


def run_cuda(args):
    import torch
    import torch.distributed as dist
    from rank_orthonormalized_optimizer_03_b300 import build, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    peaks = load_peaks()
    peaks["tf32_tflops"] = measure_tf32_tflops(dev)
    if args.configs:
        run_configs(args, dev, world, rank, peaks)
    else:
        wl = workloads.by_name(args.workload)
        out, plan, mats, cost = measure(wl, args, dev, world, args.variant, peaks, min_timed_s=0)
        if not args.no_e2e:
            out["e2e"] = run_e2e(args, mats, cost["step"].bytes, out["ms_per_step"], world)
        if not args.no_muon:
            plan.close()
            del plan, mats
            torch.cuda.empty_cache()
            plan = None
            mu = measure_muon(wl, args, dev, "bf16")
            out["muon_comparator"] = dict(mu, muon_over_dion=round(mu["ms_per_step"] / out["ms_per_step"], 3),
                                          note="same matrices, Muon momentum + cubic Newton-Schulz (cuBLAS bf16 "
                                               "GEMMs); the pages' Dion3 claim of up to 6x lower step time than "
                                               "Muon states no hardware")
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(wl, args, args.cpu_seconds)
        if plan is not None:
            plan.close()
        if rank == 0:
            print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def config_list(which):
    from rank_orthonormalized_optimizer_03_b300 import workloads
    out = []
    if which in ("all", "models"):
        for name in ("gpt160m_12L_rdiv4", "llama3b_28L_rdiv16", "llama3b_28L_rdiv4"):
            for v in ("orth", "dion"):
                out.append((workloads.by_name(name), v))
    if which in ("all", "sweep"):
        for shape in workloads.SWEEP_SHAPES:
            for r in workloads.SWEEP_RANKS:
                for v in ("orth", "dion"):
                    out.append((workloads.sweep(shape, r), v))
    return out


def crossover(lines):
    """Memory -> compute crossover of the rank sweep, per shape and variant: the
    first rank whose ideal tensor time exceeds its ideal HBM time (from the byte
    and flop counts), and the first rank whose measured step takes 1.25x the
    r = 32 step (where the measured time starts to follow the flops)."""
    out = []
    groups = {}
    for ln in lines:
        wl = ln["config"]["workload"]
        if not wl.startswith("sweep_"):
            continue
        shape = wl[len("sweep_"):].split("_r")[0]
        groups.setdefault((shape, ln["config"]["variant"]), []).append(ln)
    for (shape, v), lst in sorted(groups.items()):
        lst.sort(key=lambda x: x["config"]["ranks"][0])
        ranks = [x["config"]["ranks"][0] for x in lst]
        model = next((r for r, x in zip(ranks, lst) if x["step_roofline"]["bound"] == "tensor"), None)
        base = lst[0]["ms_per_step"]
        meas = next((r for r, x in zip(ranks, lst) if x["ms_per_step"] > 1.25 * base), None)
        out.append({"shape": shape, "variant": v, "crossover_rank_model": model, "crossover_rank_measured": meas,
                    "ms_per_step": {r: x["ms_per_step"] for r, x in zip(ranks, lst)},
                    "step_roofline_frac": {r: x["step_roofline"]["frac"] for r, x in zip(ranks, lst)}})
    return out


MUON_ITERS = 5


def measure_muon(wl, args, dev, precision, iters=MUON_ITERS, min_timed_s=1.0):
    """The Muon comparator on the same matrices (momentum + `iters` cubic
    Newton-Schulz iterations + update), timed like the Dion step."""
    import torch
    from rank_orthonormalized_optimizer_03_b300 import dion, synth
    mats = []
    for k, spec in enumerate(wl.mats):
        X0, _, G = synth.device_matrix_inputs(spec, wl, k, seed=args.seed, device=dev)
        mats.append(dict(X=X0, G=G, B=torch.zeros_like(X0), eta=spec.eta, mu=0.95, scale=spec.scale))
    plan = dion.MuonPlan(mats, iters=iters, precision=precision)
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    for _ in range(args.warmup):
        plan.step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / max(1, args.warmup)
    # about two seconds of timed steps, at most --steps and at least 3
    steps = max(3, min(args.steps, int(math.ceil(2.0 / max(est, 1e-5)))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        plan.step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # flops of the iteration: two GEMMs of 2 k^2 l each (k = min, l = max side) per matrix
    fl = iters * sum(4.0 * min(s.m, s.n) ** 2 * max(s.m, s.n) for s in wl.mats)
    out = {"comparator": "muon", "workload": wl.name, "precision": precision, "ns_iters": iters,
           "ms_per_step": round(ms, 4), "steps": steps, "ns_tflops": round(fl / (ms * 1e-3) / 1e12, 2),
           "launches_per_step": plan.launches_per_step}
    plan.close()
    del plan, mats
    torch.cuda.empty_cache()
    return out


def run_configs(args, dev, world, rank, peaks):
    """One JSON line per configuration (GPT-160M, Llama-3B at rank min/16 and min/4,
    the rank sweep; both variants), then one line with the sweep's crossover.  The
    model workloads also get a line of the Muon comparator on the same matrices
    (bf16 and tf32 Newton-Schulz) with the Dion / Muon step-time ratio."""
    import torch
    lines = []
    muon_done = {}
    for wl, v in config_list(args.configs):
        out, plan, mats, _ = measure(wl, args, dev, world, v, peaks, min_timed_s=1.0)
        plan.close()
        del plan, mats
        torch.cuda.empty_cache()
        lines.append(out)
        if rank == 0:
            print(json.dumps(out), flush=True)
        if not wl.name.startswith("sweep_") and wl.name not in muon_done:
            muon_done[wl.name] = [measure_muon(wl, args, dev, p) for p in ("bf16", "tf32")]
        if wl.name in muon_done and rank == 0:
            for mu in muon_done[wl.name]:
                print(json.dumps(dict(mu, dion_variant=v, dion_ms_per_step=out["ms_per_step"],
                                      muon_over_dion=round(mu["ms_per_step"] / out["ms_per_step"], 3))),
                      flush=True)
    if rank == 0 and any(x["config"]["workload"].startswith("sweep_") for x in lines):
        print(json.dumps({"sweep_crossover": crossover(lines)}), flush=True)


def h2d_probe_gbs(dev, nbytes=1 << 30, reps=3):
    """Plain pinned host -> device copy rate of this machine: one transfer of
    ``nbytes``, best of ``reps`` (CUDA events)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = float("inf")
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del h, d
    return nbytes / (best * 1e-3) / 1e9


def run_e2e(args, mats, step_bytes, device_ms, world):
    """The same step through the public API with host-resident gradients:
    dion.HostFedStep copies every step's gradients from pinned host memory (one
    transfer per group of matrices, each overlapping the previous group's step),
    and the per-matrix status words are read back (which synchronises).  The
    state (X, R, V) and the gradients are the workload's."""
    import torch
    from rank_orthonormalized_optimizer_03_b300 import dion
    stepper = dion.HostFedStep(mats, groups=args.e2e_groups)
    for i, d in enumerate(stepper.mats):
        stepper.host_grad(i).copy_(d["G"].cpu())
    h2d = stepper.h2d_bytes()
    d2h = 4 * len(mats)
    steps = max(2, min(args.steps, 10))
    stepper.step()
    stepper.status()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        stepper.step()
        stepper.status()        # device -> host read of the step's result
    # the slowest rank's time, as for the device-timed value
    dt = max_over_ranks((time.perf_counter() - t0) / steps * 1e3, world, mats[0]["X"].device) * 1e-3
    groups = len(stepper.plans)
    stepper.close()
    del stepper
    torch.cuda.empty_cache()
    link = h2d_probe_gbs(mats[0]["X"].device)
    link_ms = h2d / (link * 1e9) * 1e3
    return {"value": round(world * step_bytes / dt / 1e9, 2), "unit": "GB/s", "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": f"HostFedStep, {groups} groups, one pinned-slab transfer per group "
                   "(the copy of group g+1 overlaps the step of group g)",
            "h2d_probe_gbs": round(link, 2), "h2d_link_ms": round(link_ms, 3),
            "bound_ms": round(max(device_ms, link_ms), 3),
            "frac_of_bound": round(max(device_ms, link_ms) / (dt * 1e3), 4),
            "result": "per-matrix status words (the optimizer state stays on the device)"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample_inputs(wl, seed, idx):
    import numpy as np
    from rank_orthonormalized_optimizer_03_b300 import synth
    spec = wl.mats[idx]
    X0, V0_raw, G = synth.host_matrix_inputs(spec, wl, seed * 1_000_003 + idx)
    G64 = synth.bf16_bits_to_f32(G).astype(np.float64) if G.dtype == np.uint16 else G.astype(np.float64)
    return spec, X0.astype(np.float64), G64, V0_raw / math.sqrt(spec.n)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:
        return os.cpu_count()


def oracle_time(wl, args, idxs):
    import numpy as np
    from oracle import dion_oracle as O
    from rank_orthonormalized_optimizer_03_b300 import accounting
    vof = variant_of(args)
    secs, nbytes, names = 0.0, 0.0, []
    for i in idxs:
        spec, X, G, V = oracle_sample_inputs(wl, args.seed, i)
        R = np.zeros_like(X)
        t0 = time.perf_counter()
        O.oracle_step(X, G, R, V, spec.eta, spec.beta, vof(i), spec.scale)
        secs += time.perf_counter() - t0
        nbytes += accounting.step_algorithmic(spec.m, spec.n, spec.r, wl.g_dtype, vof(i)).bytes
        names.append(spec.name)
    return secs, nbytes, names


def cpu_baseline(wl, args, budget_s):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    workload's matrices (in workload order until ~budget_s seconds)."""
    secs, nbytes, names = 0.0, 0.0, []
    i = 0
    while i < len(wl.mats) and (secs < budget_s or i < min(7, len(wl.mats))):
        s, b, n = oracle_time(wl, args, [i])
        secs, nbytes, names = secs + s, nbytes + b, names + n
        i += 1
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle", "sample": f"first {len(names)} of {len(wl.mats)} matrices "
            f"({names[0]}..{names[-1]}), one step each, {secs:.1f} s; value = their algorithmic bytes / time"}


def run_reference(args):
    """The float64 oracle on the host cores, on this arm's workload and metric.
    Each step is a bounded sample of the workload: matrices in workload order
    (rotating) until the step's share of a ~150 s budget is spent, at least one
    matrix; value = the sample's algorithmic bytes / oracle time."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from rank_orthonormalized_optimizer_03_b300 import workloads
    wl = workloads.by_name(args.workload)
    per_step = 150.0 / max(1, args.steps + args.warmup)
    nxt = 0

    def one_step():
        nonlocal nxt
        t_all, b_all, count = 0.0, 0.0, 0
        while count == 0 or t_all < per_step:
            t, b, _ = oracle_time(wl, args, [nxt])
            t_all, b_all, count = t_all + t, b_all + b, count + 1
            nxt = (nxt + 1) % len(wl.mats)
        return t_all, b_all, count

    for _ in range(args.warmup):
        one_step()
    secs, nbytes, nmat = 0.0, 0.0, 0
    for _ in range(args.steps):
        t, b, c = one_step()
        secs, nbytes, nmat = secs + t, nbytes + b, nmat + c
    value = nbytes / secs / 1e9
    sample = (f"{nmat} matrix steps of {wl.name} over {args.steps} steps (workload order, rotating; "
              f"~{per_step:.1f} s of oracle time per step), oracle_step once each; "
              f"value = algorithmic bytes of the sample / oracle time")
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": bench_config(wl, args.variant, world),
           "impl": "reference", "execution": "float64 oracle on the host cores (rank 0 only)",
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
