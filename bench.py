"""Benchmark of the batched Dion / Orth-Dion optimizer step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--variant orth|dion|mixed]
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
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama3b_28L_rdiv16")
    ap.add_argument("--variant", default="orth", choices=["orth", "dion", "mixed"])
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-groups", type=int, default=14,
                    help="matrix groups of the host-fed end-to-end step (copy/compute overlap)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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


# The contractions run as 3xTF32 on the tensor core (three tf32 products per
# fp32-accurate product).  Their peak, in algorithmic (fp32-equivalent) flops,
# is the dense tf32 rate / 3, and the tf32 rate is the measured bf16 rate times
# the nominal tf32 / bf16 ratio 1.1 / 2.25.  The sustained bf16 figure applies:
# the kernels are timed inside a step that runs for a large fraction of a second.
TF32_PER_BF16 = 1.1 / 2.25


def tensor_peak_3xtf32(peaks):
    return peaks["bf16_tflops_sustained"] * TF32_PER_BF16 / 3.0


# DRAM traffic of one k_epi launch per element of X, from the ncu capture of the
# GPT-160M case (profiles/k_epi_gpt160m_rdiv4.md: 1.8646 GB for 8.49e7 elements);
# the traffic of a launch is this times the launch's elements.  Set
# EPI_TRAFFIC_CURRENT to False when k_epi changes, until it is captured again.
EPI_TRAFFIC_BYTES_PER_ELEM = (1232205312 + 632418560) / 84934656
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
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.rows.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.2)

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
def build_state(wl, dev, args):
    import torch
    from rank_orthonormalized_optimizer_03_b300 import synth
    vof = variant_of(args)
    mats = []
    for k, spec in enumerate(wl.mats):
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=args.seed, device=dev)
        # warm start: the raw Gaussian draw scaled by 1/sqrt(n); the first step
        # orthonormalises through orth(M V) itself.
        V0 = (V0_raw / math.sqrt(spec.n)).contiguous()
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=V0, eta=spec.eta, beta=spec.beta,
                         variant=vof(k), scale=spec.scale))
    torch.cuda.synchronize()
    return mats


def bench_config(wl, args, world):
    """The workload the line is quoted on (the same for both arms)."""
    state_gb = sum(s.m * s.n for s in wl.mats) * (8 + (2 if wl.g_dtype == "bf16" else 4)) / 1e9
    return {"workload": wl.name, "matrices": len(wl.mats), "elements": wl.elems, "g_dtype": wl.g_dtype,
            "variant": args.variant, "parallelism": f"replica{world}",
            "l2": f"inputs {state_gb:.0f} GB >> 126 MB L2, no flush"}


def run_cuda(args):
    import torch
    import torch.distributed as dist
    from rank_orthonormalized_optimizer_03_b300 import accounting, build, dion, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    wl = workloads.by_name(args.workload)
    mats = build_state(wl, dev, args)
    plan = dion.Plan(mats)
    stream = torch.cuda.current_stream()
    cost = accounting.step_cost(wl.mats, wl.g_dtype, variant_of(args))
    plan.upload()
    for _ in range(args.warmup):
        plan.step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- timed region: K steps, phase boundaries marked with events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            ev[s][0].record(stream)
            for ph in range(5):
                plan.phases(ph, ph)
                ev[s][ph + 1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    phase_ms = {PHASES[p]: statistics.mean(ev[s][p].elapsed_time(ev[s][p + 1]) for s in range(args.steps))
                for p in range(5)}
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    from rank_orthonormalized_optimizer_03_b300.dion import DION_MAT_SHIFTED, FATAL
    status = plan.status()
    bad = sum(1 for v in status if v & FATAL)
    shifted = sum(1 for v in status if v & DION_MAT_SHIFTED)

    step_bytes = cost["step"].bytes
    value = job_throughput_gbs(step_bytes, ms_per_step, world)

    peaks = load_peaks()
    # dominant phase: the one with the largest share of the step
    dom = max(phase_ms, key=phase_ms.get)
    dom_kernel = {"a": "k_stream<0> (P = M V)", "b": "orth(P) chain", "c": "k_stream<1> (W = M^T U)",
                  "d": "orth(W) chain", "e": "k_epi"}[dom]
    c = cost[dom]
    secs = phase_ms[dom] * 1e-3
    gbs = c.bytes / secs / 1e9
    tfl = c.flops / secs / 1e12
    tpeak = tensor_peak_3xtf32(peaks)
    hbm_frac = gbs / peaks["hbm_gbs"]
    ten_frac = tfl / tpeak
    hbm_roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(hbm_frac, 4),
                "peak_source": peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    ten_roof = {"bound": "tensor", "achieved": round(tfl, 2), "peak": round(tpeak, 1), "unit": "TFLOP/s",
                "frac": round(ten_frac, 4),
                "peak_source": peaks["source"] + " sustained bf16 x 1.1/2.25 (tf32) / 3 (3xTF32)"}
    # the binding roofline is the one whose ideal time is longer
    if c.bytes / (peaks["hbm_gbs"] * 1e9) >= c.flops / (tpeak * 1e12):
        roof, other = hbm_roof, ten_roof
    else:
        roof, other = ten_roof, hbm_roof
    traffic = EPI_TRAFFIC_BYTES_PER_ELEM * wl.elems if dom == "e" else None
    roof.update({"traffic": round(traffic) if traffic and EPI_TRAFFIC_CURRENT else None, "kernel": dom_kernel,
                 "phase": dom, "per_launch_ms": round(phase_ms[dom], 4),
                 "algorithmic_per_launch": {"bytes": c.bytes, "flops": c.flops}, "other_roofline": other})
    if traffic:
        roof["traffic_note"] = "ncu dram bytes of the GPT-160M k_epi capture, scaled by elements"
        if not EPI_TRAFFIC_CURRENT:
            roof["traffic_earlier_revision"] = round(traffic)
            roof["traffic_note"] += "; captured on an earlier revision of the kernel"
    step_roof_ms = max(step_bytes / (peaks["hbm_gbs"] * 1e9), cost["step"].flops / (tpeak * 1e12)) * 1e3
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, plan, mats, stream, step_bytes, world)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "precision": "fp32 state; contractions as 3xTF32 tensor-core products with fp32 accumulation",
        "config": bench_config(wl, args, world),
        "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
        "tflops": round(world * cost["step"].flops / (ms_per_step * 1e-3) / 1e12, 3),
        "step_roofline_ms": round(step_roof_ms, 3),
        "step_roofline_frac": round(step_roof_ms / ms_per_step, 4),
        "roofline": roof,
        "clocks": clk.summary(),
        "gpu_launches": plan.launches_per_step * args.steps,
        "status_failed": bad, "status_shifted": shifted,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, args, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, plan, mats, stream, step_bytes, world):
    """The same step through the public API with host-resident gradients:
    dion.HostFedStep copies every step's gradients from pinned host memory, in
    groups whose copy overlaps the previous group's step, and the per-matrix
    status words are read back (which synchronises)."""
    from rank_orthonormalized_optimizer_03_b300 import dion
    host_g = [d["G"].to("cpu").pin_memory() for d in mats]
    stepper = dion.HostFedStep(mats, groups=args.e2e_groups)
    h2d = stepper.h2d_bytes()
    d2h = 4 * len(mats)
    steps = max(1, min(args.steps, 5))
    stepper.step(host_g)
    stepper.status()
    t0 = time.perf_counter()
    for _ in range(steps):
        stepper.step(host_g)
        stepper.status()        # device -> host read of the step's result
    dt = (time.perf_counter() - t0) / steps
    groups = len(stepper.plans)
    stepper.close()
    return {"value": round(world * step_bytes / dt / 1e9, 2), "unit": "GB/s", "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": f"HostFedStep, {groups} groups (copy of group g+1 overlaps the step of group g)"}


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
        nbytes += sum(c.bytes for c in accounting.phase_cost(spec.m, spec.n, spec.r, wl.g_dtype, vof(i)).values())
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
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from rank_orthonormalized_optimizer_03_b300 import workloads
    wl = workloads.by_name(args.workload)
    # each step: one matrix group (a layer's worth, 7 matrices or the whole workload if smaller)
    group = min(7, len(wl.mats))
    groups = [list(range(k, min(k + group, len(wl.mats)))) for k in range(0, len(wl.mats), group)]
    for w in range(args.warmup):
        oracle_time(wl, args, groups[w % len(groups)][:1])
    secs, nbytes = 0.0, 0.0
    for s in range(args.steps):
        t, b, _ = oracle_time(wl, args, groups[s % len(groups)])
        secs += t
        nbytes += b
    value = nbytes / secs / 1e9
    sample = (f"each step: one group of {group} matrices of {wl.name} (rotating), oracle_step once each; "
              f"value = algorithmic bytes of the sample / oracle time")
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": bench_config(wl, args, world),
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
