#!/usr/bin/env python3
"""Benchmark of the MoE layout -> dispatch -> combine hot path on one GB300.

One step = mp_layout + mp_dispatch (scan + row copy) + mp_combine on the
DeepSeek-V3-shaped workload (R=8 logical ranks x N=4096 tokens, H=7168 bf16,
E=256 experts, top-8 uniform routing), the combine input being the
dispatched rows themselves (identity experts).  Inputs are synthetic and
seeded, resident in HBM for the device-timed value; the e2e value adds the
host->device copy of the step's inputs and the device->host copy of its
result, from/to pinned host memory.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead
(the reference arm of this build: a plain single-threaded C program).

Multi-GPU: the path has no exchange between GPUs (all R logical ranks live in
one GPU's memory), so N GPUs run N independent replicas (weak scaling); the
timed region is bracketed by a barrier + synchronize and the max over ranks
is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and effective HBM GB/s (% of ~8 TB/s) on 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--config", default="dsv3", choices=["dsv3", "skew", "fp8", "tiny"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(R, N, K, E, H, T, elt=2, scales_per_row=0):
    """Bytes each phase must move (read + write), not padded or dense equivalents."""
    layout = R * N * K * 4 + R * N * 4 + R * E * 4 + R * R * 4
    meta = R * N * K * 8 + R * N * 4 + T * (8 + 8 * K) + R * N * R * 4 + R * R * 4
    dispatch = R * N * H * elt + T * H * elt + (R * N + T) * scales_per_row * 4 + meta
    combine = T * H * 2 + R * N * H * 2 + R * N * R * 4
    return dict(layout=layout, dispatch=dispatch, combine=combine)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step(inp_np, E):
    import oracle
    topk, w, x = inp_np
    _, _, mask, _ = oracle.layout(topk, E)
    out, _ = oracle.dispatch(x, topk, w, mask, E)
    oracle.combine(out["recv_x"], out["send_row"])


def time_oracle(inp, budget_s: float, min_tokens: int = 64):
    """Times the oracle (layout + dispatch + combine, single thread) on the first
    n tokens of every rank, n grown until one pass takes a sizeable share of the
    budget (or reaches the full workload).  Returns (tokens/s, n, seconds)."""
    from combine_mp_layout_gb300 import workloads as wl
    import oracle
    oracle.build()
    xb = wl.bf16_bits(inp.x)
    n = min(inp.N, min_tokens)
    while True:
        args = (inp.topk_idx[:, :n].copy(), inp.topk_weights[:, :n].copy(),
                xb[:, :n].copy())
        t0 = time.perf_counter()
        oracle_step(args, inp.E)
        dt = time.perf_counter() - t0
        if n >= inp.N or dt > budget_s / 3:
            return inp.R * n / dt, n, dt
        n = min(inp.N, max(n * 2, int(n * (budget_s / 3) / max(dt, 1e-3))))


def reference_arm(args):
    """--impl reference: the oracle as it stands, on rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from combine_mp_layout_gb300 import workloads as wl
    import oracle
    oracle.build()
    inp = wl.make_ep(args.config, seed=args.seed)
    xb = wl.bf16_bits(inp.x)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    # sample size: first n tokens per rank, sized so that one step fits per_step
    n = min(inp.N, 16)
    while n < inp.N:
        a = (inp.topk_idx[:, :n].copy(), inp.topk_weights[:, :n].copy(), xb[:, :n].copy())
        t0 = time.perf_counter()
        oracle_step(a, inp.E)
        if time.perf_counter() - t0 > per_step / 2:
            break
        n = min(inp.N, n * 2)
    a = (inp.topk_idx[:, :n].copy(), inp.topk_weights[:, :n].copy(), xb[:, :n].copy())
    for _ in range(args.warmup):
        oracle_step(a, inp.E)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(a, inp.E)
    dt = time.perf_counter() - t0
    v = inp.R * n * args.steps / dt
    sample = ("first %d tokens of each of the %d ranks of the %s workload per step "
              "(layout + dispatch + combine)" % (n, inp.R, args.config))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(args.config, inp),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(name, inp):
    return {"workload": "%s: R=%d logical ranks x N=%d tokens, H=%d %s, E=%d experts, top-%d %s "
                        "routing; layout -> dispatch -> combine of the dispatched rows"
                        % (name, inp.R, inp.N, inp.H, inp.dtype, inp.E, inp.K,
                           inp.meta.get("routing", "uniform")),
            "R": inp.R, "N": inp.N, "H": inp.H, "E": inp.E, "K": inp.K,
            "global_batch": inp.R * inp.N,
            "l2": "inputs larger than L2 (x %.0f MB, receive rows ~%.0f MB vs 129 MB L2)"
                  % (inp.R * inp.N * inp.row_bytes / 1e6,
                     inp.R * inp.N * inp.row_bytes * 5.3 / 1e6),
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    import torch.distributed as dist

    from combine_mp_layout_gb300 import binding as B
    from combine_mp_layout_gb300 import workloads as wl
    from combine_mp_layout_gb300.pipeline import EPPlan

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    B.lib()  # fail loudly if the library is missing
    inp = wl.make_ep(args.config, seed=args.seed)
    R, N, K, E, H = inp.R, inp.N, inp.K, inp.E, inp.H
    plan = EPPlan(R, N, K, E, H, inp.dtype)
    plan.load(inp)
    torch.cuda.synchronize()
    y = None
    if inp.dtype != "bf16":  # e4m3 dispatch, bf16 combine of synthetic expert outputs
        B.check(plan.layout())
        B.check(plan.dispatch())
        torch.cuda.synchronize()
        y = wl.gathered_bf16(plan.num_recv(), H, seed=args.seed + 1).cuda()
    stream = torch.cuda.current_stream()

    # warm-up (also checks the run is error-free)
    for _ in range(max(3, args.warmup)):
        plan.step(y)
    torch.cuda.synchronize()
    assert plan.device_error() == 0, B.mp_status_string(plan.device_error())
    T = plan.num_recv()
    nb = algorithmic_bytes(R, N, K, E, H, T, elt=2 if inp.dtype == "bf16" else 1,
                           scales_per_row=0 if inp.dtype == "bf16" else H // 128)

    # timed region: K steps, per-phase CUDA events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        e = ev[i]
        e[0].record(stream)
        B.check(plan.layout())
        e[1].record(stream)
        B.check(plan.dispatch())
        e[2].record(stream)
        B.check(plan.combine(y))
        e[3].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    ph = {"layout": 0.0, "dispatch": 0.0, "combine": 0.0}
    for e in ev:
        ph["layout"] += e[0].elapsed_time(e[1])
        ph["dispatch"] += e[1].elapsed_time(e[2])
        ph["combine"] += e[2].elapsed_time(e[3])
    ph = {k: v / args.steps for k, v in ph.items()}
    assert plan.device_error() == 0, B.mp_status_string(plan.device_error())

    t_max = torch.tensor([total_ms], dtype=torch.float64, device="cuda")
    if world > 1:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    total_ms = float(t_max.item())
    ms_step = total_ms / args.steps
    tokens = R * N * world
    value = tokens * args.steps / (total_ms / 1e3)
    step_bytes = nb["layout"] + nb["dispatch"] + nb["combine"]
    eff_gbs = step_bytes * world / (ms_step / 1e3) / 1e9

    # end to end through the public API with host buffers (pinned)
    e2e = None
    if args.e2e_steps > 0:
        h_topk = torch.from_numpy(inp.topk_idx).pin_memory()
        h_w = torch.from_numpy(inp.topk_weights).pin_memory()
        h_x = inp.x.pin_memory()
        h_xs = inp.x_scales.pin_memory() if inp.x_scales is not None else None
        h_out = torch.empty(plan.out.shape, dtype=plan.out.dtype).pin_memory()
        h2d = h_topk.nbytes + h_w.nbytes + h_x.nbytes + (h_xs.nbytes if h_xs is not None else 0)
        d2h = h_out.nbytes

        def e2e_step():
            plan.topk_idx.copy_(h_topk, non_blocking=True)
            plan.topk_weights.copy_(h_w, non_blocking=True)
            plan.x.copy_(h_x, non_blocking=True)
            if h_xs is not None:
                plan.x_scales.copy_(h_xs, non_blocking=True)
            plan.step(y)
            h_out.copy_(plan.out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        b.record(stream)
        barrier()
        e_ms = torch.tensor([a.elapsed_time(b)], dtype=torch.float64, device="cuda")
        if world > 1:
            dist.all_reduce(e_ms, op=dist.ReduceOp.MAX)
        e2e = {"value": tokens * args.e2e_steps / (float(e_ms.item()) / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": float(e_ms.item()) / args.e2e_steps}

    # roofline of the dominant kernel (the larger of dispatch and combine)
    peak, peak_kind = peaks()
    dom = "dispatch" if ph["dispatch"] >= ph["combine"] else "combine"
    achieved = nb[dom] / (ph[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": {"dispatch": "mp_dispatch (scan + row copy)",
                                           "combine": "mp_k_combine"}[dom],
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "traffic": None,
                "all_phases": {k: {"ms": ph[k], "algorithmic_bytes": nb[k],
                                   "GB/s": nb[k] / (ph[k] / 1e3) / 1e9} for k in ph}}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = time_oracle(inp, args.cpu_budget_s)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": "first %d of %d tokens per rank, %d ranks, one layout + dispatch + "
                         "combine pass (%.1f s)" % (n, N, R, dt)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": inp.dtype, "data": "synthetic",
            "config": config_block(args.config, inp),
            "effective_hbm_gbs": eff_gbs, "frac_of_8tbs": eff_gbs / world / NOMINAL_HBM_GBS,
            "frac_of_measured_copy_peak": eff_gbs / world / peak,
            "receive_rows": T, "phases_ms": ph,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 4 * args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
