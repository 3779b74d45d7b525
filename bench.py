#!/usr/bin/env python3
"""Benchmark of the MoE layout -> dispatch -> combine hot path on one GB300.

One step = mp_layout_dispatch (at this size layout + receive offsets in one
cooperative launch, then the row copy launched as its programmatic dependent; at
up to 16,384 top-k ids, as in the small-batch rows, one kernel) + mp_combine
(launched as the dispatch's programmatic dependent) on the DeepSeek-V3-shaped workload
(R=8 logical ranks x N=4096 tokens, H=7168 bf16, E=256 experts, top-8 uniform
routing), the combine input being synthetic expert outputs, one bf16 row per
receive row, in a buffer of their own.  Inputs are synthetic and
seeded, resident in HBM for the device-timed value; the e2e value adds the
host->device copy of the step's inputs and the device->host copy of its
result, from/to pinned host memory.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead
(a plain single-threaded C program that defines every step).

Multi-GPU: the path has no exchange between GPUs (all R logical ranks live in
one GPU's memory), so N GPUs run N independent replicas (weak scaling); the
timed region is bracketed by a barrier + synchronize and the max over ranks
is reported.
"""
from __future__ import annotations

import argparse
import json
import math
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
    ap.add_argument("--tokens", type=int, default=0,
                    help="override N (tokens per rank), e.g. for small profiler captures")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-rows", action="store_true",
                    help="skip timing the e4m3 dispatch and reduce-scatterv / all-gatherv rows")
    ap.add_argument("--other-rows-scale", type=int, default=1,
                    help="divide the other rows' token counts by this (a cut-down run for "
                         "profiling; >1 also runs them beside --tokens)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    return ap.parse_args()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the slowest replica sets the time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of N independent replicas: every rank's units over the
    slowest rank's time."""
    return units_per_rank * world * steps / (ms_max / 1e3)


def _source_digest(slices) -> str:
    """sha256 over the given pieces of source: whole files, or the text of a file
    from a `begin` marker up to (not including) an `end` marker."""
    import hashlib
    h = hashlib.sha256()
    for sl in slices:
        with open(os.path.join(ROOT, sl["file"]), "rb") as f:
            text = f.read()
        if "begin" in sl:
            b = text.index(sl["begin"].encode())
            e = text.index(sl["end"].encode(), b)
            text = text[b:e]
        h.update(text)
    return h.hexdigest()


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when there is none or when the kernel's
    source (its own text, its launcher and the shared device helpers) has
    changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        if _source_digest(rec["source"]) != rec["source_sha256"]:
            return None
        return int(rec["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(R, N, K, E, H, T, elt=2, scales_per_row=0):
    """Bytes each phase must move (read + write), not padded or dense equivalents.
    offsets: mask + topk ids/weights read, send_row + per-row metadata written;
    rows: each token row read once and written once per destination (+ its scales);
    combine: every receive row read once, each token row written once."""
    layout = R * N * K * 4 + R * N * 4 + R * E * 4 + R * R * 4
    offsets = R * N * K * 8 + R * N * 4 + T * (8 + 8 * K) + R * N * R * 4 + R * R * 4
    rows = R * N * H * elt + T * H * elt + (R * N + T) * scales_per_row * 4 + R * N * R * 4
    combine = T * H * 2 + R * N * H * 2 + R * N * R * 4
    return dict(layout=layout, offsets=offsets, rows=rows, dispatch=offsets + rows,
                combine=combine)


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
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1,
                         "host_cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(name, inp):
    return {"workload": "%s: R=%d logical ranks x N=%d tokens, H=%d %s, E=%d experts, top-%d %s "
                        "routing; layout -> dispatch -> combine of synthetic expert outputs"
                        % (name, inp.R, inp.N, inp.H, inp.dtype, inp.E, inp.K,
                           inp.meta.get("routing", "uniform")),
            "R": inp.R, "N": inp.N, "H": inp.H, "E": inp.E, "K": inp.K,
            "global_batch": inp.R * inp.N,
            "l2": "inputs larger than L2 (x %.0f MB, receive rows and expert outputs ~%.0f MB "
                  "each vs 129 MB L2)"
                  % (inp.R * inp.N * inp.row_bytes / 1e6,
                     inp.R * inp.N * inp.row_bytes * 5.3 / 1e6),
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# the other rows of the path on their own workloads (device-timed)
# ---------------------------------------------------------------------------
def measure_other_rows(steps: int, peak: float, scale: int = 1):
    """The rows besides the dsv3 step: in-kernel quantise-dispatch (e4m3, MXFP8, MXFP4) of
    the dsv3 rows; e4m3 dispatch (R=8, N=8192, H=7168, per-128-channel fp32 scales,
    top-8 of 256) with its bf16 combine; reduce-scatterv / all-gatherv (R=8, H=4096,
    per-rank rows U{0..16384}) and the all-gatherv with quantisation fused in; the
    skewed step (R=16, Zipf routing).  Inputs are synthetic (mostly drawn on the
    device: only the timing is used here; parity on these workloads is in the tests)."""
    import numpy as np
    import torch

    from combine_mp_layout_gb300 import binding as B
    from combine_mp_layout_gb300 import workloads as wl
    from combine_mp_layout_gb300.pipeline import EPPlan, RSVPlan

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    def row(ms, nbytes):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"ms": ms, "algorithmic_bytes": int(nbytes), "GB/s": gbs, "frac_of_peak": gbs / peak}

    out = {}
    # in-kernel e4m3 quantisation on dispatch, on the dsv3 workload
    cfg = wl.CONFIGS["dsv3"]
    R, N, H, E, K = cfg["R"], cfg["N"] // scale, cfg["H"], cfg["E"], cfg["K"]
    rng = np.random.default_rng(0)
    g = torch.Generator(device="cuda").manual_seed(0)
    plan = EPPlan(R, N, K, E, H, "bf16")
    plan.topk_idx.copy_(torch.from_numpy(wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K)))
    plan.topk_weights.copy_(torch.from_numpy(wl.softmax_weights(rng, R, N, K)))
    plan.x.copy_(torch.randn((R, N, H), generator=g, device="cuda").to(torch.bfloat16))
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    torch.cuda.synchronize()
    T = plan.num_recv()
    rq = torch.empty((plan.cap, H), dtype=torch.uint8, device="cuda")
    rs = torch.empty((plan.cap, H // 128), dtype=torch.float32, device="cuda")
    ms_q = timed(lambda: B.check(B.mp_dispatch_rows_e4m3(R, N, H, plan.x, plan.send_row, plan.cap,
                                                          rq, rs)), steps)
    out["dispatch_rows_quantise_e4m3"] = dict(
        row(ms_q, R * N * H * 2 + T * (H + H // 128 * 4) + R * N * R * 4),
        workload="dsv3 rows quantised in-kernel: bf16 in, e4m3 + fp32 scale per 128 channels out")
    rc = torch.empty((plan.cap, H // 32), dtype=torch.uint8, device="cuda")
    ms_mx = timed(lambda: B.check(B.mp_dispatch_rows_mxfp8(R, N, H, plan.x, plan.send_row,
                                                           plan.cap, rq, rc)), steps)
    out["dispatch_rows_quantise_mxfp8"] = dict(
        row(ms_mx, R * N * H * 2 + T * (H + H // 32) + R * N * R * 4),
        workload="dsv3 rows quantised in-kernel: bf16 in, MXFP8 (e4m3 + UE8M0 byte per 32 "
                 "channels) out")
    # the same row copy through the bulk-copy (TMA) engine
    rxb = torch.empty((plan.cap, H), dtype=torch.bfloat16, device="cuda")
    ms_bulk = timed(lambda: B.check(B.mp_dispatch_rows_bulk(R, N, H, B.MP_BF16, plan.x, None,
                                                            plan.send_row, plan.cap, rxb, None,
                                                            plan.dev_err)), steps)
    assert plan.device_error() == 0
    out["dispatch_rows_bulk_copy"] = dict(
        row(ms_bulk, algorithmic_bytes(R, N, K, E, H, T)["rows"]),
        workload="dsv3 rows, bf16, copied by cp.async.bulk through shared memory")
    del rxb
    rq4 = torch.empty((plan.cap, H // 2), dtype=torch.uint8, device="cuda")
    ms_m4 = timed(lambda: B.check(B.mp_dispatch_rows_mxfp4(R, N, H, plan.x, plan.send_row,
                                                           plan.cap, rq4, rc)), steps)
    out["dispatch_rows_quantise_mxfp4"] = dict(
        row(ms_m4, R * N * H * 2 + T * (H // 2 + H // 32) + R * N * R * 4),
        workload="dsv3 rows quantised in-kernel: bf16 in, MXFP4 (two e2m1 codes per byte + "
                 "UE8M0 byte per 32 channels) out")
    del rq4
    # global expert ids with a sentinel (the same scan) and the combined top-k weights
    gids = torch.empty_like(plan.recv_topk_idx)
    ms_g = timed(lambda: B.check(B.mp_dispatch_offsets_global(
        R, N, K, E, plan.topk_idx, plan.topk_weights, plan.is_token_in_rank,
        plan.num_tokens_per_rank, plan.num_tokens_per_expert, plan.cap, E, plan.recv_src_rank,
        plan.recv_src_idx, gids, plan.recv_topk_weights, plan.dest_offsets, plan.rank_prefix,
        plan.num_recv_tokens_per_expert, plan.send_row, plan.dev_err, plan.workspace)), steps)
    cw = torch.empty((R, N, K), dtype=torch.float32, device="cuda")
    ms_cw = timed(lambda: B.check(B.mp_combine_weights(R, N, K, plan.recv_topk_weights, plan.cap,
                                                       plan.send_row, cw, plan.dev_err)), steps)
    assert plan.device_error() == 0
    out["dispatch_offsets_global_ids"] = dict(
        row(ms_g, algorithmic_bytes(R, N, K, E, H, T)["offsets"]),
        workload="dsv3 receive offsets with global expert ids (sentinel E)")
    out["combine_topk_weights"] = dict(row(ms_cw, T * K * 4 + R * N * R * 4 + R * N * K * 4),
                                       workload="dsv3 combined top-k weights")
    del plan, rq, rs, rc, gids, cw
    torch.cuda.empty_cache()

    cfg = wl.CONFIGS["fp8"]
    R, N, H, E, K = cfg["R"], cfg["N"] // scale, cfg["H"], cfg["E"], cfg["K"]
    rng = np.random.default_rng(0)
    plan = EPPlan(R, N, K, E, H, "e4m3")
    plan.topk_idx.copy_(torch.from_numpy(wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K)))
    plan.topk_weights.copy_(torch.from_numpy(wl.softmax_weights(rng, R, N, K)))
    g = torch.Generator(device="cuda").manual_seed(0)
    plan.x.copy_(torch.randn((R, N, H), generator=g, device="cuda").to(torch.float8_e4m3fn))
    plan.x_scales.copy_(torch.rand(plan.x_scales.shape, generator=g, device="cuda") * 1.5 + 0.5)
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    torch.cuda.synchronize()
    T = plan.num_recv()
    y = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
    spr = H // 128
    ms_rows = timed(lambda: B.check(plan.dispatch_rows()), steps)
    ms_comb = timed(lambda: B.check(plan.combine(y)), steps)
    assert plan.device_error() == 0
    out["fp8_dispatch_rows"] = dict(row(ms_rows, R * N * H + T * H + (R * N + T) * spr * 4
                                        + R * N * R * 4), workload="fp8: R=8, N=8192, H=7168 e4m3 "
                                   "+ fp32 scale per 128 channels, E=256, top-8", receive_rows=T)
    out["fp8_combine_bf16"] = row(ms_comb, T * H * 2 + R * N * H * 2 + R * N * R * 4)
    del plan, y
    torch.cuda.empty_cache()

    cfg = wl.CONFIGS["rsv"]
    sizes = np.random.default_rng(0).integers(0, cfg["max_rows"] // scale + 1, cfg["R"]).tolist()
    rp = RSVPlan(cfg["R"], cfg["H"], sizes)
    rp.x.normal_(generator=g)
    rp.shards.normal_(generator=g)
    S, Rr, Hh = rp.S, cfg["R"], cfg["H"]
    ms_rs = timed(lambda: B.check(rp.reducescatterv()), max(5, steps // 4))
    ms_ag = timed(lambda: B.check(rp.allgatherv()), max(5, steps // 4))
    out["reducescatterv"] = dict(row(ms_rs, Rr * S * Hh * 2 + S * Hh * 2),
                                 workload="rsv: R=8, H=4096 bf16, rows per rank U{0..16384}, S=%d" % S)
    out["allgatherv"] = row(ms_ag, S * Hh * 2 + Rr * S * Hh * 2)
    # all-gatherv with the quantisation fused in: rows quantised once, codes and
    # scales written to every rank's copy
    qx = torch.empty((Rr, S, Hh), dtype=torch.uint8, device="cuda")
    qs = torch.empty((Rr, S, Hh // 128), dtype=torch.float32, device="cuda")
    ms_agq = timed(lambda: B.check(B.mp_allgatherv_e4m3(Rr, Hh, sizes, rp.shards, qx, qs)),
                   max(5, steps // 4))
    out["allgatherv_quantise_e4m3"] = dict(
        row(ms_agq, S * Hh * 2 + Rr * S * (Hh + Hh // 128 * 4)),
        workload="rsv shards quantised once (fp32 scale per 128 channels), gathered to 8 ranks")
    del qs
    qc = torch.empty((Rr, S, Hh // 32), dtype=torch.uint8, device="cuda")
    ms_agm = timed(lambda: B.check(B.mp_allgatherv_mxfp8(Rr, Hh, sizes, rp.shards, qx, qc)),
                   max(5, steps // 4))
    out["allgatherv_quantise_mxfp8"] = dict(
        row(ms_agm, S * Hh * 2 + Rr * S * (Hh + Hh // 32)),
        workload="rsv shards quantised once (MXFP8, UE8M0 byte per 32 channels), gathered "
                 "to 8 ranks")
    qx4 = torch.empty((Rr, S, Hh // 2), dtype=torch.uint8, device="cuda")
    ms_ag4 = timed(lambda: B.check(B.mp_allgatherv_mxfp4(Rr, Hh, sizes, rp.shards, qx4, qc)),
                   max(5, steps // 4))
    out["allgatherv_quantise_mxfp4"] = dict(
        row(ms_ag4, S * Hh * 2 + Rr * S * (Hh // 2 + Hh // 32)),
        workload="rsv shards quantised once (MXFP4), gathered to 8 ranks")
    del qx4
    # multi-tensor all-gatherv: e4m3 data and its fp32 scales in one launch
    del qc
    qd = torch.randint(0, 256, (S, Hh), generator=g, device="cuda", dtype=torch.uint8)
    qs = torch.rand((S, Hh // 128), generator=g, device="cuda")
    qso = torch.empty((Rr, S, Hh // 128), dtype=torch.float32, device="cuda")
    ms_mt = timed(lambda: B.check(B.mp_allgatherv_multi(Rr, [Hh, Hh // 128 * 4], sizes, [qd, qs],
                                                        [qx, qso])), max(5, steps // 4))
    out["allgatherv_multi_e4m3_and_scales"] = dict(
        row(ms_mt, (S + Rr * S) * (Hh + Hh // 128 * 4)),
        workload="rsv rows as e4m3 data + fp32 scale per 128 channels, two tensors, one launch")
    del rp, qx, qd, qs, qso
    torch.cuda.empty_cache()

    # Small problems fit in L2 (129 MB), so they rotate through P buffer sets whose
    # combined size is several times L2: a set's inputs and expert outputs have been
    # evicted by the time it is used again, and each kernel reads from HBM.
    L2_BYTES = 129e6

    def n_sets(bytes_per_set):
        return max(2, 1 + int(math.ceil(3 * L2_BYTES / bytes_per_set)))

    s_cap = torch.cuda.Stream()

    def as_graph(fn):  # fn captured once as a CUDA graph (after one call outside)
        s_cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_cap):
            fn()
        torch.cuda.current_stream().wait_stream(s_cap)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        return gr

    def phases(sets, calls, names, n):  # per-call CUDA-event times, us
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(n)]
        for i, ev in enumerate(evs):
            st = sets[i % len(sets)]
            ev[0].record()
            for c, call in enumerate(calls):
                call(st)
                ev[c + 1].record()
        torch.cuda.synchronize()
        return {nm: sum(ev[c].elapsed_time(ev[c + 1]) for ev in evs) / n * 1e3
                for c, nm in enumerate(names)}

    # low-latency expert-major layout at the pages' small-batch shape (R=8, N=128,
    # H=7168, top-8 of 256): LL offsets + LL rows -> weighted LL combine, launched one
    # by one and replayed as one CUDA graph
    R, N, H, E, K = 8, 128, 7168, 256, 8
    cap = R * N * K
    rng = np.random.default_rng(1)
    topk_ll = torch.from_numpy(wl.topk_uniform(rng, R * N, E, K).reshape(R, N, K))
    w_ll = torch.from_numpy(wl.softmax_weights(rng, R, N, K))
    ll_set_bytes = R * N * H * 2 * 2 + cap * H * 2 * 2
    ll_sets = []
    for _ in range(n_sets(ll_set_bytes)):
        plan = EPPlan(R, N, K, E, H, "bf16")
        plan.topk_idx.copy_(topk_ll)
        plan.topk_weights.copy_(w_ll)
        plan.x.normal_(generator=g)
        ll_sets.append(dict(
            plan=plan, eoff=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
            esoff=torch.empty((E, R), dtype=torch.int32, device="cuda"),
            doff=torch.empty(R + 1, dtype=torch.int32, device="cuda"),
            dsoff=torch.empty((R, R), dtype=torch.int32, device="cuda"),
            src=torch.empty(cap, dtype=torch.int32, device="cuda"),
            slot=torch.empty((R, N, K), dtype=torch.int32, device="cuda"),
            rx=torch.empty((cap, H), dtype=torch.bfloat16, device="cuda"),
            yl=torch.randn((cap, H), generator=g, device="cuda").to(torch.bfloat16),
            lo=torch.empty((R, N, H), dtype=torch.bfloat16, device="cuda")))

    ll_bytes = (R * N * K * 8 + cap * 4 + (E + 1) * 4 + E * R * 4  # LL offsets
                + R * N * H * 2 + cap * H * 2 + R * N * K * 4           # LL rows
                + cap * H * 2 + R * N * K * 8 + R * N * H * 2)          # weighted LL combine

    def ll_dispatch(st, rank_major=0):
        p = st["plan"]
        B.check(B.mp_dispatch_ll(R, N, K, E, H, B.MP_BF16, rank_major, p.x, None, p.topk_idx,
                                 None, cap, st["doff"] if rank_major else st["eoff"],
                                 st["dsoff"] if rank_major else st["esoff"], st["src"],
                                 st["slot"], st["rx"], None, p.dev_err))

    def ll_combine(st):
        p = st["plan"]
        B.check(B.mp_combine_ll(R, N, K, H, st["yl"], cap, st["slot"], p.topk_weights, st["lo"],
                                p.dev_err))

    def ll_offsets(st):
        p = st["plan"]
        B.check(B.mp_dispatch_ll_offsets(R, N, K, E, p.topk_idx, None, cap, st["eoff"],
                                         st["esoff"], st["src"], st["slot"], p.dev_err))

    def ll_rows(st):
        p = st["plan"]
        B.check(B.mp_dispatch_ll_rows(R, N, K, H, B.MP_BF16, p.x, None, st["slot"], cap,
                                      st["rx"], None))

    def over_sets(sets, *calls):
        def run():
            for st in sets:
                for c in calls:
                    c(st)
        return run

    def ll_errors():
        return sum(st["plan"].device_error() for st in ll_sets)

    P = len(ll_sets)
    # one call for the LL offsets and rows (the sort, then the row copy as its
    # programmatic dependent), then the weighted combine (the copy's dependent)
    ms_ll = timed(over_sets(ll_sets, ll_dispatch, ll_combine), max(1, steps // P)) / P
    ll_phase_us = phases(ll_sets, [ll_dispatch, ll_combine], ("dispatch_ll", "combine_ll"), steps)
    graph = as_graph(over_sets(ll_sets, ll_dispatch, ll_combine))
    ms_llg = timed(graph.replay, max(1, steps // P)) / P
    assert ll_errors() == 0
    out["low_latency_step_n128"] = dict(
        row(ms_ll, ll_bytes), us_per_step=ms_ll * 1e3, us_per_step_cuda_graph=ms_llg * 1e3,
        phases_us=ll_phase_us, receive_rows=int(cap), buffer_sets=P,
        GBs_cuda_graph=ll_bytes / (ms_llg / 1e3) / 1e9,
        workload="R=8, N=128, H=7168 bf16, E=256, top-8: mp_dispatch_ll (LL offsets counting "
                 "the experts themselves, then the LL rows as a programmatic dependent) + "
                 "weighted LL combine of synthetic expert outputs; %d buffer sets in turn "
                 "(L2 never holds a set's inputs)" % P)

    # the same step as three calls: LL offsets, LL rows, weighted combine
    ms_ll3 = timed(over_sets(ll_sets, ll_offsets, ll_rows, ll_combine), max(1, steps // P)) / P
    ll3_phase_us = phases(ll_sets, [ll_offsets, ll_rows, ll_combine],
                          ("ll_offsets", "ll_rows", "combine_ll"), steps)
    graph3 = as_graph(over_sets(ll_sets, ll_offsets, ll_rows, ll_combine))
    ms_ll3g = timed(graph3.replay, max(1, steps // P)) / P
    assert ll_errors() == 0
    out["low_latency_three_calls_step_n128"] = dict(
        row(ms_ll3, ll_bytes), us_per_step=ms_ll3 * 1e3, us_per_step_cuda_graph=ms_ll3g * 1e3,
        phases_us=ll3_phase_us, GBs_cuda_graph=ll_bytes / (ms_ll3g / 1e3) / 1e9,
        workload="as low_latency_step_n128 with the LL offsets and the LL rows as two calls "
                 "(3 launches)")

    def ll_dispatch_rm(st):
        ll_dispatch(st, rank_major=1)

    ms_rm = timed(over_sets(ll_sets, ll_dispatch_rm, ll_combine), max(1, steps // P)) / P
    assert ll_errors() == 0
    rm_bytes = ll_bytes - (E + 1) * 4 - E * R * 4 + (R + 1) * 4 + R * R * 4
    out["low_latency_rank_major_step_n128"] = dict(
        row(ms_rm, rm_bytes), us_per_step=ms_rm * 1e3,
        workload="as low_latency_step_n128 with rank-major output (rows grouped by the rank "
                 "owning the expert)")
    # the low-latency dispatch with the quantisation in the row copy (e4m3 with an fp32
    # scale per 128 channels, and MXFP8), then the weighted combine of bf16 expert outputs
    for fmt, qcode, sbytes, cbytes in (("e4m3", B.MP_Q_E4M3, H // 128 * 4, H),
                                       ("mxfp8", B.MP_Q_MXFP8, H // 32, H),
                                       ("mxfp4", B.MP_Q_MXFP4, H // 32, H // 2)):
        for st in ll_sets:
            st["rq"] = torch.empty((cap, cbytes), dtype=torch.uint8, device="cuda")
            st["rs"] = torch.empty((cap, sbytes), dtype=torch.uint8, device="cuda")

        def ll_quant(st, qcode=qcode):
            p = st["plan"]
            B.check(B.mp_dispatch_ll_quant(R, N, K, E, H, qcode, 0, p.x, p.topk_idx, None, cap,
                                           st["eoff"], st["esoff"], st["src"], st["slot"],
                                           st["rq"], st["rs"], p.dev_err))

        ms_q = timed(over_sets(ll_sets, ll_quant, ll_combine), max(1, steps // P)) / P
        q_phase_us = phases(ll_sets, [ll_quant, ll_combine], ("dispatch_ll_quant", "combine_ll"),
                            steps)
        assert ll_errors() == 0
        q_bytes = ll_bytes - cap * H * 2 + cap * (cbytes + sbytes)
        out["low_latency_quantised_%s_step_n128" % fmt] = dict(
            row(ms_q, q_bytes), us_per_step=ms_q * 1e3, phases_us=q_phase_us,
            workload="as low_latency_step_n128 with mp_dispatch_ll_quant: bf16 rows quantised "
                     "in the row copy to %s (%s), then the weighted combine of bf16 expert "
                     "outputs" % (fmt, "fp32 scale per 128 channels" if fmt == "e4m3"
                                  else "UE8M0 scale per 32 channels"))
        for st in ll_sets:
            del st["rq"], st["rs"]
    del ll_sets, graph, graph3
    torch.cuda.empty_cache()

    # the DeepSeek-V3 shape at small batches (the pages' EP bench defaults to 128 tokens
    # per rank): the step as timed above (one-call dispatch + combine of synthetic expert
    # outputs, launched one by one), as three calls, and replayed as a CUDA graph
    for nb_tok in (128, 512, 1024):
        inp = wl.make_ep("dsv3", seed=0, N=nb_tok)
        R, N, H, E, K = inp.R, inp.N, inp.H, inp.E, inp.K
        sets = []
        probe = EPPlan(R, N, K, E, H, "bf16")
        probe.load(inp)
        B.check(probe.layout_dispatch())
        torch.cuda.synchronize()
        T = probe.num_recv()
        del probe
        nsets = n_sets(R * N * H * 2 * 2 + T * H * 2 * 2)
        for _ in range(nsets):
            plan = EPPlan(R, N, K, E, H, "bf16")
            plan.load(inp)
            sets.append(dict(plan=plan, y=torch.randn((T, H), generator=g, device="cuda")
                             .to(torch.bfloat16)))
        del inp

        def one(st):
            st["plan"].step(st["y"])

        def three(st):
            st["plan"].step_three_calls(st["y"])

        P = len(sets)
        ms1 = timed(over_sets(sets, one), max(1, steps // P)) / P
        ms3 = timed(over_sets(sets, three), max(1, steps // P)) / P
        graph = as_graph(over_sets(sets, one))
        msg = timed(graph.replay, max(1, steps // P)) / P
        assert sum(st["plan"].device_error() for st in sets) == 0
        ab = algorithmic_bytes(R, N, K, E, H, T)
        nbytes = ab["layout"] + ab["dispatch"] + ab["combine"]
        out["dsv3_small_batch_n%d" % nb_tok] = dict(
            row(ms1, nbytes), us_per_step=ms1 * 1e3, tokens_per_s=R * N / (ms1 / 1e3),
            us_per_step_three_calls=ms3 * 1e3, us_per_step_cuda_graph=msg * 1e3,
            GBs_cuda_graph=nbytes / (msg / 1e3) / 1e9, receive_rows=T, buffer_sets=P,
            workload="dsv3 shape at N=%d tokens per rank: mp_layout_dispatch + mp_combine of "
                     "synthetic expert outputs, eager; %d buffer sets in turn (L2 never holds "
                     "a set's inputs)" % (N, P))
        del sets, graph
    torch.cuda.empty_cache()

    # the skewed workload: Zipf(1.2) routing, rank 0 hot
    inp = wl.make_ep("skew", seed=0, N=wl.CONFIGS["skew"]["N"] // scale)
    R, N, H, E, K = inp.R, inp.N, inp.H, inp.E, inp.K
    plan = EPPlan(R, N, K, E, H, "bf16")
    plan.load(inp)
    del inp
    B.check(plan.layout())
    B.check(plan.dispatch_offsets())
    torch.cuda.synchronize()
    T = plan.num_recv()
    y = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)

    def skew_step():
        plan.step(y)

    ms_sk = timed(skew_step, steps)
    assert plan.device_error() == 0
    ab = algorithmic_bytes(R, N, K, E, H, T)
    nbytes = ab["layout"] + ab["dispatch"] + ab["combine"]
    out["skew_step"] = dict(row(ms_sk, nbytes), tokens_per_s=R * N / (ms_sk / 1e3),
                            receive_rows=T,
                            workload="skew: R=16, N=2048, H=4096 bf16, E=64, top-6 Zipf(1.2); "
                                     "layout + dispatch + combine")
    del plan, y
    torch.cuda.empty_cache()
    return out


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
    over = {"N": args.tokens} if args.tokens > 0 else {}
    inp = wl.make_ep(args.config, seed=args.seed, **over)
    R, N, K, E, H = inp.R, inp.N, inp.K, inp.E, inp.H
    plan = EPPlan(R, N, K, E, H, inp.dtype)
    plan.load(inp)
    torch.cuda.synchronize()
    # the combine's input: synthetic expert outputs (bf16, one per receive row) in a
    # buffer of their own, so that the combine reads HBM rather than the rows the
    # dispatch has just written (some of which would still be in L2)
    B.check(plan.layout_dispatch())
    torch.cuda.synchronize()
    y = torch.empty((max(plan.num_recv(), 1), H), dtype=torch.bfloat16, device="cuda")
    gy = torch.Generator(device="cuda").manual_seed(args.seed + 1)
    for r0 in range(0, y.shape[0], 16384):  # in slices: no full-size fp32 temporary
        y[r0:r0 + 16384].copy_(torch.randn((min(16384, y.shape[0] - r0), H), generator=gy,
                                           device="cuda"))
    stream = torch.cuda.current_stream()

    # warm-up (also checks the run is error-free)
    for _ in range(max(3, args.warmup)):
        plan.step(y)
    torch.cuda.synchronize()
    assert plan.device_error() == 0, B.mp_status_string(plan.device_error())
    T = plan.num_recv()
    ab = algorithmic_bytes(R, N, K, E, H, T, elt=2 if inp.dtype == "bf16" else 1,
                           scales_per_row=0 if inp.dtype == "bf16" else H // 128)
    nb = {"layout_offsets": ab["layout"] + ab["offsets"], "rows": ab["rows"],
          "combine": ab["combine"]}
    nb["dispatch"] = nb["layout_offsets"] + nb["rows"]

    # timed region: K steps, per-phase CUDA events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
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
        B.check(plan.layout_dispatch(), "mp_layout_dispatch")
        e[1].record(stream)
        B.check(plan.combine(y), "mp_combine")
        e[2].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    ph = {"dispatch": 0.0, "combine": 0.0}
    for e in ev:
        ph["dispatch"] += e[0].elapsed_time(e[1])
        ph["combine"] += e[1].elapsed_time(e[2])
    ph = {k: v / args.steps for k, v in ph.items()}
    step_ms = sorted(e[0].elapsed_time(e[2]) for e in ev)  # each step, launch to launch
    step_stats = {"median": step_ms[len(step_ms) // 2], "min": step_ms[0], "max": step_ms[-1]}
    assert plan.device_error() == 0, B.mp_status_string(plan.device_error())

    # The same step as three calls (layout + offsets, rows, combine), timed per call
    # outside the timed region: the split of the dispatch and the gain of the one call.
    three = None
    if N > 0:
        ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
               for _ in range(min(args.steps, 50))]
        for _ in range(3):
            plan.step_three_calls(y)
        torch.cuda.synchronize()
        for e in ev3:
            e[0].record(stream)
            B.check(plan.layout_and_offsets())
            e[1].record(stream)
            B.check(plan.dispatch_rows())
            e[2].record(stream)
            B.check(plan.combine(y))
            e[3].record(stream)
        torch.cuda.synchronize()
        assert plan.device_error() == 0, B.mp_status_string(plan.device_error())
        n3 = len(ev3)
        three = {"layout_offsets": sum(e[0].elapsed_time(e[1]) for e in ev3) / n3,
                 "rows": sum(e[1].elapsed_time(e[2]) for e in ev3) / n3,
                 "combine": sum(e[2].elapsed_time(e[3]) for e in ev3) / n3,
                 "step": sum(e[0].elapsed_time(e[3]) for e in ev3) / n3}

    total_ms = max_over_ranks(total_ms, world, device="cuda")
    ms_step = total_ms / args.steps
    tokens = R * N * world
    value = replica_throughput(R * N, args.steps, world, total_ms)
    step_bytes = nb["dispatch"] + nb["combine"]
    eff_gbs = step_bytes * world / (ms_step / 1e3) / 1e9

    # End to end through the public API with host buffers (pinned): every step
    # copies its inputs host->device, runs layout -> dispatch -> combine and
    # copies its result device->host.  Steps are pipelined the way a serving
    # loop would run them: two buffer sets, the copies of step i+1 / i-1 on
    # their own streams overlapping the kernels of step i.
    e2e = None
    if args.e2e_steps > 0:
        h_topk = torch.from_numpy(inp.topk_idx).pin_memory()
        h_w = torch.from_numpy(inp.topk_weights).pin_memory()
        h_x = inp.x.pin_memory()
        h_xs = inp.x_scales.pin_memory() if inp.x_scales is not None else None
        plans = [plan, EPPlan(R, N, K, E, H, inp.dtype)]
        h_out = [torch.empty(plan.out.shape, dtype=plan.out.dtype).pin_memory() for _ in plans]
        h2d = h_topk.nbytes + h_w.nbytes + h_x.nbytes + (h_xs.nbytes if h_xs is not None else 0)
        d2h = h_out[0].nbytes
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        s_run = stream
        ev_in = [torch.cuda.Event() for _ in plans]
        ev_run = [torch.cuda.Event() for _ in plans]
        ev_out = [torch.cuda.Event() for _ in plans]

        def e2e_steps(n):
            for i in range(n):
                j = i % 2
                p = plans[j]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_run[j])  # step i-2 has consumed p's inputs
                    p.topk_idx.copy_(h_topk, non_blocking=True)
                    p.topk_weights.copy_(h_w, non_blocking=True)
                    p.x.copy_(h_x, non_blocking=True)
                    if h_xs is not None:
                        p.x_scales.copy_(h_xs, non_blocking=True)
                    ev_in[j].record(s_in)
                s_run.wait_event(ev_in[j])
                if i >= 2:
                    s_run.wait_event(ev_out[j])  # step i-2's result has left p.out
                p.step(y, stream=s_run)
                ev_run[j].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_run[j])
                    h_out[j].copy_(p.out, non_blocking=True)
                    ev_out[j].record(s_out)

        e2e_steps(4)
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        e2e_steps(args.e2e_steps)
        s_in.wait_stream(s_out)
        b.record(s_in)
        torch.cuda.synchronize()
        barrier()
        for p in plans:
            assert p.device_error() == 0, B.mp_status_string(p.device_error())
        e_ms = max_over_ranks(a.elapsed_time(b), world, device="cuda")
        e2e = {"value": replica_throughput(R * N, args.e2e_steps, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms / args.e2e_steps,
               "pipelining": "two buffer sets; H2D, kernels and D2H on separate streams"}
        del plans[1]

    # The same step captured once as a CUDA graph and replayed: the device-side time of
    # the three launches without the host's launch cost (beside `value`, not instead).
    s_cap = torch.cuda.Stream()
    s_cap.wait_stream(stream)
    with torch.cuda.stream(s_cap):
        plan.step(y)
    stream.wait_stream(s_cap)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        plan.step(y)
    for _ in range(3):
        step_graph.replay()
    torch.cuda.synchronize()
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record(stream)
    for _ in range(args.steps):
        step_graph.replay()
    gb.record(stream)
    torch.cuda.synchronize()
    assert plan.device_error() == 0, B.mp_status_string(plan.device_error())
    ms_graph = ga.elapsed_time(gb) / args.steps
    del step_graph

    # roofline of the dominant kernel: the combine, the step's largest single kernel (the
    # dispatch phase is two kernels, the cooperative layout + offsets and the row copy)
    peak, peak_kind = peaks()
    dom = "combine"
    achieved = nb[dom] / (ph[dom] / 1e3) / 1e9
    kname = "mp_k_combine<8,1,3,0>"
    traffic = recorded_traffic(kname) if (args.config == "dsv3" and args.tokens == 0) else None
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": traffic,
                "traffic_note": "ncu dram read+write per launch, scaled by tokens from an "
                                "N=1536 capture summarised under profiles/; null if the "
                                "kernel source changed since",
                "all_phases": {k: {"ms": ph[k], "algorithmic_bytes": nb[k],
                                   "GB/s": nb[k] / (ph[k] / 1e3) / 1e9} for k in ph},
                "three_calls_ms": three,
                "three_calls_GBs": None if three is None else {
                    k: nb[k] / (three[k] / 1e3) / 1e9
                    for k in ("layout_offsets", "rows", "combine")}}

    other = None
    if not args.no_other_rows and args.config == "dsv3" and (args.tokens == 0 or
                                                            args.other_rows_scale > 1):
        if args.other_rows_scale > 1:  # a cut-down run (for profiling): token counts / scale
            other = measure_other_rows(max(1, min(args.steps, 100)), peaks()[0],
                                       args.other_rows_scale)
            other["token_counts_divided_by"] = args.other_rows_scale
        else:
            other = measure_other_rows(max(10, min(args.steps, 100)), peaks()[0])

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = time_oracle(inp, args.cpu_budget_s)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
               "kind": "oracle",
               "sample": "first %d of %d tokens per rank, %d ranks, one layout + dispatch + "
                         "combine pass (%.1f s; single-threaded, 1 of the host's %s cores)"
                         % (n, N, R, dt, os.cpu_count())}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": inp.dtype, "data": "synthetic",
            "config": config_block(args.config, inp),
            "effective_hbm_gbs": eff_gbs, "frac_of_8tbs": eff_gbs / world / NOMINAL_HBM_GBS,
            "frac_of_measured_copy_peak": eff_gbs / world / peak,
            "receive_rows": T, "phases_ms": ph, "step_ms": step_stats,
            "ms_per_step_cuda_graph": ms_graph,
            # the pages' bench convention, for comparison only: tokens x hidden bytes per
            # dispatch / combine (no count of the expanded receive rows)
            "send_side_convention": {
                "bytes": R * N * H * (2 if inp.dtype == "bf16" else 1),
                "dispatch_GBs": R * N * H * (2 if inp.dtype == "bf16" else 1)
                                / (ph["dispatch"] / 1e3) / 1e9,
                "combine_GBs": R * N * H * 2 / (ph["combine"] / 1e3) / 1e9},
            "roofline": roofline, "other_rows": other, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 3 * args.steps if N > 0 else 0, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
