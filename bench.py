#!/usr/bin/env python
"""Benchmark of the verify-round MoE layer on one GB300 (or N independent replicas).

Metric: µs per MoE decode layer and HBM GB/s (fraction of peak) vs verify rows
1/4/16.  A step is one round over the 40-layer 35B-A3B-shaped stack
(H 2048, 128 experts, top-8, intermediate 768, int4 blocks of 32 + fp16 scales);
the headline row count is 1, the 4- and 16-row rounds (1 + 3 MTP drafts; 16
near-duplicate lookup-copy rows) run on the same weights and are reported under
"rows".  `value` is achieved HBM GB/s on algorithmic bytes (unique routed-expert
bytes + router + activations in/out), whole job; `us_per_layer` is the same time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --impl reference the CPU oracle is timed instead (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per MoE decode layer and HBM GB/s (fraction of peak) vs verify rows 1/4/16"
UNIT = "GB/s"
L2_NOTE = ("no L2 flush: a 1-row round streams ~0.9 GB of distinct layer weights, "
           "far above the 129 MB L2, so each layer's experts are evicted before reuse")
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (0 = 40)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=1, choices=[1, 4, 16],
                    help="rows of the headline round (1 = the decode-width workload; 4 and 16 "
                         "put that round first, e.g. to profile its first launch)")
    return ap.parse_args()


def peak_bf16():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def reduce_max(v: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the timing rule: slowest rank counts)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_round: float, world: int, ms_round: float) -> float:
    """Replicas: every rank streams its own round, so the job moves world x the bytes
    in the slowest rank's time."""
    return world * bytes_per_round / (ms_round * 1e-3) / 1e9


def layer_bytes(cfg, U, rows):
    return U * cfg.expert_bytes + cfg.router_bytes + rows * cfg.hidden * (2 + 4)


def workload_config(cfg, rows, L):
    return {"workload": f"{cfg.name}: MoE decode layer H{cfg.hidden} E{cfg.experts} top-{cfg.top_k} "
                        f"I{cfg.inter}, int4 blocks of 32 + fp16 scales, {rows} row(s), {L}-layer round",
            "hidden": cfg.hidden, "experts": cfg.experts, "top_k": cfg.top_k, "inter": cfg.inter,
            "rows": rows, "layers": L, "row_sigma": cfg.row_sigma, "seed": cfg.seed, "l2": L2_NOTE}


# ---- clocks during the timed region ---------------------------------------------------

REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (t, sm_mhz, max_mhz, reasons_mask)
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "-i", str(self.index),
               "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            try:
                sm, mx, rs = [v.strip() for v in line.split(",")]
                self.samples.append((time.time(), float(sm), float(mx), int(rs, 16)))
            except Exception:
                pass

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win and self.samples:
            mid = (t0 + t1) / 2
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        mask = 0
        for s in win:
            mask |= s[3]
        reasons = [n for b, n in REASON_BITS.items() if mask & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win)}


# ---- CPU baseline / reference arm: the oracle --------------------------------------------

def oracle_sample(cfg, layers, budget_s, rows=None, sigma=None, warm=0):
    """Times oracle.route + oracle.layer (single-threaded) over `layers` in turn until the
    budget is spent; input generation is outside the timed region."""
    import oracle
    import syngen
    t_total, bytes_total, n = 0.0, 0, 0
    per_layer = []
    i = 0
    while True:
        l = layers[i % len(layers)]
        router = syngen.router(cfg, l)
        xb = syngen.rows(cfg, l, rows, sigma)
        rt0 = oracle.route(router, xb, cfg.top_k)
        ew = syngen.experts_stacked(cfg, l, rt0.union)
        t0 = time.perf_counter()
        rt = oracle.route(router, xb, cfg.top_k)
        oracle.layer(router, xb, cfg.top_k, rt.union, ew)
        dt = time.perf_counter() - t0
        if i >= warm:
            t_total += dt
            bytes_total += layer_bytes(cfg, rt.union.size, xb.shape[0])
            per_layer.append(dt)
            n += 1
        i += 1
        if (t_total >= budget_s and n >= 1) or (budget_s <= 0 and n >= len(layers)):
            break
    return t_total, bytes_total, n


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on one host core.

    A step is a bounded sample of the 1-row round: one layer's routing (router GEMV,
    top-k, weights, union) plus the SwiGLU FFN of one of its routed experts, layers and
    ranks cycling; GB/s counts the bytes that sample touches (router + one expert +
    row in/out).  Input generation is outside the timed region."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import syngen
    cfg = syngen.CONFIGS["a3b_r1"]
    L = args.layers or cfg.layers
    times, byts = [], 0
    for step in range(args.warmup + args.steps):
        l = (step // cfg.top_k) % L
        j = step % cfg.top_k
        router = syngen.router(cfg, l)
        xb = syngen.rows(cfg, l)
        rt0 = oracle.route(router, xb, cfg.top_k)
        ew = syngen.experts_stacked(cfg, l, [int(rt0.ids[0, j])], threads=1)
        t0 = time.perf_counter()
        rt = oracle.route(router, xb, cfg.top_k)
        oracle.expert_ffn(xb[0], ew, 0)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            byts += cfg.expert_bytes + cfg.router_bytes + cfg.hidden * 6
    t = sum(times)
    gbs = byts / t / 1e9
    sample = (f"{len(times)} steps; each = routing of one 1-row layer + the FFN of one of its "
              f"routed experts (layers 0..{L - 1} cycling), oracle only, one host core")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)",
            "config": workload_config(cfg, 1, L),
            "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- our arm ---------------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import spec_verify_layer_gb300 as mv  # fails loudly when the library is missing
    import syngen
    from spec_verify_layer_gb300.weights import Packer, workspace

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    cfg = syngen.CONFIGS["a3b_r1"]
    L = args.layers or cfg.layers
    H = cfg.hidden
    max_rows = 16
    dims = mv.make_dims(H, cfg.experts, cfg.top_k, cfg.inter, max_rows)
    packer = Packer(dims)
    layers = []
    for l in range(L):
        packer.pack_all(lambda e, l=l: syngen.expert(cfg, l, e))
        layers.append(packer.upload(syngen.router(cfg, l), dev))
    wl = [ly.w for ly in layers]
    handle = mv.moe_create(dims, local)
    ws = workspace(dims, max_rows, dev)
    stream = torch.cuda.Stream(dev)
    st = stream.cuda_stream

    def buffers(rows, sigma):
        xs = np.stack([syngen.rows(cfg, l, rows, sigma) for l in range(L)])
        x = torch.from_numpy(xs.view(np.int16)).to(dev)
        out = torch.empty((L, rows, H), dtype=torch.float32, device=dev)
        stats = torch.zeros(L, dtype=torch.int32, device=dev)
        return xs, x, out, stats

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        return reduce_max(v, world, dev)

    def time_rounds(rows, sigma, steps, warmup, sampler=None):
        xs, x, out, stats = buffers(rows, sigma)
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                mv.moe_round(handle, wl, x.data_ptr(), rows, out.data_ptr(), stats.data_ptr(),
                             ws.data_ptr(), ws.numel(), True, st)
        launches_per_round = mv.moe_last_launch_count(handle)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                mv.moe_round(handle, wl, x.data_ptr(), rows, out.data_ptr(), stats.data_ptr(),
                             ws.data_ptr(), ws.numel(), True, st)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        t_wall1 = time.time()
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1))
        assert mv.moe_last_device_status(handle, st) == mv.MOE_OK
        U = stats.cpu().numpy()
        per_round_bytes = sum(layer_bytes(cfg, int(u), rows) for u in U)
        return {"ms_total": ms, "steps": steps, "U": U, "bytes_per_round": per_round_bytes,
                "launches_per_round": launches_per_round, "t_wall": (t_wall0, t_wall1),
                "x": x, "out": out, "xs": xs}

    def round_percentiles(rows, x, out, n):
        """Per-replay device times of the round graph (an event pair around each replay,
        outside the timed region): p10 / p50 / p90 in us per round."""
        stats_q = torch.zeros(L, dtype=torch.int32, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for a0, a1 in evs:
                a0.record(stream)
                mv.moe_round(handle, wl, x.data_ptr(), rows, out.data_ptr(), stats_q.data_ptr(), ws.data_ptr(),
                             ws.numel(), True, st)
                a1.record(stream)
        torch.cuda.synchronize(dev)
        t = sorted(1e3 * a0.elapsed_time(a1) for a0, a1 in evs)
        return {"p10": t[n // 10], "p50": t[n // 2], "p90": t[(9 * n) // 10], "replays": n}

    def single_layers(rows, x, out, n):
        """One moe_decode_layer launch per layer, rotating over the L distinct layers
        (eager, stream-ordered): us per layer, for the fused round's launch saving."""
        with torch.cuda.stream(stream):
            for l in range(L):
                mv.moe_decode_layer(handle, wl[l], x[l].data_ptr(), rows, out[l].data_ptr(), ws.data_ptr(),
                                    ws.numel(), st)
        torch.cuda.synchronize(dev)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a0.record(stream)
            for i in range(n):
                l = i % L
                mv.moe_decode_layer(handle, wl[l], x[l].data_ptr(), rows, out[l].data_ptr(), ws.data_ptr(),
                                    ws.numel(), st)
            a1.record(stream)
        torch.cuda.synchronize(dev)
        assert mv.moe_last_device_status(handle, st) == mv.MOE_OK
        return {"us_per_layer": 1e3 * a0.elapsed_time(a1) / n, "launches": n}

    def profile_phases(rows, x, out, n_rounds):
        """Eager rounds with per-phase device timestamps (outside every timed region)."""
        stats_p = torch.zeros(L, dtype=torch.int32, device=dev)
        mv.moe_profile(handle, True)
        with torch.cuda.stream(stream):
            for _ in range(n_rounds):
                mv.moe_round(handle, wl, x.data_ptr(), rows, out.data_ptr(), stats_p.data_ptr(), ws.data_ptr(),
                             ws.numel(), False, st)
        eager_ms, eager_n = mv.moe_profile_read(handle, mv.KIND_ROUND)
        ph = {k: {"mean_us": v[0], "max_us": v[1]} for k, v in mv.moe_profile_phases(handle).items()}
        mv.moe_profile(handle, False)
        return ph, eager_ms, eager_n

    peak, peak_src = peak_hbm()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    SIGMA = {1: 0.0, 4: 0.5, 16: 0.1}
    R0 = args.rows
    head = time_rounds(R0, SIGMA[R0], args.steps, max(args.warmup, 3))
    sampler.stop()
    clocks = sampler.summary(*head["t_wall"])

    ms_round = head["ms_total"] / head["steps"]
    us_layer = 1e3 * ms_round / L
    value = whole_job_gbs(head["bytes_per_round"], world, ms_round)

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region;
    # right after the device-timed round, under the same conditions
    x1, out1 = head["x"], head["out"]
    stats1 = torch.zeros(L, dtype=torch.int32, device=dev)
    xh = torch.from_numpy(head["xs"].view(np.int16)).pin_memory()
    oh = torch.empty((L, R0, H), dtype=torch.float32).pin_memory()
    e2e_steps = max(10, min(args.steps, 500))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x1.copy_(xh, non_blocking=True)
            mv.moe_round(handle, wl, x1.data_ptr(), R0, out1.data_ptr(), stats1.data_ptr(), ws.data_ptr(),
                         ws.numel(), True, st)
            oh.copy_(out1, non_blocking=True)
            stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            x1.copy_(xh, non_blocking=True)
            mv.moe_round(handle, wl, x1.data_ptr(), R0, out1.data_ptr(), stats1.data_ptr(), ws.data_ptr(),
                         ws.numel(), True, st)
            oh.copy_(out1, non_blocking=True)
            stream.synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0) / e2e_steps
    e2e = {"value": world * head["bytes_per_round"] / t_e2e / 1e9, "unit": UNIT,
           "h2d_bytes_per_step": int(xh.numel() * 2), "d2h_bytes_per_step": int(oh.numel() * 4),
           "us_per_layer": 1e6 * t_e2e / L, "steps": e2e_steps}


    # rows sweep on the same weights
    sweep = {}
    for rows in (r for r in (1, 4, 16) if r != R0):
        sigma, name = SIGMA[rows], f"a3b_r{rows}"
        r = time_rounds(rows, sigma, max(20, args.steps // 4), max(args.warmup, 3))
        msr = r["ms_total"] / r["steps"]
        gbs = r["bytes_per_round"] / (msr * 1e-3) / 1e9
        sweep[f"r{rows}"] = {"workload": name, "us_per_layer": 1e3 * msr / L, "us_per_round": 1e3 * msr,
                             "hbm_gbs": gbs, "frac_of_peak": gbs / peak,
                             "unique_experts_per_layer": float(np.mean(r["U"])),
                             "picks_per_layer": rows * cfg.top_k,
                             "tokens_per_round_equiv_per_s": rows / (msr * 1e-3)}
        sweep[f"r{rows}"]["phases_per_layer_us"] = profile_phases(rows, r["x"], r["out"], 3)[0]
    # the same 4-row round with the routing tail skip at the page's rank 7 (an
    # approximation: experts every row ranks 7th or lower are not evaluated)
    mv.moe_set_tail_skip(handle, 7)
    try:
        r = time_rounds(4, 0.5, max(20, args.steps // 4), max(args.warmup, 3))
    finally:
        mv.moe_set_tail_skip(handle, 0)
    msr = r["ms_total"] / r["steps"]
    gbs = r["bytes_per_round"] / (msr * 1e-3) / 1e9
    sweep["r4_tail7"] = {"workload": "a3b_r4 with routing tail skip at rank 7", "us_per_layer": 1e3 * msr / L,
                         "us_per_round": 1e3 * msr, "hbm_gbs": gbs, "frac_of_peak": gbs / peak,
                         "unique_experts_per_layer": float(np.mean(r["U"])),
                         "tokens_per_round_equiv_per_s": 4 / (msr * 1e-3)}

    # The price of a verify column: rounds of R = 1..16 rows on the same 40-layer stack
    # (the draft rows at sigma 0.5 around the first row, as for 4 rows), a short timing
    # each; R <= 7 runs on the CUDA cores, R >= 8 on the tensor cores.
    by_rows = {}
    for rows in range(1, 17):
        r = time_rounds(rows, 0.0 if rows == 1 else 0.5, max(20, args.steps // 40), max(args.warmup, 3))
        msr = r["ms_total"] / r["steps"]
        gbs = r["bytes_per_round"] / (msr * 1e-3) / 1e9
        by_rows[str(rows)] = {"us_per_layer": round(1e3 * msr / L, 3), "hbm_gbs": round(gbs, 1),
                              "unique_experts_per_layer": round(float(np.mean(r["U"])), 3)}
    sweep["rows_sweep"] = {"workload": "a3b layers, R = 1..16 rows, draft rows at sigma 0.5",
                           "by_rows": by_rows}

    # The prefill-width layer (many tokens per call: counting sort by expert, per-expert
    # GEMMs): PF_T tokens of diverse rows, layers cycling so every call streams distinct
    # weights; device time over the calls.
    sweep["prefill"] = prefill_leg(mv, cfg, wl, handle, dev, stream, L, max(10, args.steps // 50),
                                   max(args.warmup, 3))

    # The round is one kernel launch (k_round): its average launch duration is the timed
    # region's per-step time, from CUDA events on the launching stream.  A separate
    # eager pass records where the time goes inside it (device timestamps per phase).
    alg_per_launch = float(head["bytes_per_round"])
    avg_launch_us = 1e3 * ms_round
    achieved = alg_per_launch / (avg_launch_us * 1e-6) / 1e9
    prof_rounds = max(3, min(20, args.steps // 50))
    phases, eager_ms, eager_n = profile_phases(R0, x1, out1, prof_rounds)
    pct = round_percentiles(R0, x1, out1, max(20, min(200, args.steps // 10)))
    single = single_layers(R0, x1, out1, max(L, min(4 * L, args.steps)))
    roofline = {"bound": "hbm", "kernel": "k_round", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": read_traffic("k_round", L, R0), "peak_source": peak_src,
                "alg_bytes_per_launch": alg_per_launch, "avg_launch_us": avg_launch_us,
                "launch": f"one cooperative launch per {L}-layer round, timed over {args.steps} graph replays",
                "phases_per_layer_us": phases,
                "eager_round_us": 1e3 * eager_ms / max(eager_n, 1),
                "round_us_percentiles": pct,
                "single_layer_launches": single}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, b, n = oracle_sample(cfg, list(range(L)), budget_s=10.0)
        cpu = {"value": b / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "us_per_layer": 1e6 * t / n,
               "sample": f"{n} single-row layers of the same stack, oracle route + layer only, "
                         f"one host core, ~10 s of CPU work"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": max(args.warmup, 3), "ms_per_step": ms_round, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded counter-based generator; random int4 weights, bf16 rows)",
                "config": workload_config(cfg, R0, L),
                "us_per_layer": us_layer, "us_per_round": 1e3 * ms_round,
                "hbm_gbs_per_gpu": value / world, "frac_of_peak": value / world / peak,
                "tokens_per_round_equiv_per_s": R0 / (ms_round * 1e-3),
                "unique_experts_per_layer": float(np.mean(head["U"])),
                "rows": {f"r{R0}": {"us_per_layer": us_layer, "hbm_gbs": value / world,
                                "frac_of_peak": value / world / peak,
                                "unique_experts_per_layer": float(np.mean(head["U"]))}, **sweep},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": int(head["launches_per_round"] * args.steps)}
        print(json.dumps(line), flush=True)
    mv.moe_destroy(handle)
    if world > 1:
        dist.destroy_process_group()
    return 0


PF_T = 2048


def prefill_leg(mv, cfg, wl, handle, dev, stream, L, steps, warmup):
    import numpy as np
    import torch
    import syngen
    T = PF_T
    xs = [torch.from_numpy(syngen.rows(cfg, l, T, 1.0).view(np.int16)).to(dev) for l in range(min(L, 4))]
    out = torch.empty((T, cfg.hidden), dtype=torch.float32, device=dev)
    counts = torch.zeros(cfg.experts, dtype=torch.int32, device=dev)
    nbytes = mv.moe_prefill_workspace_bytes(mv.make_dims(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, 16), T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = stream.cuda_stream

    def call(i):
        l = i % L
        mv.moe_prefill_layer(handle, wl[l], xs[l % len(xs)].data_ptr(), T, out.data_ptr(), counts.data_ptr(),
                             ws.data_ptr(), nbytes, st)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            call(warmup + i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    assert mv.moe_last_device_status(handle, st) == mv.MOE_OK
    us = 1e3 * e0.elapsed_time(e1) / steps
    U = int((counts.cpu().numpy() > 0).sum())
    flops = 2.0 * T * cfg.experts * cfg.hidden + 6.0 * T * cfg.top_k * cfg.hidden * cfg.inter
    byts = layer_bytes(cfg, U, T)
    peak, src = peak_bf16()
    tflops = flops / (us * 1e-6) / 1e12
    return {"workload": f"{T} tokens (rows x0 + 1.0 N(0,1)) of the {cfg.name} layer, one moe_prefill_layer call",
            "tokens": T, "us_per_layer": us, "tokens_per_s": T / (us * 1e-6), "tflops": tflops,
            "bf16_peak_tflops": peak, "peak_source": src, "frac_of_bf16_peak": tflops / peak,
            "alg_flops": flops, "unique_experts": U, "hbm_gbs": byts / (us * 1e-6) / 1e9,
            "launches_per_call": mv.moe_last_launch_count(handle), "steps": steps}


def read_traffic(kernel, layers, rows):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (its recorded source digest matches) for a round of `rows`
    rows; scaled from the captured layer count to `layers` (traffic grows in
    proportion).  Else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "spec_verify_layer_gb300", "csrc", "moe_verify.cu")
    try:
        kv = dict(l.split(":", 1) for l in open(path) if ":" in l and not l.startswith("#"))
        kv = {k.strip(): v.strip() for k, v in kv.items()}
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if kv.get("kernel") == kernel and kv.get("source_sha256_16") == digest and int(kv.get("rows", "1")) == rows:
            return float(kv["dram_bytes_per_launch"]) * layers / float(kv["layers"])
    except Exception:
        pass
    return None


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
