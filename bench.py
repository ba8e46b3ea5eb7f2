#!/usr/bin/env python
"""Benchmark of the masked-attention hot path on GB300.

One step = one pass of the whole path over one batch: plan build from the
mask (host checks, GPU planner, one header readback, exact allocation,
CSR + payload + schedule) followed by the masked forward.  Metric: TFLOPS on
visible (q, k) pairs (4 * d FLOPs per visible pair), per step, with the plan
build time reported beside it.  Default workload: the largest single-GPU
configuration, video-style block-sparse attention (B=1, H=24, S=32768,
d=128, 64x64 logical blocks active at 10% plus the diagonal, bf16).  The same
line carries `per_config`: forward time, TFLOPS on visible pairs, roofline
fraction and plan build time for each of the five workloads.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on bounded samples of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "masked attn fwd TFLOPS on visible pairs, % of GB300 BF16 roofline; plan build µs"
# clock cycles of the sleep kernel queued ahead of each timed forward launch (about 0.1 ms)
SLEEP_CYCLES = 200_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_DESC = {
    "tiny_causal": "tiny causal B=1 H=2 S=256 d=64 BSHD",
    "sliding_sink": "sliding window 1024 + sink 4, B=4 H=16 S=4096 d=128 BSHD",
    "varlen_doc_causal": "varlen document-causal THD 16384 tokens / 8 docs, H=16 d=128",
    "video_block_sparse": "block-sparse 64x64 blocks 10% + diagonal, B=1 H=24 S=32768 d=128",
    "prefix_alibi_softcap": "prefixLM + ALiBi + softcap 50, B=2 H=32 S=8192 d=128",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="video_block_sparse", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload table (the headline workload only)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


FWD_SOURCES = ("attn_fwd.cu", "attn_fwd_pair.cu", "attn_fwd_kt.cu", "ptx.cuh", "internal.h")
DECODE_SOURCES = ("attn_decode.cu", "ptx.cuh", "internal.h")


def kernel_hash(files=FWD_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_sparse_masked_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def fwd_kernel_name(w) -> str:
    """The forward kernel the library launches for this workload."""
    mods = bool(w.softcap and w.softcap > 0) or w.alibi_slopes is not None
    if w.mask_kind == "intervals" and not mods:
        return "k_fwd_pair (attention forward, two Q tiles per task)"
    if (w.mask_kind == "blocks" and not mods and w.d == 128 and w.block_q % 64 == 0
            and w.block_kv % 64 == 0):
        return "k_fwd_kt (keys-major attention forward, 64-row halves x pairs of 64x64 quadrants)"
    return "k_fwd (attention forward, one Q tile per task)"


def known_traffic(workload: str):
    """DRAM bytes per forward launch from a committed ncu summary, if it matches this kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    kh = kernel_hash(DECODE_SOURCES if workload == "decode_paged" else FWD_SOURCES)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == kh:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Work of every rank in one step over the (max-over-ranks) step time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def visible_flops(info: dict, Hq: int, d: int) -> float:
    vp = info["visible_pairs"]
    heads = Hq if info["mask_heads"] == 1 else 1
    return 4.0 * d * vp * heads


def algorithmic_bytes(w, info: dict) -> float:
    """Bytes one forward launch must move at least once: Q, K, V read, O and
    LSE written, and the plan it reads (CSR offsets and lists, task list, and
    the packed predicate payload of the partial entries; the keys-major
    kernel reads the per-entry quadrant bytes instead and the predicate words
    only of quadrants that are not fully visible, none for 64-aligned block
    masks over lengths that are multiples of 64)."""
    qkv = sum(t.numel() * t.element_size() for t in (w.q, w.k, w.v))
    o = w.q.numel() * w.q.element_size()
    lse = 4 * w.Hq * w.total_q
    hdr = info["header"]
    plan_meta = 4 * (2 * (info["mask_heads"] * hdr[0] + 1) + hdr[1] + hdr[2]) + 16 * info["num_tasks"]
    if fwd_kernel_name(w).startswith("k_fwd_kt"):
        aligned = w.Sq % 64 == 0 and w.Sk % 64 == 0
        payload = hdr[1] + (0 if aligned else info["payload_bytes"])
    else:
        payload = info["payload_bytes"]
    return float(qkv + o + lse + plan_meta + payload)


def roofline(flops: float, alg_bytes: float, ms: float, peaks: dict, peak_src: str, traffic):
    """The bound of one launch: tensor (visible FLOPs at the bf16 peak) or HBM
    (algorithmic bytes at the copy bandwidth), whichever takes longer at its
    peak; the fraction is the achieved rate of that resource over its peak."""
    tflops_peak = float(peaks["bf16_tflops"])
    gbs_peak = float(peaks["hbm_gbs"])
    t_tensor = flops / (tflops_peak * 1e12)
    t_hbm = alg_bytes / (gbs_peak * 1e9)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    if t_tensor >= t_hbm:
        r = {"bound": "tensor", "achieved": tflops, "peak": tflops_peak, "unit": "TFLOP/s",
             "frac": tflops / tflops_peak,
             "peak_source": f"{peak_src} bf16 dense burst (kernel timed alone per event pair)"}
    else:
        r = {"bound": "hbm", "achieved": gbs, "peak": gbs_peak, "unit": "GB/s", "frac": gbs / gbs_peak,
             "peak_source": f"{peak_src} HBM copy bandwidth"}
    r.update({"traffic": traffic, "alg_bytes": alg_bytes, "tflops": tflops, "alg_gbs": gbs,
              "t_tensor_ms_at_peak": t_tensor * 1e3, "t_hbm_ms_at_peak": t_hbm * 1e3})
    return r


def plan_kw(w) -> dict:
    """Block plans ask for quadrant bits only: the library keeps them alone
    when they are exact (64-aligned blocks over 64-multiple lengths), which
    is all the Direct 64x64 forward reads; otherwise it builds the words."""
    return {"quadrant_payload": True} if w.mask_kind == "blocks" else {}


def time_forward_alone(runner, dp, plan, flush, stream, reps: int, choice: int = 0):
    """Event pairs around each forward launch; L2 flushed first, and a queued
    sleep keeps the host ahead so that the pair brackets the launch itself."""
    import torch
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for i in range(reps):
        flush.zero_()
        torch.cuda._sleep(SLEEP_CYCLES)
        kev[i][0].record(stream)
        runner.forward(dp, plan, choice=choice)
        kev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in kev]


def time_plan_builds(fa, runner, dp, flush, stream, reps: int, **kw):
    """Host microseconds of each build (the call, including its one header
    read-back) and stream milliseconds until its last planner kernel ends."""
    import torch
    host_us, gpu_ms = [], []
    for _ in range(reps):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        p = runner.build_plan(dp, **kw)
        e1.record(stream)
        host_us.append(fa.fa_plan_info_get(p)["build_us"])
        torch.cuda.synchronize()
        gpu_ms.append(e0.elapsed_time(e1))
        p.free()
    return statistics.median(host_us), statistics.median(gpu_ms)


def time_backward(fa, runner, dp, flush, stream, reps: int, fwd_flops: float, peaks: dict):
    """fa_bwd (Delta, dQ, dK/dV launches) timed alone; TFLOPS on visible pairs
    with the usual 2.5x-forward count (five d-deep products per pair)."""
    import torch
    w = dp.w
    if w.d != 128:
        return {"skipped": "the backward supports head_dim 128"}
    plan = runner.build_plan(dp, backward=True)
    runner.forward(dp, plan)
    dout = torch.randn(dp.q.shape, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    for _ in range(2):
        runner.backward(dp, plan, dout)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for i in range(reps):
        flush.zero_()
        torch.cuda._sleep(SLEEP_CYCLES)
        ev[i][0].record(stream)
        runner.backward(dp, plan, dout)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    b_us = fa.fa_plan_info_get(plan)["build_us"]
    plan.free()
    tf = 2.5 * fwd_flops / (ms * 1e-3) / 1e12
    return {"bwd_ms": ms, "tflops": tf, "frac_bf16_peak": tf / float(peaks["bf16_tflops"]),
            "flops_convention": "2.5 x forward visible FLOPs (10 d per visible pair)",
            "plan_build_us_with_backward_view": b_us, "launches": 3}


def per_config_table(fa, runner, W, flush, stream, peaks, peak_src, reps: int, seed: int):
    """Forward alone, plan build and roofline of every workload (one seed)."""
    import torch
    out = {}
    for name in WORKLOAD_DESC:
        w = W.make(name, seed)
        dp = runner.to_device(w)
        plan = runner.build_plan(dp)
        info = fa.fa_plan_info_get(plan, count_visible=True)
        flops = visible_flops(info, w.Hq, w.d)
        for _ in range(3):
            runner.forward(dp, plan)
        torch.cuda.synchronize()
        ms = statistics.mean(time_forward_alone(runner, dp, plan, flush, stream, reps))
        # the other physical plan for this mask (Tessera-style plan choice),
        # timed the same way; the library's rule picks the default one
        alt = None
        if w.mask_kind == "blocks" and w.d == 128 and w.block_q % 64 == 0 and w.block_kv % 64 == 0:
            alt = ("coarsened_128x128", fa.FA_FWD_COARSENED, "direct_64x64")
        elif w.mask_kind == "intervals" and not (w.softcap and w.softcap > 0) and w.alibi_slopes is None:
            alt = ("one_q_tile_per_task", fa.FA_FWD_ONE_TILE, "two_q_tiles_per_task")
        choices = None
        if alt is not None:
            for _ in range(2):
                runner.forward(dp, plan, choice=alt[1])
            torch.cuda.synchronize()
            alt_ms = statistics.mean(time_forward_alone(runner, dp, plan, flush, stream, reps, alt[1]))
            choices = {alt[2] + "_ms": ms, alt[0] + "_ms": alt_ms, "default": alt[2],
                       "regret_of_default": ms / min(ms, alt_ms)}
        plan.free()
        b_us, b_ms = time_plan_builds(fa, runner, dp, flush, stream, max(10, reps // 2))
        if plan_kw(w):
            qb_us, qb_ms = time_plan_builds(fa, runner, dp, flush, stream, max(10, reps // 2), **plan_kw(w))
            choices = dict(choices or {}, plan_build_us_quadrant_payload=qb_us,
                           plan_gpu_ms_quadrant_payload=qb_ms)
        rf = roofline(flops, algorithmic_bytes(w, info), ms, peaks, peak_src, known_traffic(name))
        bwd = time_backward(fa, runner, dp, flush, stream, max(5, reps // 2), flops, peaks)
        out[name] = {"workload": WORKLOAD_DESC[name], "fwd_ms": ms, "tflops": rf["tflops"],
                     "frac_bf16_peak": rf["tflops"] / float(peaks["bf16_tflops"]),
                     "bound": rf["bound"], "frac": rf["frac"], "alg_bytes": rf["alg_bytes"],
                     "traffic": rf["traffic"], "plan_build_us": b_us, "plan_gpu_ms": b_ms,
                     "visible_pairs": info["visible_pairs"] * (w.Hq if info["mask_heads"] == 1 else 1),
                     "kernel": fwd_kernel_name(w), "plan_choices": choices, "backward": bwd}
        del dp, plan, w
        torch.cuda.empty_cache()
    out["decode_paged"] = time_decode(fa, runner, W, flush, stream, peaks, peak_src, reps, seed)
    torch.cuda.empty_cache()
    return out


DECODE_DESC = ("decode over a paged KV cache: B=32 sequences, k_len ~ U[2048, 32768], Hq=32 Hk=8 d=128, "
               "64-token pages, causal at the query's absolute position")


def time_decode(fa, runner, W, flush, stream, peaks, peak_src, reps: int, seed: int):
    """fa_decode_paged (page conversion + unit split, decode kernel, unit
    merge) timed alone, L2 flushed before each call.  Algorithmic bytes: the
    K and V rows of every visible key once per K/V head, Q read, O and LSE
    written; the bound is HBM."""
    import torch
    w = W.decode_paged(seed)
    dp = runner.decode_to_device(w)
    plan = runner.decode_plan(dp)
    info = fa.fa_plan_info_get(plan, count_visible=True)
    vis_keys = info["visible_pairs"]  # summed over the mask heads' rows
    kv_heads = w.Hk if info["mask_heads"] == 1 else 1
    alg = float(vis_keys * kv_heads * w.d * 2 * 2 + 2 * w.q.numel() * 2 + 4 * w.Hq * w.B)
    for _ in range(3):
        runner.decode(dp, plan)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for i in range(reps):
        flush.zero_()
        torch.cuda._sleep(SLEEP_CYCLES)
        ev[i][0].record(stream)
        runner.decode(dp, plan)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flops = 4.0 * w.d * vis_keys * w.Hq
    rf = roofline(flops, alg, ms, peaks, peak_src, known_traffic("decode_paged"))
    plan.free()
    return {"workload": DECODE_DESC, "decode_ms": ms, "bound": rf["bound"], "frac": rf["frac"],
            "alg_bytes": alg, "alg_gbs": rf["alg_gbs"], "tflops": rf["tflops"], "traffic": rf["traffic"],
            "visible_keys_per_kv_head": vis_keys, "launches": 3,
            "kernel": "k_decode<16> (persistent keys-major decode; prep and merge kernels beside it)"}


def cpu_baseline(w, budget_s: float):
    """Oracle (fp64, numpy) attention on a bounded sample of rows, visible TFLOPS."""
    import numpy as np
    from oracle import attention as OA
    from oracle import mask as OM

    rng = np.random.default_rng(0)
    bounds = w.sample_bounds()
    t0 = time.perf_counter()
    flops = 0.0
    rows_done = 0
    pairs = 0
    while time.perf_counter() - t0 < budget_s:
        b = int(rng.integers(0, len(bounds)))
        _, q_len, _, _ = bounds[b]
        if q_len == 0:
            continue
        h = int(rng.integers(0, w.Hq))
        start = int(rng.integers(0, max(1, q_len - 128)))
        rows = np.arange(start, min(q_len, start + 128))
        hm = 0 if w.Hmask == 1 else h
        vis = OM.visible_rows(w, hm, b, rows)
        OA.attention_rows(w, b, h, rows)
        flops += 4.0 * w.d * float(vis.sum())
        rows_done += rows.size
        pairs += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"{pairs} blocks of up to 128 consecutive Q rows of random (sample, head), "
                      f"{rows_done} rows, all visible keys, fp64 numpy, {dt:.1f} s"}


def workload_config(args) -> dict:
    """The `config` object of both arms: which workload, seed and step."""
    return {"workload": WORKLOAD_DESC[args.workload], "seed": args.seed,
            "step": "plan build + masked forward",
            "l2": "256 MB buffer written between timed steps"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    from block_sparse_masked_gb300 import workloads as W
    w = W.make(args.workload, args.seed)
    per_step = max(0.5, min(3.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, per_step / 4)
    vals = []
    t0 = time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(w, per_step)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    v = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args),
        "reference_timing": "fp64 oracle on bounded samples of the workload on the host cores; "
                            "no GPU, so the L2 flush of the config does not apply",
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    from block_sparse_masked_gb300 import build as fb

    if world > 1:
        if local == 0:
            fb.build()
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist.barrier()
    else:
        fb.build()
    torch.cuda.set_device(local)
    import block_sparse_masked_gb300 as fa
    from block_sparse_masked_gb300 import runner
    from block_sparse_masked_gb300 import workloads as W

    w = W.make(args.workload, args.seed + rank)
    dp = runner.to_device(w)
    stream = torch.cuda.current_stream()
    pkw = plan_kw(w)
    plan = runner.build_plan(dp, **pkw)
    info = fa.fa_plan_info_get(plan, count_visible=True)
    plan.free()
    flops_step = visible_flops(info, w.Hq, w.d)
    launches_per_step = 3 + 1  # planner (front, schedule, back) + forward
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        p = runner.build_plan(dp, **pkw)
        if ev is not None:
            ev[1].record(stream)
        runner.forward(dp, p)
        if ev is not None:
            ev[2].record(stream)
        bu = fa.fa_plan_info_get(p)["build_us"]
        p.free()
        return bu

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    build_us = []
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # L2 flush outside the per-step events
        torch.cuda.synchronize()  # each step starts from a drained queue
        build_us.append(step(evs[i]))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    plan_ms = [e[0].elapsed_time(e[1]) for e in evs]
    fwd_in_step_ms = [e[1].elapsed_time(e[2]) for e in evs]
    tot_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = tot_ms / args.steps
    value = whole_job_tflops(flops_step, world, ms_per_step)

    # The forward kernel alone, for the roofline (see time_forward_alone).
    plan_f = runner.build_plan(dp, **pkw)
    torch.cuda.synchronize()
    fwd_ms = time_forward_alone(runner, dp, plan_f, flush, stream, args.steps)
    plan_f.free()
    clk = clocks.stop()
    fwd_mean = statistics.mean(fwd_ms)
    fwd_tflops = flops_step / (fwd_mean * 1e-3) / 1e12

    # end to end through the public API with host buffers: H2D inputs, plan, forward, D2H output
    hq = [t.pin_memory() for t in (w.q, w.k, w.v)]
    hmask = torch.from_numpy(np.ascontiguousarray(
        w.mask_func if w.mask_kind == "intervals" else w.block_mask)).pin_memory()
    ho = torch.empty(dp.o.shape, dtype=dp.o.dtype).pin_memory()
    hl = torch.empty(dp.lse.shape, dtype=dp.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hq) + hmask.numel() * hmask.element_size()
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    # Two device copies of the inputs and outputs, used in turn: a step's
    # host->device copies (two side streams) run while the previous step's
    # plan and forward use the other copy, once the forward two steps back
    # has read this one; O and LSE leave on a third stream.
    dps = [dp, runner.to_device(w)]
    s_in = [torch.cuda.Stream(), torch.cuda.Stream()]
    s_out = torch.cuda.Stream()
    used = [torch.cuda.Event(), torch.cuda.Event()]  # the last forward on copy i has finished
    outd = [torch.cuda.Event(), torch.cuda.Event()]  # copy i's O/LSE have reached the host
    for ev in used + outd:
        ev.record(stream)
    n_e2e = [0]

    def e2e_step():
        i = n_e2e[0] % 2
        n_e2e[0] += 1
        b = dps[i]
        for j, (dst, src) in enumerate(zip((b.q, b.k, b.v, b.mask), (*hq, hmask))):
            s_in[j % 2].wait_event(used[i])
            with torch.cuda.stream(s_in[j % 2]):
                dst.copy_(src, non_blocking=True)
        for si in s_in:
            stream.wait_stream(si)
        stream.wait_event(outd[i])  # this copy's previous O/LSE have left the device
        p = runner.build_plan(b, **pkw)
        runner.forward(b, p)
        used[i].record(stream)
        s_out.wait_event(used[i])
        with torch.cuda.stream(s_out):
            ho.copy_(b.o, non_blocking=True)
            hl.copy_(b.lse, non_blocking=True)
        outd[i].record(s_out)
        p.free()

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ksteps = max(5, args.steps // 2)
    e0.record(stream)
    for _ in range(ksteps):
        e2e_step()
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ksteps, world)
    e2e_val = whole_job_tflops(flops_step, world, e2e_ms)
    assert fa.fa_device_error_flags() == 0, "device error flags set"

    peaks, peak_src = load_peaks()
    rf = roofline(flops_step, algorithmic_bytes(w, info), fwd_mean, peaks, peak_src,
                  known_traffic(args.workload))
    rf.update({"timing": "forward launch between two events queued behind a sleep kernel, "
                         "L2 flushed before each launch",
               "kernel": fwd_kernel_name(w)})
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args),
        "plan_build_us": statistics.median(build_us),
        "plan_gpu_ms": statistics.median(plan_ms),
        "plan_flags": "FA_PLAN_QUADRANT_PAYLOAD" if pkw else "none",
        "fwd_ms": fwd_mean,
        "fwd_ms_in_step": statistics.mean(fwd_in_step_ms),
        "fwd_tflops": fwd_tflops,
        "visible_pairs": info["visible_pairs"] * (w.Hq if info["mask_heads"] == 1 else 1),
        "roofline": rf,
        "e2e": {"value": e2e_val, "unit": "TFLOPS", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "note": "host->device input copies (pinned, ~0.2 TB/s on this machine) bound this number"},
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed": t_wall,
    }
    if not args.no_per_config:
        clocks2 = ClockSampler(local)
        clocks2.start()
        pc = per_config_table(fa, runner, W, flush, stream, peaks, peak_src, max(10, args.steps // 2),
                              args.seed + rank)
        line["per_config"] = pc
        line["per_config_clocks"] = clocks2.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
