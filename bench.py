"""Benchmark: block-sparse attention forward on the 480p-shaped video layer.

Workload (one step = the whole hot path on one synthetic request):
  21 frames x 30 x 52 latents = 32,760 tokens, B = 1, H = 24, d = 128, bf16
  Q/K/V ~ N(0, 1); per head a banded-plus-random 64 x 64 logical block mask with
  density ~ U(10%, 40%) (seed 2).  A step = tsr_plan (mask ingest, physical
  mapping, task organisation, regime lookup -- all GPU kernels) + tsr_bsa_forward.

Metric: effective TFLOP/s over unmasked work, 4 * d * |E| per call (|E| = allowed
(query, key) pairs), as a fraction of the measured dense bf16 peak, and ms/call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
reference arm of this project: a plain fp64 implementation of the definition)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "video480p_blockmask_64x64_N32760_H24_d128"
METRIC = "effective TFLOP/s (unmasked FLOPs) per BSA call"
UNIT = "TFLOP/s"
D = 128


def allowed_pairs_uniform(spec) -> int:
    """|E| of a UNIFORM block mask: sum over allowed blocks of rows x cols, with
    the last block row / column truncated at N."""
    N = spec.N
    rq = np.minimum(spec.bq, N - np.arange(spec.blocks.shape[2]) * spec.bq)
    rk = np.minimum(spec.bk, N - np.arange(spec.blocks.shape[3]) * spec.bk)
    return int(np.einsum("bhij,i,j->", spec.blocks.astype(np.int64), rq.astype(np.int64),
                         rk.astype(np.int64)))


def launches_per_step(spec, stats) -> int:
    """Kernels of this library launched per step (re-plan + forward).  SVG
    temporal heads of radius 0 take the launch-list compaction at plan time and
    the per-position kernel after the attention kernel; on the tiles they need
    no kernel of their own (the attention kernel applies the temporal-major
    permutation in its loads and stores).  A split plan adds the unit cut."""
    import workloads as W
    if spec.kind == W.MASK_KEYLIST:
        # count (validating), schedule, emit; a separate validation pass above
        # 196,608 tokens; + attention
        n = (4 if spec.N > 196608 else 3) + 1
    else:
        n = 3 + 1                          # count, schedule, emit + attention
        if spec.kind in (W.MASK_UNIFORM, W.MASK_SEGMENTS):
            n += 1                         # logical-block count (mask density)
        if stats.get("temporal_band"):
            n += 2                         # launch-list compaction + per-position kernel
    if stats.get("kv_split", 1) > 1:
        n += 1
    return n


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself with one rank): the
    whole job is as slow as its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_rank: float, ms_step: float, world: int) -> float:
    """Aggregate TFLOP/s of `world` ranks that each process flops_per_rank per
    step, the step taking ms_step (the maximum over ranks)."""
    return world * flops_per_rank / (ms_step * 1e-3) / 1e12


def sum_over_ranks(x: float, dist, device) -> float:
    """x summed over all ranks (x itself with one rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def head_range(H: int, world: int, rank: int):
    """Heads [lo, hi) of an H-head request that rank `rank` of `world` runs: the
    forward pass of every (b, h) is independent, so the request splits by head
    with no exchange between ranks; the split is balanced to within one head."""
    return (rank * H) // world, ((rank + 1) * H) // world


def slice_heads(spec, lo: int, hi: int):
    """The same mask restricted to heads [lo, hi) (every batch): block grids and
    head kinds are sliced, key lists keep their (b, h, query block) order with
    indptr rebased to the kept lists."""
    import copy
    import workloads as W
    out = copy.copy(spec)
    out.H = hi - lo
    out.meta = dict(spec.meta, heads=(lo, hi))
    if spec.blocks is not None:
        out.blocks = np.ascontiguousarray(spec.blocks[:, lo:hi])
    if spec.head_kind is not None:
        out.head_kind = np.ascontiguousarray(spec.head_kind[lo:hi])
    if spec.kind == W.MASK_KEYLIST:
        nqb = -(-spec.N // spec.slice_m)
        rows = np.concatenate([np.arange((b * spec.H + lo) * nqb, (b * spec.H + hi) * nqb)
                               for b in range(spec.B)]) if hi > lo else np.zeros(0, np.int64)
        lens = spec.indptr[rows + 1] - spec.indptr[rows]
        out.indptr = np.zeros(len(rows) + 1, dtype=np.int64)
        np.cumsum(lens, out=out.indptr[1:])
        out.indices = (np.concatenate([spec.indices[spec.indptr[r]:spec.indptr[r + 1]] for r in rows])
                       if len(rows) else np.zeros(0, np.int32)).astype(np.int32)
    return out


def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16": d.get("bf16_tflops"), "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d.get("hbm_gbs"), "src": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "src": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the attention kernels' sources (both tile orientations), with
    comments and blank lines removed: a profile stays attached to the code it
    measured when only a comment changes."""
    import re
    h = hashlib.sha256()
    for f in ("fwd_kernel.cuh", "fwd_t_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "block_sparse_attention_tsr_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        lines = [ln.rstrip() for ln in src.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def attention_kernel(stats) -> str:
    """The attention kernel a plan launches: key-major plans run the
    transposed-tile kernel."""
    return "bsa_fwd_t_kernel" if stats and stats.get("orient") == 2 else "bsa_fwd_kernel"


def read_traffic(kernel: str, kernel_hash: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary of the 480p workload, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_video480p.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_launch_full_size")


class ClockSampler:
    """nvidia-smi samples (its own 25 ms loop, each with its timestamp), started
    before the warm-up; summary() keeps the samples taken inside the timed
    region (a wall-clock window)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 25

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = f"/tmp/tsr_clocks_{os.getpid()}.csv"
        self.rows = []

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        t = _smi_time(parts[0])
                        self.rows.append((t, float(parts[2]), float(parts[3]),
                                          float(parts[4]), parts[6:10]))
                    except ValueError:
                        continue

    def summary(self, t0: float, t1: float):
        """Samples with wall time in [t0, t1] (the timed region)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [r for r in self.rows if t0 <= r[0] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples_total": len(self.rows)}
        load = [r for r in rows if r[3] > 200.0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in load for n, v in zip(names, r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in load), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "period_ms": self.PERIOD_MS, "power_w_max": max(r[3] for r in rows)}


def _smi_time(stamp: str) -> float:
    """nvidia-smi's timestamp field ("YYYY/MM/DD HH:MM:SS.mmm", local time) as
    seconds since the epoch, comparable with time.time()."""
    import datetime
    return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()



def cpu_baseline(spec, q, k, v, target_s: float = 12.0) -> dict:
    """The oracle (plain fp64 CPU definition), as it stands, on a bounded sample of
    whole output rows of the same workload, timed on all host cores."""
    import oracle
    rng = np.random.Generator(np.random.PCG64(99))
    nthreads = oracle.max_threads()

    def timed(nrows):
        rows = np.sort(rng.choice(spec.B * spec.H * spec.N, size=nrows, replace=False))
        t0 = time.perf_counter()
        _, _, cnt = oracle.attention_rows(spec, q, k, v, rows, nthreads)
        return time.perf_counter() - t0, int(cnt.sum())

    # calibrate on a sample large enough that thread start-up does not dominate
    n = 512
    t, _ = timed(n)
    while t < 0.5 and n < spec.B * spec.H * spec.N // 4:
        n *= 4
        t, _ = timed(n)
    n = int(min(spec.B * spec.H * spec.N, max(n, n * target_s / max(t, 1e-3))))
    t, pairs = timed(n)
    return {"value": 4.0 * D * pairs / t / 1e12, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{n} random whole query rows of the {WORKLOAD} workload "
                      f"({pairs} allowed pairs, {t:.1f} s)", "seconds": t}


WORKLOADS = {
    # name: (description, generator)
    "video480p": (WORKLOAD, lambda W, h: W.video_block_mask(seed=2, H=h)),
    "svg480p": ("svg480p_spatial_temporal_F21_S1560_H24_d128",
                lambda W, h: W.svg_mask(1, h, n_frames=21, frame_size=1560)),
    "keylist720p": ("fg720p_keylist_M64_15pct_N75600_H24_d128",
                    lambda W, h: W.keylist_mask(seed=4, H=h)),
}


def make_workload(heads: int = 24, name: str = "video480p"):
    import workloads as W
    if name.startswith("sweep"):
        spec = W.sweep_mask(int(name[5:] or 0), H=heads)
    else:
        spec = WORKLOADS[name][1](W, heads)
    seed = {"video480p": 2, "svg480p": 3, "keylist720p": 4}.get(name, 10)
    q, k, v = W.qkv(spec.B, spec.H, spec.N, D, seed=seed)
    return spec, q, k, v


def allowed_pairs(spec) -> int:
    """|E| for any mask form (counted from the logical mask, no attention)."""
    import workloads as W
    if spec.kind == W.MASK_UNIFORM:
        return allowed_pairs_uniform(spec)
    if spec.kind == W.MASK_SVG:
        S, F, N, r = spec.frame_size, spec.n_frames, spec.N, spec.temporal_radius
        temporal = F * F * (S * (2 * r + 1) - r * (r + 1)) if r < S else N * N
        per = [S * S * (2 * F - 1) if int(k) == W.HEAD_SPATIAL else temporal for k in spec.head_kind]
        return int(sum(per)) * spec.B
    if spec.kind == W.MASK_KEYLIST:
        M, N = spec.slice_m, spec.N
        lens = np.diff(spec.indptr).reshape(spec.B * spec.H, -1)
        rows = np.minimum(M, N - np.arange(lens.shape[1]) * M)
        return int((lens * rows[None, :]).sum())
    rq = np.diff(spec.q_bounds)
    rk = np.diff(spec.k_bounds)
    return int(np.einsum("bhij,i,j->", spec.blocks.astype(np.int64), rq, rk))


def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    spec, q, k, v = make_workload()
    target = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(spec, q, k, v, target_s=min(target, 3.0))
    vals, secs = [], []
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(spec, q, k, v, target_s=target)
        vals.append(last["value"])
        secs.append(last["seconds"])
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": last["sample"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sweep(args) -> None:
    """Mask sweep through the regime table: members 0 .. K-1 of the seeded sweep
    (block shape from five, density U(0.05, 0.60)); each mask is planned and run
    with the table's regime and with every compiled variant forced, and the
    table's regret against the best variant is reported.  One JSON line."""
    import torch
    import block_sparse_attention_tsr_gb300 as tsr
    import workloads as W
    from block_sparse_attention_tsr_gb300.regimes_build import VARIANTS

    tsr.build()
    tsr.lib()
    dev = torch.device("cuda", 0)
    N, H = 32760, args.heads
    q, k, v = (x.to(dev) for x in W.qkv(1, H, N, D, seed=10))
    out = torch.empty_like(q)
    lse = torch.empty((1, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(mask, opts, reps=3):
        plan = tsr.tsr_plan(mask, opts, stream)
        for _ in range(2):
            plan.update(mask, stream)
            tsr.tsr_bsa_forward(q, k, v, plan, out, lse, stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            plan.update(mask, stream)
            tsr.tsr_bsa_forward(q, k, v, plan, out, lse, stream)
        b.record(stream)
        torch.cuda.synchronize()
        tsr.tsr_plan_device_status(plan)
        st = plan.stats()
        plan.destroy()
        return a.elapsed_time(b) / reps, (st["bn"], st["stages"], st["ctas_per_sm"], st["orient"])

    rows = []
    t0 = time.time()
    for m in range(args.sweep_masks):
        spec = W.sweep_mask(m, H=H, N=N)
        mask = tsr.make_mask(spec.kind, 1, H, N, D, **W.mask_tensors(spec, dev))
        flops = 4.0 * D * allowed_pairs(spec)
        t_lut, picked = timed(mask, None)
        t_var = {vv: timed(mask, {"bn": vv[0], "stages": vv[1], "ctas_per_sm": vv[2],
                                  "orient": vv[3]})[0]
                 for vv in VARIANTS[D]}
        best = min(t_var, key=t_var.get)
        rows.append({"m": m, "shape": f"{spec.bq}x{spec.bk}", "rho": spec.meta["rho"],
                     "flops": flops, "ms_lut": t_lut, "ms_best": t_var[best], "lut": picked,
                     "best": best})
    regret = np.array([r["ms_lut"] / r["ms_best"] - 1.0 for r in rows])
    tot_flops = sum(r["flops"] for r in rows)
    tot_ms = sum(r["ms_lut"] for r in rows)
    shapes = {}
    for r in rows:
        shapes.setdefault(r["shape"], []).append(r["flops"] / r["ms_lut"] / 1e9)
    line = {"metric": METRIC, "value": tot_flops / tot_ms / 1e9, "unit": UNIT, "n_gpus": 1,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"sweep_{args.sweep_masks}_masks_N{N}_H{H}_d{D}",
                       "step": "tsr_plan_update + tsr_bsa_forward per mask, regime from the table",
                       "l2": "inputs exceed L2; no flush"},
            "lut_regret": {"mean": float(regret.mean()), "median": float(np.median(regret)),
                           "p90": float(np.quantile(regret, 0.9)), "max": float(regret.max()),
                           "picked_best_within_2pct": float(np.mean(regret <= 0.02))},
            "tflops_by_shape": {k: float(np.mean(v)) for k, v in sorted(shapes.items())},
            "key_major_picked": int(sum(1 for r in rows if r["lut"][3] == 2)),
            "key_major_best": int(sum(1 for r in rows if r["best"][3] == 2)),
            "seconds": time.time() - t0}
    if args.sweep_detail:
        line["masks"] = rows
    print(json.dumps(line, default=str), flush=True)


def run_batch(args) -> None:
    """Several requests of different shapes served together: the same requests
    run one launch each (tsr_bsa_forward, back to back on one stream) and in one
    batched launch (tsr_bsa_forward_batch).  Requests (d = 128, regime BN 64 /
    2 stages / 2 CTAs per SM for all): 480p block masks with 2, 4 and 6 heads,
    SVG 480p with 4 heads, a 8,192-token block mask with 8 heads and a
    2,048-token one with 16 heads.  One JSON line; planning is not timed."""
    import torch
    import block_sparse_attention_tsr_gb300 as tsr
    import workloads as W

    tsr.build()
    tsr.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    opts = {"bn": 64, "stages": 2, "ctas_per_sm": 2}
    specs = [W.video_block_mask(seed=21, H=2), W.video_block_mask(seed=22, H=4),
             W.video_block_mask(seed=23, H=6), W.svg_mask(1, 4, n_frames=21, frame_size=1560),
             W.video_block_mask(seed=24, H=8, N=8192), W.video_block_mask(seed=25, H=16, N=2048)]
    reqs, flops = [], 0.0
    for i, spec in enumerate(specs):
        q, k, v = (x.to(dev) for x in W.qkv(spec.B, spec.H, spec.N, D, seed=30 + i))
        mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, D, **W.mask_tensors(spec, dev))
        plan = tsr.tsr_plan(mask, opts, stream)
        out = torch.empty_like(q)
        lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32, device=dev)
        reqs.append((q, k, v, plan, out, lse))
        flops += 4.0 * D * allowed_pairs(spec)

    def one_by_one():
        for q, k, v, plan, out, lse in reqs:
            tsr.tsr_bsa_forward(q, k, v, plan, out, lse, stream)

    def batched():
        tsr.tsr_bsa_forward_batch(reqs, stream)

    res = {}
    for name, fn in (("separate_launches", one_by_one), ("one_batched_launch", batched)):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        res[name] = {"ms": ms, "tflops": flops / ms / 1e9}
    tsr.tsr_plan_device_status(reqs[0][3])
    line = {"metric": METRIC, "value": res["one_batched_launch"]["tflops"], "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["one_batched_launch"]["ms"], "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "batch_6_requests_mixed_shapes_d128",
                       "requests": [f"{s.meta.get('workload', s.kind)} H{s.H} N{s.N}" for s in specs],
                       "step": "attention of all requests (plans made once)"},
            "separate_launches": res["separate_launches"],
            "one_batched_launch": res["one_batched_launch"]}
    print(json.dumps(line), flush=True)


def time_steps(tsr, plan, mask, qd, kd, vd, out, lse, stream, steps: int, warmup: int,
               before_timed=None):
    """Warm-up, then `steps` steps (re-plan + forward) on `stream`, each forward
    bracketed by its own CUDA events.  Returns (total ms, per-step forward ms,
    wall-clock window of the timed region)."""
    import torch

    def step(ev_pair=None):
        # the mask is re-planned every step (dynamic masks); the plan's device
        # storage is reused
        plan.update(mask, stream)
        if ev_pair is not None:
            ev_pair[0].record(stream)
        tsr.tsr_bsa_forward(qd, kd, vd, plan, out, lse, stream)
        if ev_pair is not None:
            ev_pair[1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    tsr.tsr_plan_device_status(plan)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if before_timed is not None:
        before_timed()
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    tsr.tsr_plan_device_status(plan)
    return t_start.elapsed_time(t_end), [a.elapsed_time(b) for a, b in evs], (w0, w1)


def other_workloads(tsr, names, steps: int, warmup: int, dev, stream, peak: float) -> dict:
    """The other full-size video workloads of the same path, timed the same way
    (one request of 24 heads, re-plan + forward per step, Q/K/V drawn on the
    device): forward and step times, effective TFLOP/s, fraction of the dense
    bf16 peak and tile fill."""
    import torch
    import workloads as W
    res = {}
    for name in names:
        spec = WORKLOADS[name][1](W, 24)
        qd, kd, vd = W.qkv(spec.B, spec.H, spec.N, D, seed=7, device=str(dev))
        mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, D, **W.mask_tensors(spec, dev))
        out = torch.empty_like(qd)
        lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32, device=dev)
        plan = tsr.tsr_plan(mask, None, stream)
        total_ms, fwd, _ = time_steps(tsr, plan, mask, qd, kd, vd, out, lse, stream, steps, warmup)
        st = plan.stats()
        flops = 4.0 * D * allowed_pairs(spec)
        fwd_ms = sum(fwd) / len(fwd)
        res[name] = {"workload": WORKLOADS[name][0], "step_ms": total_ms / steps,
                     "forward_ms": fwd_ms, "plan_ms": total_ms / steps - fwd_ms,
                     "step_tflops": flops / (total_ms / steps) / 1e9,
                     "forward_tflops": flops / fwd_ms / 1e9,
                     "forward_frac_of_peak": flops / fwd_ms / 1e9 / peak,
                     "fill": fill_of(spec, st, plan), "tiles": st["n_entries"],
                     "regime": {k: st[k] for k in ("bm", "bn", "stages", "ctas_per_sm", "regime_id")},
                     **({"temporal_heads": "by spatial position (F x F blocks, own kernel); "
                                           "fill over the spatial heads' tiles"}
                        if st.get("temporal_band") else {})}
        plan.destroy()
        del qd, kd, vd, out, lse, mask
        torch.cuda.empty_cache()
    return res


def fill_of(spec, stats, plan=None) -> float:
    """Allowed pairs over the elements of the computed physical tiles.  When
    the SVG temporal heads run by spatial position (no tiles), over the spatial
    heads' tiles only, counted from the plan's export (items of layout 0)."""
    if stats.get("temporal_band") and plan is not None:
        import workloads as W
        buf = plan.export()
        n_items = int(np.frombuffer(buf, np.int64, 1, 48)[0])
        items = np.frombuffer(buf, np.int32, 8 * n_items, 80).reshape(n_items, 8)
        spatial = items[:, 4] == 0
        tiles = int((items[spatial, 3] - items[spatial, 2]).sum())
        S, F = spec.frame_size, spec.n_frames
        n_sp = int(sum(int(k) == W.HEAD_SPATIAL for k in spec.head_kind)) * spec.B
        computed = tiles * stats["bm"] * stats["bn"]
        return S * S * (2 * F - 1) * n_sp / computed if computed else None
    computed = stats["n_entries"] * stats["bm"] * stats["bn"]
    return allowed_pairs(spec) / computed if computed else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tsr", choices=["tsr", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the SVG 480p and 720p key-list workloads after the headline")
    ap.add_argument("--replicas", action="store_true",
                    help="with several ranks: every rank runs the whole request (weak scaling) "
                         "instead of its share of the heads")
    ap.add_argument("--bn", type=int, default=0, help="force the K/V tile width (0 = table)")
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--ctas", type=int, default=0)
    ap.add_argument("--orient", type=int, default=0,
                    help="force the tile orientation: 1 = 128 query rows, 2 = 64-query "
                         "transposed tiles (0 = table)")
    ap.add_argument("--workload", default="video480p",
                    help="video480p (the benchmark), svg480p, keylist720p, sweepM (one member), "
                         "sweep (regime-table regret over --sweep-masks members), "
                         "batch (six requests: separate launches vs one batched launch)")
    ap.add_argument("--heads", type=int, default=24,
                    help="heads of the workload (24 = the benchmark; fewer for profiling)")
    ap.add_argument("--sweep-masks", type=int, default=32,
                    help="with --workload sweep: how many sweep members (256 = all)")
    ap.add_argument("--sweep-detail", action="store_true", help="per-mask rows in the sweep line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload == "sweep":
        if rank == 0:
            run_sweep(args)
        return
    if args.workload == "batch":
        if rank == 0:
            run_batch(args)
        return

    import torch
    import block_sparse_attention_tsr_gb300 as tsr
    import workloads as W

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    tsr.build()
    tsr.lib()

    full_spec, q, k, v = make_workload(args.heads, args.workload)
    # several ranks: each runs its share of the request's heads (no exchange),
    # unless --replicas gives every rank the whole request
    lo, hi = (0, full_spec.H) if (world == 1 or args.replicas) else head_range(full_spec.H, world, rank)
    spec = slice_heads(full_spec, lo, hi) if (lo, hi) != (0, full_spec.H) else full_spec
    q, k, v = (x[:, lo:hi].contiguous() for x in (q, k, v))
    pairs = allowed_pairs(spec) if hi > lo else 0
    flops = 4.0 * D * pairs
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks = read_peaks()

    opts = None
    if args.bn or args.stages or args.ctas or args.orient:
        opts = {"bn": args.bn, "stages": args.stages, "ctas_per_sm": args.ctas, "orient": args.orient}

    clk = ClockSampler(local)
    stats, fwd_avg, total_ms, window = None, 0.0, 0.0, (0.0, 0.0)
    with clk:
        if hi > lo:
            qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
            mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, D, **W.mask_tensors(spec, dev))
            out = torch.empty_like(qd)
            lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32, device=dev)
            plan = tsr.tsr_plan(mask, opts, stream)
            barrier = (lambda: dist.barrier()) if dist is not None else None
            total_ms, fwd_ms, window = time_steps(tsr, plan, mask, qd, kd, vd, out, lse, stream,
                                                  args.steps, args.warmup, barrier)
            stats = plan.stats()
            fwd_avg = sum(fwd_ms) / len(fwd_ms)
        elif dist is not None:
            dist.barrier()
        if dist is not None:
            dist.barrier()
    total_ms = max_over_ranks(total_ms, dist, dev)
    job_flops = sum_over_ranks(flops, dist, dev)
    ms_step = total_ms / args.steps
    value = job_flops / (ms_step * 1e-3) / 1e12
    long_region = total_ms > 2000.0
    peak = peaks["bf16_sustained"] if long_region else peaks["bf16"]
    achieved = flops / (fwd_avg * 1e-3) / 1e12 if fwd_avg > 0 else 0.0
    khash = kernel_source_hash()
    kname = attention_kernel(stats)
    traffic = read_traffic(kname, khash) if args.workload == "video480p" and args.heads == 24 else None

    e2e = None
    if not args.no_e2e and hi > lo:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
        marr = {k2: v2 for k2, v2 in dict(bq=spec.bq, bk=spec.bk, blocks=spec.blocks,
                                            q_bounds=spec.q_bounds, k_bounds=spec.k_bounds,
                                            head_kind=spec.head_kind, n_frames=spec.n_frames,
                                            frame_size=spec.frame_size, slice_m=spec.slice_m,
                                            indptr=spec.indptr, indices=spec.indices).items()
                if v2 is not None}
        mask_bytes = sum(np.asarray(v2).nbytes for v2 in marr.values() if isinstance(v2, np.ndarray))
        # the mask arrays are inputs of the step too: pinned like Q, K, V
        marr = {k2: (torch.from_numpy(np.ascontiguousarray(v2)).pin_memory()
                     if isinstance(v2, np.ndarray) else v2) for k2, v2 in marr.items()}

        def host_call():
            tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, D, qh, kh, vh, oh, lh,
                                   opts=opts, **marr)

        for _ in range(2):
            host_call()
        n_e2e = max(3, args.steps // 4)
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_call()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, dist, dev)
        e2e = {"value": job_flops / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(sum_over_ranks(3 * qh.numel() * 2 + mask_bytes, dist, dev)),
               "d2h_bytes_per_step": int(sum_over_ranks(oh.numel() * 2 + lh.numel() * 4, dist, dev)),
               "ms_per_step": 1e3 * e2e_s}

    route = None
    if spec.kind == W.MASK_SVG and hi > lo:
        # the step before the path: routing the heads from 64 sampled query rows
        smp = np.sort(np.random.Generator(np.random.PCG64(64)).choice(spec.N, size=64,
                                                                      replace=False))
        for _ in range(2):
            tsr.tsr_svg_route(qd, kd, vd, spec.n_frames, spec.frame_size, smp, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            tsr.tsr_svg_route(qd, kd, vd, spec.n_frames, spec.frame_size, smp, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        route = {"samples": 64, "ms": a.elapsed_time(b) / 5, "timed": "separately, not in the step"}

    others = None
    if (rank == 0 and world == 1 and args.workload == "video480p" and args.heads == 24
            and not args.no_other_workloads):
        del qd, kd, vd, out, lse
        torch.cuda.empty_cache()
        others = other_workloads(tsr, ("svg480p", "keylist720p"), min(args.steps, 30),
                                 args.warmup, dev, stream, peaks["bf16"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(spec, q, k, v)
        cpu.pop("seconds", None)

    wname = WORKLOADS[args.workload][0] if args.workload in WORKLOADS else args.workload
    split = world > 1 and not args.replicas
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wname if args.heads == 24 else f"{wname}_heads{args.heads}",
                       "B": full_spec.B, "H": full_spec.H, "N": full_spec.N, "d": D,
                       "parallelism": (f"heads split over {world} ranks, no collective" if split
                                       else ("replicas" if world > 1 else "single GPU")),
                       "rank0_heads": [lo, hi],
                       "mask_kind": int(spec.kind), "logical_block": [spec.bq, spec.bk],
                       "allowed_pairs": pairs,
                       "density": pairs / max(1, spec.B * spec.H * spec.N * spec.N),
                       "step": "tsr_plan_update (re-plan of the mask) + tsr_bsa_forward",
                       "l2": (f"inputs ({3 * spec.B * (hi - lo) * spec.N * D * 2 / 1e6:.0f} MB Q/K/V) "
                              + ("exceed the 129 MB L2; no flush"
                                 if 3 * spec.B * (hi - lo) * spec.N * D * 2 > 129e6
                                 else "fit the 129 MB L2; not flushed (parity-size run)")),
                       "regime": ({k2: stats[k2] for k2 in ("bm", "bn", "stages", "ctas_per_sm",
                                                             "regime_id")} if stats else None),
                       "tiles": stats["n_entries"] if stats else 0,
                       "boundary_tiles": stats["n_boundary"] if stats else 0,
                       "fill": fill_of(spec, stats, plan) if stats else None,
                       **({"temporal_heads": "by spatial position (F x F blocks, own kernel); "
                                             "fill over the spatial heads' tiles"}
                          if stats and stats.get("temporal_band") else {}),
                       "forward_ms": fwd_avg, "plan_ms": ms_step - fwd_avg,
                       **({"svg_route": route} if route else {}),
                       **({"other_workloads": others} if others else {}),
                       "forward_tflops": achieved,
                       "forward_frac_of_peak": achieved / peak},
            "pct_of_peak": 100.0 * value / (world * peak),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peaks['src']} bf16 "
                                        f"{'sustained' if long_region else 'burst'}",
                         "kernel": kname, "kernel_source_hash": khash},
            "clocks": clk.summary(*window),
            "gpu_launches": args.steps * launches_per_step(spec, stats or {}),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
