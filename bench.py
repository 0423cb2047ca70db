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
    """Kernels of this library launched per step (re-plan + forward).  Temporal
    SVG heads need no kernel of their own: the attention kernel applies the
    temporal-major permutation in its loads and stores."""
    import workloads as W
    if spec.kind == W.MASK_KEYLIST:
        # count (validating), schedule, emit; a separate validation pass above
        # 196,608 tokens; + attention
        return (4 if spec.N > 196608 else 3) + 1
    n = 3 + 1                              # count, schedule, emit + attention
    if spec.kind in (W.MASK_UNIFORM, W.MASK_SEGMENTS):
        n += 1                             # logical-block count (mask density)
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


def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16": d.get("bf16_tflops"), "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d.get("hbm_gbs"), "src": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "src": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("fwd_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "block_sparse_attention_tsr_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(kernel_hash: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "bsa_fwd_kernel_video480p.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_launch_full_size")


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = f"/tmp/tsr_clocks_{os.getpid()}.csv"

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.05)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r[2] > 200.0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in load for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r[2] for r in rows)}


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
        return a.elapsed_time(b) / reps, (st["bn"], st["stages"], st["ctas_per_sm"])

    rows = []
    t0 = time.time()
    for m in range(args.sweep_masks):
        spec = W.sweep_mask(m, H=H, N=N)
        mask = tsr.make_mask(spec.kind, 1, H, N, D, **W.mask_tensors(spec, dev))
        flops = 4.0 * D * allowed_pairs(spec)
        t_lut, picked = timed(mask, None)
        t_var = {vv: timed(mask, {"bn": vv[0], "stages": vv[1], "ctas_per_sm": vv[2]})[0]
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tsr", choices=["tsr", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--bn", type=int, default=0, help="force the K/V tile width (0 = table)")
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--ctas", type=int, default=0)
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

    spec, q, k, v = make_workload(args.heads, args.workload)
    pairs = allowed_pairs(spec)
    flops = 4.0 * D * pairs
    dev = torch.device("cuda", local)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    mt = W.mask_tensors(spec, dev)
    mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, D, **mt)
    out = torch.empty_like(qd)
    lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    opts = None
    if args.bn or args.stages or args.ctas:
        opts = {"bn": args.bn, "stages": args.stages, "ctas_per_sm": args.ctas}

    plan = tsr.tsr_plan(mask, opts, stream)

    def step(ev_pair=None):
        # the mask is re-planned every step (dynamic masks); the plan's device
        # storage is reused
        plan.update(mask, stream)
        if ev_pair is not None:
            ev_pair[0].record(stream)
        tsr.tsr_bsa_forward(qd, kd, vd, plan, out, lse, stream)
        if ev_pair is not None:
            ev_pair[1].record(stream)
        return plan

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    tsr.tsr_plan_device_status(plan)
    stats = plan.stats()
    computed = stats["n_entries"] * 128 * stats["bn"]

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(total_ms, dist, dev)
    tsr.tsr_plan_device_status(plan)
    ms_step = total_ms / args.steps
    value = whole_job_rate(flops, ms_step, world)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    peaks = read_peaks()
    achieved = flops / (fwd_avg * 1e-3) / 1e12
    long_region = total_ms > 2000.0
    peak = peaks["bf16_sustained"] if long_region else peaks["bf16"]
    khash = kernel_source_hash()
    traffic = read_traffic(khash)

    e2e = None
    if not args.no_e2e:
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
            tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, D, qh, kh, vh, oh, lh, **marr)

        for _ in range(2):
            host_call()
        n_e2e = max(3, args.steps // 4)
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_call()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, dist, dev)
        e2e = {"value": whole_job_rate(flops, 1e3 * e2e_s, world), "unit": UNIT,
               "h2d_bytes_per_step": 3 * qh.numel() * 2 + mask_bytes,
               "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4,
               "ms_per_step": 1e3 * e2e_s}

    route = None
    if spec.kind == W.MASK_SVG:
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

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(spec, q, k, v)
        cpu.pop("seconds", None)

    wname = WORKLOADS[args.workload][0] if args.workload in WORKLOADS else args.workload
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wname if args.heads == 24 else f"{wname}_heads{args.heads}",
                       "B": spec.B, "H": spec.H, "N": spec.N, "d": D,
                       "mask_kind": int(spec.kind), "logical_block": [spec.bq, spec.bk],
                       "allowed_pairs": pairs,
                       "density": pairs / (spec.B * spec.H * spec.N * spec.N),
                       "step": "tsr_plan_update (re-plan of the mask) + tsr_bsa_forward",
                       "l2": "inputs (603 MB Q/K/V) exceed the 129 MB L2; no flush",
                       "regime": {k2: stats[k2] for k2 in ("bn", "stages", "ctas_per_sm", "regime_id")},
                       "tiles": stats["n_entries"], "boundary_tiles": stats["n_boundary"],
                       "fill": pairs / computed if computed else None,
                       "forward_ms": fwd_avg, "plan_ms": ms_step - fwd_avg,
                       **({"svg_route": route} if route else {}),
                       "forward_tflops": achieved,
                       "forward_frac_of_peak": achieved / peak},
            "pct_of_peak": 100.0 * value / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peaks['src']} bf16 "
                                        f"{'sustained' if long_region else 'burst'}",
                         "kernel": "bsa_fwd_kernel", "kernel_source_hash": khash},
            "clocks": clk.summary(),
            "gpu_launches": args.steps * launches_per_step(spec, stats),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
