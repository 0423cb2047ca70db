"""Offline profiling that fills the regime table (Tessera abstract:
profile-guided regime selection through a lookup table built by offline
profiling).

For every mask class -- logical block shape, density bucket, sequence-length
bucket, head dimension -- a few seeded synthetic masks of that class are planned
and run with every kernel variant (tile orientation: 128-row query tiles or
key-major 64-query tiles; for 128-row tiles the tile width, pipeline depth and
CTAs per SM); the fastest variant (median over the masks of plan + forward
time) becomes the row of that class.  Run on the target GPU:

    python -m block_sparse_attention_tsr_gb300.regimes_build [--out PATH] [--quick]

and commit the written table (``regimes_gb300.txt`` next to this file), which
the binding loads at start-up.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import block_sparse_attention_tsr_gb300 as tsr  # noqa: E402
import workloads as W  # noqa: E402

SHAPES = ((32, 32), (64, 64), (128, 128), (64, 256), (256, 64))
DENSITY_EDGES = (0.0, 0.15, 0.30, 0.45, 0.60, 1.01)
N_BUCKETS = ((0, 8191, 4096), (8192, 1 << 24, 32760))   # (n_min, n_max, N used to profile)
# (bn, stages, ctas per SM, orientation): 1 = 128-row query tiles, 2 = the
# key-major kernel (d = 128 only; its ring shape is fixed)
ROWS, KEYS = 1, 2
VARIANTS = {128: ((128, 3, 1, ROWS), (128, 2, 1, ROWS), (64, 4, 1, ROWS), (64, 2, 2, ROWS),
                  (64, 2, 1, KEYS)),
            64: ((128, 4, 1, ROWS), (64, 4, 1, ROWS), (64, 3, 2, ROWS))}
# key-list (M x 1 slice) masks: classes by slice height and listed-key fraction;
# the gathered kernel variants
KEYLIST_M = (64, 128)
KEYLIST_EDGES = (0.0, 0.10, 0.20, 0.35, 0.60, 1.01)
VARIANTS_GATHERED = {128: ((128, 3, 1, ROWS), (64, 2, 2, ROWS), (64, 2, 1, KEYS)),
                     64: ((128, 4, 1, ROWS), (64, 3, 2, ROWS))}


def keylist_spec(N, M, frac, heads, seed):
    """A key-list mask of one head's lists (clustered runs), repeated for every
    head: the generator is slow at high densities, and identical heads time the
    same as distinct ones of the same class."""
    one = W.keylist_mask(seed=seed, B=1, H=1, N=N, slice_m=M, frac=frac)
    indptr = np.concatenate([[0]] + [one.indptr[1:] + h * one.indptr[-1] for h in range(heads)])
    return W.MaskSpec(W.MASK_KEYLIST, 1, heads, N, slice_m=M, indptr=indptr.astype(np.int64),
                      indices=np.tile(one.indices, heads))


def time_variant(mask, q, k, v, out, lse, variant, reps):
    bn, stages, ctas, orient = variant
    plan = tsr.tsr_plan(mask, {"bn": bn, "stages": stages, "ctas_per_sm": ctas, "orient": orient})
    stream = torch.cuda.current_stream()
    for _ in range(2):
        plan.update(mask)
        tsr.tsr_bsa_forward(q, k, v, plan, out, lse)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        plan.update(mask)
        tsr.tsr_bsa_forward(q, k, v, plan, out, lse)
    b.record(stream)
    torch.cuda.synchronize()
    tsr.tsr_plan_device_status(plan)
    plan.destroy()
    return a.elapsed_time(b) / reps


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                  "regimes_gb300.txt"))
    ap.add_argument("--heads", type=int, default=8)
    ap.add_argument("--masks", type=int, default=2, help="seeded masks per class")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--quick", action="store_true", help="d = 128, long sequences only")
    args = ap.parse_args()
    tsr.build()
    tsr.lib()
    tsr.tsr_regime_load(None)
    rows = []
    t0 = time.time()
    dims = (128,) if args.quick else (128, 64)
    nbs = N_BUCKETS[1:] if args.quick else N_BUCKETS
    for d in dims:
        for n_min, n_max, N in nbs:
            q, k, v = (x.cuda() for x in W.qkv(1, args.heads, N, d, seed=5))
            out = torch.empty_like(q)
            lse = torch.empty((1, args.heads, N), device="cuda")
            for bq, bk in SHAPES:
                for lo, hi in zip(DENSITY_EDGES[:-1], DENSITY_EDGES[1:]):
                    times = {vv: [] for vv in VARIANTS[d]}
                    for m in range(args.masks):
                        r = np.random.Generator(np.random.PCG64(1000 * bq + bk + 7919 * m))
                        dens = np.clip(r.uniform(lo, min(hi, 1.0), size=(1, args.heads)), 0.01, 1.0)
                        blocks = W.banded_blocks(1, args.heads, W.cdiv(N, bq), W.cdiv(N, bk), dens, r)
                        spec = W.MaskSpec(W.MASK_UNIFORM, 1, args.heads, N, bq=bq, bk=bk, blocks=blocks)
                        mask = tsr.make_mask(spec.kind, 1, args.heads, N, d, **W.mask_tensors(spec))
                        for vv in VARIANTS[d]:
                            times[vv].append(time_variant(mask, q, k, v, out, lse, vv, args.reps))
                    med = {vv: float(np.median(t)) for vv, t in times.items()}
                    best = min(med, key=med.get)
                    rows.append((W.MASK_UNIFORM, bq, bk, n_min, n_max, lo, hi, d) + best)
                    print(f"d={d} N={N} {bq}x{bk} dens[{lo:.2f},{hi:.2f}) -> {best}  " +
                          " ".join(f"{vv}:{t:.3f}ms" for vv, t in med.items()), flush=True)
            # key-list masks (listed keys drawn in clustered runs, mean length 8)
            for M in KEYLIST_M:
                for lo, hi in zip(KEYLIST_EDGES[:-1], KEYLIST_EDGES[1:]):
                    times = {vv: [] for vv in VARIANTS_GATHERED[d]}
                    for m in range(args.masks):
                        spec = keylist_spec(N, M, 0.5 * (lo + min(hi, 1.0)), args.heads,
                                            seed=31 * M + 7 * m + int(100 * lo))
                        mask = tsr.make_mask(spec.kind, 1, args.heads, N, d, **W.mask_tensors(spec))
                        for vv in VARIANTS_GATHERED[d]:
                            times[vv].append(time_variant(mask, q, k, v, out, lse, vv, args.reps))
                    med = {vv: float(np.median(t)) for vv, t in times.items()}
                    best = min(med, key=med.get)
                    rows.append((W.MASK_KEYLIST, M, 1, n_min, n_max, lo, hi, d) + best)
                    print(f"d={d} N={N} keylist M={M} frac[{lo:.2f},{hi:.2f}) -> {best}  " +
                          " ".join(f"{vv}:{t:.3f}ms" for vv, t in med.items()), flush=True)
            # head-routed (SVG) masks: one row per length bucket
            F = 21 if N >= 8192 else 16         # >= 16 frames: at most 8 segments per tile
            S = N // F
            spec = W.svg_mask(1, args.heads, n_frames=F, frame_size=S)
            qs, ks, vs = (x.cuda() for x in W.qkv(1, args.heads, F * S, d, seed=6))
            outs = torch.empty_like(qs)
            lses = torch.empty((1, args.heads, F * S), device="cuda")
            mask = tsr.make_mask(spec.kind, 1, args.heads, F * S, d, **W.mask_tensors(spec))
            med = {vv: time_variant(mask, qs, ks, vs, outs, lses, vv, args.reps)
                   for vv in VARIANTS[d]}
            best = min(med, key=med.get)
            rows.append((W.MASK_SVG, "*", "*", n_min, n_max, "*", "*", d) + best)
            print(f"d={d} N={F * S} svg -> {best}  " +
                  " ".join(f"{vv}:{t:.3f}ms" for vv, t in med.items()), flush=True)
    # anything else: one default row per head dimension
    rows.append(("*", "*", "*", "*", "*", "*", "*", 128, 64, 2, 2, ROWS))
    rows.append(("*", "*", "*", "*", "*", "*", "*", 64, 64, 3, 2, ROWS))
    with open(args.out, "w") as f:
        f.write("# Regime table for GB300 (sm_103a), written by regimes_build.py\n")
        f.write(f"# {time.strftime('%Y-%m-%d')}: {args.masks} seeded masks per class (banded-plus-"
                f"random blocks; clustered key lists, one head's repeated; SVG routing), "
                f"{args.heads} heads, median of plan + forward time\n")
        f.write("# kind bq bk n_min n_max dens_min dens_max d bn stages ctas orient\n")
        for r in rows:
            f.write(" ".join(f"{x:.2f}" if isinstance(x, float) else str(x) for x in r) + "\n")
    print(f"wrote {len(rows)} rows to {args.out} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
