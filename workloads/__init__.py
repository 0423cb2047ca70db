"""Seeded synthetic inputs for block-sparse attention (shared by the oracle side
and the CUDA side; holds none of the attention arithmetic).

Everything here draws random numbers and lays them out; nothing here computes
attention, expands a mask to elements or plans tiles.  The shapes and mask
families stand in for the video-shaped workloads that the pages describe
(Tessera abstract: dynamic block-sparse masks on video diffusion transformers;
Sparse VideoGen digest: spatial / temporal head patterns; FG-Attn abstract:
M x 1 key slices with M = 64 and more than 30K tokens for a 5-second clip).
The pages' own masks and models are not available, so every input is synthetic.

Random sources:
  * Q, K, V: ``torch.Generator`` on the CPU, fp32 ``randn`` rounded to bf16
    (round to nearest even, which is what ``Tensor.to(torch.bfloat16)`` does).
  * masks: NumPy ``Generator(PCG64(seed))``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

MASK_UNIFORM = 0
MASK_SEGMENTS = 1
MASK_SVG = 2
MASK_KEYLIST = 3

HEAD_SPATIAL = 0
HEAD_TEMPORAL = 1


@dataclass
class MaskSpec:
    """A logical mask in one of the four forms the library accepts.

    UNIFORM : ``blocks`` uint8 [B, H, ceil(N/bq), ceil(N/bk)] over a grid of
              bq x bk logical blocks (the last row / column truncated at N).
    SEGMENTS: ``blocks`` uint8 [B, H, n_qseg, n_kseg] over variable segments
              given by ``q_bounds`` (n_qseg+1 ascending int32, 0 .. N) and
              ``k_bounds``.
    SVG     : ``head_kind`` int8 [H] (0 spatial, 1 temporal), ``n_frames`` F and
              ``frame_size`` S with N = F * S, tokens in frame-major order.
    KEYLIST : CSR over (b, h, query block of ``slice_m`` rows): ``indptr`` int64
              [B*H*ceil(N/M) + 1], ``indices`` int32 sorted, unique, < N.
    """
    kind: int
    B: int
    H: int
    N: int
    bq: int = 0
    bk: int = 0
    blocks: Optional[np.ndarray] = None
    q_bounds: Optional[np.ndarray] = None
    k_bounds: Optional[np.ndarray] = None
    head_kind: Optional[np.ndarray] = None
    n_frames: int = 0
    frame_size: int = 0
    slice_m: int = 0
    indptr: Optional[np.ndarray] = None
    indices: Optional[np.ndarray] = None
    temporal_radius: int = 0
    meta: dict = field(default_factory=dict)


def qkv(B: int, H: int, N: int, d: int, seed: int, scale: float = 1.0, device: str = "cpu"):
    """bf16 Q, K, V of shape [B, H, N, d] drawn from N(0, scale^2), seeded.
    ``device="cuda"`` draws them with the GPU's generator (same distribution,
    other values; for timing runs that never compare against the oracle)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    for _ in range(3):
        t = torch.randn((B, H, N, d), generator=g, dtype=torch.float32, device=device)
        if scale != 1.0:
            t = t * scale
        out.append(t.to(torch.bfloat16))
    return tuple(out)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


# --------------------------------------------------------------------------
# UNIFORM block masks
# --------------------------------------------------------------------------

def bernoulli_blocks(B: int, H: int, nqb: int, nkb: int, p: float, seed: int,
                     diag: bool = True, zero_rows: int = 0) -> np.ndarray:
    """i.i.d. Bernoulli(p) grid, diagonal forced on (when requested), then
    ``zero_rows`` whole query-block rows (chosen from the seed) zeroed, their
    diagonal included, to make fully masked query rows."""
    r = _rng(seed)
    blk = (r.random((B, H, nqb, nkb)) < p).astype(np.uint8)
    if diag:
        n = min(nqb, nkb)
        blk[:, :, np.arange(n), np.arange(n)] = 1
    for bh in range(B * H):
        b, h = divmod(bh, H)
        for z in r.choice(nqb, size=zero_rows, replace=False) if zero_rows else []:
            blk[b, h, z, :] = 0
    return blk


def banded_blocks(B: int, H: int, nqb: int, nkb: int, densities: np.ndarray,
                  r: np.random.Generator, width: float = 16.0,
                  boost: float = 4.0, diag: bool = True) -> np.ndarray:
    """Banded-plus-random grid: weight w_ij = 1 + boost * exp(-|i' - j'| / width)
    (i', j' on a common block scale so non-square blocks keep the band on the
    token diagonal), p_ij = min(1, c * w_ij) with c found by bisection so that
    mean(p) equals the head's density; Bernoulli draws; diagonal forced on."""
    densities = np.asarray(densities, dtype=np.float64).reshape(B, H)
    qi = (np.arange(nqb) + 0.5) / nqb
    kj = (np.arange(nkb) + 0.5) / nkb
    scale = max(nqb, nkb)
    w = 1.0 + boost * np.exp(-np.abs(qi[:, None] - kj[None, :]) * scale / width)
    out = np.zeros((B, H, nqb, nkb), dtype=np.uint8)
    # mean(min(1, c w)) from the sorted weights: the k weights below 1 / c
    # contribute c * (their sum), the rest 1 each
    ws = np.sort(w.ravel())
    cum = np.concatenate([[0.0], np.cumsum(ws)])
    n = ws.size

    def mean_p(c: float) -> float:
        k = int(np.searchsorted(ws, 1.0 / c, side="left"))
        return (c * cum[k] + (n - k)) / n

    for b in range(B):
        for h in range(H):
            rho = float(densities[b, h])
            lo, hi = 0.0, 1.0 / w.min()
            for _ in range(60):
                c = 0.5 * (lo + hi)
                if mean_p(c) < rho:
                    lo = c
                else:
                    hi = c
            p = np.minimum(1.0, 0.5 * (lo + hi) * w)
            out[b, h] = (r.random((nqb, nkb)) < p).astype(np.uint8)
    if diag:
        # force on every block that the token diagonal passes through
        for i in range(nqb):
            out[:, :, i, min(nkb - 1, (i * nkb) // nqb)] = 1
            out[:, :, i, min(nkb - 1, ((i + 1) * nkb - 1) // nqb)] = 1
    return out


def tiny_block_mask(seed: int = 1, B: int = 1, H: int = 2, N: int = 1024,
                    blk: int = 64, p: float = 0.3) -> MaskSpec:
    """Small case: 64 x 64 logical blocks, Bernoulli(0.3), diagonal forced on,
    then one fully masked query block per head."""
    nb = cdiv(N, blk)
    blocks = bernoulli_blocks(B, H, nb, nb, p, seed, diag=True, zero_rows=1)
    return MaskSpec(MASK_UNIFORM, B, H, N, bq=blk, bk=blk, blocks=blocks,
                    meta={"workload": f"tiny_block_mask_N{N}_H{H}_b{blk}_p{p}"})


def video_block_mask(seed: int = 2, B: int = 1, H: int = 24, N: int = 32760,
                     bq: int = 64, bk: int = 64, lo: float = 0.10,
                     hi: float = 0.40) -> MaskSpec:
    """480p-shaped layer (21 frames of 30 x 52 latents = 32,760 tokens): a
    banded-plus-random logical block mask per head, density ~ U(lo, hi)."""
    r = _rng(seed)
    dens = r.uniform(lo, hi, size=(B, H))
    blocks = banded_blocks(B, H, cdiv(N, bq), cdiv(N, bk), dens, r)
    return MaskSpec(MASK_UNIFORM, B, H, N, bq=bq, bk=bk, blocks=blocks,
                    meta={"workload": f"video_block_mask_N{N}_H{H}_{bq}x{bk}",
                          "densities": dens})


SWEEP_SHAPES = ((32, 32), (64, 64), (128, 128), (64, 256), (256, 64))


def sweep_mask(m: int, B: int = 1, H: int = 24, N: int = 32760) -> MaskSpec:
    """Member m of the seeded sweep: logical block shape uniform over five
    shapes, base density ~ U(0.05, 0.60), per-head jitter of +-20% relative,
    banded-plus-random generator at the logical grid."""
    r = _rng(10000 + m)
    bq, bk = SWEEP_SHAPES[int(r.integers(0, len(SWEEP_SHAPES)))]
    rho = r.uniform(0.05, 0.60)
    dens = np.clip(rho * r.uniform(0.8, 1.2, size=(B, H)), 0.01, 1.0)
    blocks = banded_blocks(B, H, cdiv(N, bq), cdiv(N, bk), dens, r)
    return MaskSpec(MASK_UNIFORM, B, H, N, bq=bq, bk=bk, blocks=blocks,
                    meta={"workload": f"sweep_{m}", "rho": rho, "bq": bq, "bk": bk,
                          "densities": dens})


# --------------------------------------------------------------------------
# SEGMENTS masks (variable logical block boundaries)
# --------------------------------------------------------------------------

def random_segments(N: int, lo: int, hi: int, r: np.random.Generator) -> np.ndarray:
    b = [0]
    while b[-1] < N:
        b.append(min(N, b[-1] + int(r.integers(lo, hi + 1))))
    return np.asarray(b, dtype=np.int32)


def segment_mask(seed: int, B: int, H: int, N: int, lo: int = 16, hi: int = 200,
                 p: float = 0.3) -> MaskSpec:
    r = _rng(seed)
    qb = random_segments(N, lo, hi, r)
    kb = random_segments(N, lo, hi, r)
    blocks = (r.random((B, H, len(qb) - 1, len(kb) - 1)) < p).astype(np.uint8)
    return MaskSpec(MASK_SEGMENTS, B, H, N, blocks=blocks, q_bounds=qb, k_bounds=kb,
                    meta={"workload": f"segments_N{N}"})


# --------------------------------------------------------------------------
# SVG head-routed masks
# --------------------------------------------------------------------------

def svg_mask(B: int = 1, H: int = 24, n_frames: int = 21, frame_size: int = 1560,
             kinds: Optional[np.ndarray] = None, temporal_radius: int = 0) -> MaskSpec:
    """Half the heads spatial, half temporal (first half spatial), unless
    ``kinds`` gives the routing explicitly.  ``temporal_radius`` r widens a
    temporal head to the spatial indices within r of the query's."""
    if kinds is None:
        kinds = np.array([HEAD_SPATIAL] * (H // 2) + [HEAD_TEMPORAL] * (H - H // 2),
                         dtype=np.int8)
    kinds = np.asarray(kinds, dtype=np.int8)
    assert kinds.shape == (H,)
    return MaskSpec(MASK_SVG, B, H, n_frames * frame_size, head_kind=kinds,
                    n_frames=n_frames, frame_size=frame_size, temporal_radius=temporal_radius,
                    meta={"workload": f"svg_F{n_frames}_S{frame_size}_H{H}_r{temporal_radius}"})


# --------------------------------------------------------------------------
# KEYLIST (M x 1 key-slice) masks
# --------------------------------------------------------------------------

def svg_routing_heads(B: int, kinds, n_frames: int, frame_size: int, d: int, seed: int,
                      contrast: float = 12.0, noise: float = 0.5):
    """bf16 Q, K, V [B, H, N, d] (H = len(kinds)) whose heads are built to be
    spatial (kinds[h] = 0: Q and K carry a code of the token's frame) or
    temporal (kinds[h] = 1: a code of the token's spatial index).  Codes are
    seeded random unit vectors scaled by ``contrast``, so tokens sharing the
    code score about contrast^2 / sqrt(d) above the rest; N(0, noise^2) is added
    to every dimension of Q and K; V ~ N(0, 1).  Inputs for routing tests only:
    which pattern a head follows is set here by design."""
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    kinds = np.asarray(kinds, dtype=np.int8)
    H, N = len(kinds), n_frames * frame_size
    t = torch.arange(N)
    codes = []
    for h in range(H):
        n_codes = n_frames if kinds[h] == 0 else frame_size
        e = torch.randn((n_codes, d), generator=g)
        e = contrast * e / e.norm(dim=1, keepdim=True)
        codes.append(e[t // frame_size] if kinds[h] == 0 else e[t % frame_size])
    code = torch.stack(codes)[None].expand(B, H, N, d)
    q = code + noise * torch.randn((B, H, N, d), generator=g)
    k = code + noise * torch.randn((B, H, N, d), generator=g)
    v = torch.randn((B, H, N, d), generator=g)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def clustered_keys(N: int, target: int, r: np.random.Generator,
                   mean_run: float = 8.0) -> np.ndarray:
    """Sorted unique key indices: runs with uniform starts and Geometric
    lengths (support >= 1, mean ``mean_run``) are added in draw order until at
    least ``target`` distinct keys are covered; the last run is trimmed so that
    exactly ``target`` keys remain."""
    target = min(target, N)
    n_runs = int(target / mean_run * 1.5) + 16
    while True:
        starts = r.integers(0, N, size=n_runs)
        lens = r.geometric(1.0 / mean_run, size=n_runs)
        ends = np.minimum(starts + lens, N)
        span = ends - starts
        total = int(span.sum())
        run_of = np.repeat(np.arange(n_runs), span)
        offs = np.arange(total) - np.repeat(np.cumsum(span) - span, span)
        pos = np.repeat(starts, span) + offs
        # first[j] = index of the earliest run (in draw order) covering key j
        first = np.full(N, n_runs, dtype=np.int64)
        np.minimum.at(first, pos, run_of)
        counts = np.bincount(first[first < n_runs], minlength=n_runs)
        cum = np.cumsum(counts)
        if cum[-1] < target:
            n_runs *= 2
            continue
        r_last = int(np.searchsorted(cum, target))
        before = int(cum[r_last - 1]) if r_last > 0 else 0
        keep = first < r_last
        # keys first covered by the crossing run, taken in the run's own order
        s, e = int(starts[r_last]), int(ends[r_last])
        seg = np.arange(s, e)
        seg = seg[first[s:e] == r_last][: target - before]
        keep[seg] = True
        out = np.nonzero(keep)[0].astype(np.int32)
        assert out.size == target
        return out


def keylist_mask(seed: int = 4, B: int = 1, H: int = 24, N: int = 75600,
                 slice_m: int = 64, frac: float = 0.15, mean_run: float = 8.0,
                 heads: Optional[range] = None) -> MaskSpec:
    """Per 64-query block a sorted key list covering ``frac`` of the keys."""
    r = _rng(seed)
    nqb = cdiv(N, slice_m)
    target = int(np.ceil(frac * N))
    lists = []
    for _ in range(B * H * nqb):
        lists.append(clustered_keys(N, target, r, mean_run))
    lengths = np.array([len(x) for x in lists], dtype=np.int64)
    indptr = np.zeros(B * H * nqb + 1, dtype=np.int64)
    np.cumsum(lengths, out=indptr[1:])
    indices = np.concatenate(lists).astype(np.int32) if lists else np.zeros(0, np.int32)
    return MaskSpec(MASK_KEYLIST, B, H, N, slice_m=slice_m, indptr=indptr,
                    indices=indices,
                    meta={"workload": f"keylist_N{N}_H{H}_f{frac}", "target": target})


def random_keylist(seed: int, B: int, H: int, N: int, slice_m: int = 64,
                   lo: int = 0, hi: Optional[int] = None) -> MaskSpec:
    """Small KEYLIST masks with list lengths ~ U[lo, hi] (empty lists allowed)."""
    r = _rng(seed)
    hi = N if hi is None else hi
    nqb = cdiv(N, slice_m)
    lists = []
    for _ in range(B * H * nqb):
        n = int(r.integers(lo, hi + 1))
        lists.append(np.sort(r.choice(N, size=min(n, N), replace=False)).astype(np.int32))
    lengths = np.array([len(x) for x in lists], dtype=np.int64)
    indptr = np.zeros(B * H * nqb + 1, dtype=np.int64)
    np.cumsum(lengths, out=indptr[1:])
    indices = np.concatenate(lists).astype(np.int32) if lists else np.zeros(0, np.int32)
    return MaskSpec(MASK_KEYLIST, B, H, N, slice_m=slice_m, indptr=indptr, indices=indices,
                    meta={"workload": f"random_keylist_N{N}"})


# --------------------------------------------------------------------------
# marshalling to device tensors (no arithmetic)
# --------------------------------------------------------------------------

def mask_tensors(spec: MaskSpec, device="cuda") -> dict:
    """The mask's arrays as contiguous torch tensors on `device`, keyed by the
    argument names of the library's mask description."""
    import torch

    def t(x, dt):
        return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).to(device)

    kw = dict(bq=spec.bq, bk=spec.bk, n_frames=spec.n_frames, frame_size=spec.frame_size,
              slice_m=spec.slice_m, temporal_radius=spec.temporal_radius)
    kw["blocks"] = t(spec.blocks, np.uint8)
    kw["q_bounds"] = t(spec.q_bounds, np.int32)
    kw["k_bounds"] = t(spec.k_bounds, np.int32)
    kw["head_kind"] = t(spec.head_kind, np.int8)
    kw["indptr"] = t(spec.indptr, np.int64)
    kw["indices"] = t(spec.indices, np.int32)
    return kw
