"""SVG head routing by sampled queries -- TEST INFRASTRUCTURE ONLY.

Same status as the rest of ``oracle/``: only ``tests/`` and ``bench.py``'s CPU
legs may use it.

Reading (the pages say only that Sparse VideoGen assigns each attention head
to a spatial or a temporal sparse pattern on the fly, Sparse VideoGen digest,
section "Sparse VideoGen"; they give no criterion): for a set of sampled query
rows, the head's attention output under each pattern is compared with dense
attention, and the head goes to the pattern with the smaller squared error.
For head (b, h) and samples i:

    stats[b, h, 0] = sum_i |O_spatial(i)  - O_dense(i)|^2
    stats[b, h, 1] = sum_i |O_temporal(i) - O_dense(i)|^2
    stats[b, h, 2] = sum_i |O_dense(i)|^2

(relative errors are stats[..., 0] / stats[..., 2] and stats[..., 1] /
stats[..., 2]), and head h is temporal iff sum_b stats[b, h, 1] <
sum_b stats[b, h, 0], spatial otherwise (ties go to spatial).

Each output is the oracle's fp64 masked attention of that row (``oracle.c``)
under the dense mask, the all-spatial SVG mask and the all-temporal SVG mask.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import SVG, UNIFORM, attention_rows


@dataclass
class _Spec:
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


def route(q, k, v, n_frames: int, frame_size: int, samples, temporal_radius: int = 0,
          nthreads: int = 0):
    """(stats fp64 [B, H, 3], head_kind int8 [H]) for bf16 q, k, v [B, H, N, d]
    and sampled query rows ``samples`` (int, shared by every head)."""
    B, H, N, _ = q.shape
    assert N == n_frames * frame_size
    samples = np.asarray(samples, dtype=np.int64)
    rows = (np.arange(B * H, dtype=np.int64)[:, None] * N + samples[None, :]).reshape(-1)
    dense = _Spec(UNIFORM, B, H, N, bq=N, bk=N, blocks=np.ones((B, H, 1, 1), np.uint8))
    spatial = _Spec(SVG, B, H, N, head_kind=np.zeros(H, np.int8), n_frames=n_frames,
                    frame_size=frame_size)
    temporal = _Spec(SVG, B, H, N, head_kind=np.ones(H, np.int8), n_frames=n_frames,
                     frame_size=frame_size, temporal_radius=temporal_radius)
    O, _, _ = attention_rows(dense, q, k, v, rows, nthreads)
    Os, _, _ = attention_rows(spatial, q, k, v, rows, nthreads)
    Ot, _, _ = attention_rows(temporal, q, k, v, rows, nthreads)
    n = len(samples)
    stats = np.stack([((Os - O) ** 2).sum(axis=1), ((Ot - O) ** 2).sum(axis=1),
                      (O ** 2).sum(axis=1)], axis=1).reshape(B, H, n, 3).sum(axis=2)
    tot = stats.sum(axis=0)
    head_kind = (tot[:, 1] < tot[:, 0]).astype(np.int8)
    return stats, head_kind
