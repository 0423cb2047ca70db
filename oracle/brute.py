"""Dense brute-force masked attention for tiny inputs -- TEST INFRASTRUCTURE ONLY.

A second, independent statement of the same definition as ``oracle.c``: the
whole score matrix is formed at once, the mask is built as a dense boolean
matrix by array operations (Kronecker products, broadcasting, scatter), and
softmax uses an additive -inf mask.  It shares no code with ``oracle.c``, so an
index or mask-expansion mistake in either shows up as a disagreement.
Memory is O(N^2): use it for N up to a few hundred.
"""
from __future__ import annotations

import numpy as np

from . import UNIFORM, SEGMENTS, SVG, KEYLIST, as_u16


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense_mask(spec, b: int, h: int) -> np.ndarray:
    """Boolean [N, N] allowed matrix of head (b, h)."""
    N = spec.N
    if spec.kind == UNIFORM:
        grid = np.asarray(spec.blocks)[b, h].astype(bool)
        return np.kron(grid, np.ones((spec.bq, spec.bk), dtype=bool))[:N, :N].astype(bool)
    if spec.kind == SEGMENTS:
        grid = np.asarray(spec.blocks)[b, h].astype(bool)
        rq = np.diff(np.asarray(spec.q_bounds))
        rk = np.diff(np.asarray(spec.k_bounds))
        return np.repeat(np.repeat(grid, rq, axis=0), rk, axis=1)
    if spec.kind == SVG:
        t = np.arange(N)
        S = spec.frame_size
        if int(spec.head_kind[h]) == 0:
            f = t // S
            return (f[:, None] == f[None, :]) | (f[None, :] == 0)
        s = t % S
        return np.abs(s[:, None] - s[None, :]) <= int(getattr(spec, "temporal_radius", 0))
    if spec.kind == KEYLIST:
        M = spec.slice_m
        nqb = -(-N // M)
        out = np.zeros((N, N), dtype=bool)
        for qb in range(nqb):
            r = (b * spec.H + h) * nqb + qb
            keys = np.asarray(spec.indices)[spec.indptr[r]:spec.indptr[r + 1]]
            out[qb * M:min(N, (qb + 1) * M)][:, keys] = True
        return out
    raise ValueError("unknown mask kind")


def attention(spec, q, k, v):
    """(O [B,H,N,d], lse [B,H,N]) in fp64; empty rows give 0 and -inf."""
    Q, K, V = (bf16_to_f64(as_u16(x)) for x in (q, k, v))
    B, H, N, d = Q.shape
    O = np.zeros((B, H, N, d))
    L = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            allowed = dense_mask(spec, b, h)
            S = Q[b, h] @ K[b, h].T / np.sqrt(d)
            S = np.where(allowed, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            has = np.isfinite(mx[:, 0])
            mx = np.where(np.isfinite(mx), mx, 0.0)
            E = np.exp(S - mx)
            den = E.sum(axis=1, keepdims=True)
            P = np.divide(E, den, out=np.zeros_like(E), where=den > 0)
            O[b, h] = P @ V[b, h]
            L[b, h] = np.where(has, mx[:, 0] + np.log(np.where(has, den[:, 0], 1.0)), -np.inf)
    return O, L
