"""CPU oracle for masked attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The library
(``block_sparse_attention_tsr_gb300``) never imports it, and this package
imports nothing from the library: the two share only the seeded generators in
``workloads``.

Contents:
  * ``oracle.c``   fp64 masked attention by the definition (see its header for
                   the passages it follows and the readings it takes);
  * ``brute.py``   an independent dense NumPy brute force for tiny inputs;
  * ``coverage.c`` expansion of an exported tile plan into element sets, to be
                   compared bit-exactly with the oracle's allowed set;
  * ``oracle_mask.h`` the mask description both C files share;
  * ``route.py``   SVG head routing by sampled queries (error of each pattern
                   against dense attention), built on ``oracle.c``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, dense library attention for the all-ones mask, per-block dense
attention for block-diagonal masks, Q = 0 / one-key / constant-V closed forms,
counted densities, permutation invariance); ``coverage.c`` by
``tests/test_coverage_pins.py`` (hand-built plan exports of every descriptor
form, each planted plan mistake reported with its code); ``route.py`` by
``tests/test_oracle_route.py`` (K = 0 means, brute force, dense radius,
structured heads).  ``tests/test_oracle_mutants.py`` plants one mistake at a
time in copies of ``oracle.c`` and ``coverage.c`` and checks that a named pin
fails on each.  The pages print no values for any
input, so nothing is pinned to a worked example of the pages themselves.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = None
_LOCK = threading.Lock()

UNIFORM, SEGMENTS, SVG, KEYLIST = 0, 1, 2, 3


class _Mask(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32),
        ("bq", ctypes.c_int32), ("bk", ctypes.c_int32),
        ("n_qseg", ctypes.c_int32), ("n_kseg", ctypes.c_int32),
        ("q_bounds", ctypes.c_void_p), ("k_bounds", ctypes.c_void_p),
        ("blocks", ctypes.c_void_p),
        ("n_frames", ctypes.c_int32), ("frame_size", ctypes.c_int32),
        ("head_kind", ctypes.c_void_p),
        ("slice_m", ctypes.c_int32),
        ("indptr", ctypes.c_void_p), ("indices", ctypes.c_void_p),
        ("temporal_radius", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "liboracle.so")
    srcs = [os.path.join(_HERE, f) for f in ("oracle.c", "coverage.c")]
    deps = srcs + [os.path.join(_HERE, "oracle_mask.h")]
    if not force and os.path.exists(out) and all(
            os.path.getmtime(out) >= os.path.getmtime(s) for s in deps):
        return out
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", out + ".tmp"] + srcs
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True)          # no OpenMP: one thread
    os.replace(out + ".tmp", out)
    return out


def _bind(L):
    """Declare the C functions' signatures on a loaded build of the oracle."""
    P = ctypes.c_void_p
    L.oracle_attention_rows.argtypes = [P, P, P, P, P, ctypes.c_int64, P, P, P, ctypes.c_int]
    L.oracle_attention_rows.restype = ctypes.c_int
    L.oracle_attention.argtypes = [P, P, P, P, P, P, ctypes.c_int]
    L.oracle_attention.restype = ctypes.c_int
    L.oracle_probs_row.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, P, P, P, P]
    L.oracle_probs_row.restype = ctypes.c_int64
    L.oracle_row_keys.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P]
    L.oracle_row_keys.restype = ctypes.c_int64
    L.oracle_count_allowed.argtypes = [P, P, ctypes.c_int]
    L.oracle_count_allowed.restype = ctypes.c_int64
    L.oracle_max_threads.restype = ctypes.c_int
    L.coverage_check.argtypes = [P, P, ctypes.c_size_t, P, ctypes.c_int64, P, ctypes.c_int]
    L.coverage_check.restype = ctypes.c_int64
    return L


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = _bind(ctypes.CDLL(build()))
    return _LIB


@contextlib.contextmanager
def swapped_library(path: str):
    """For the planted-mistake tests only: every function of this package runs
    on another build of the C sources (a copy with one deliberate mistake) until
    the block exits; the normal build is then restored."""
    global _LIB
    normal = lib()
    with _LOCK:
        _LIB = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _LOCK:
            _LIB = normal


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _ptr(a) -> int:
    return a.ctypes.data if a is not None else 0


class _Bound:
    """A ctypes mask struct plus the arrays it points into (kept alive)."""

    def __init__(self, spec, d: int):
        self.keep = []

        def arr(x, dt):
            if x is None:
                return None
            a = np.ascontiguousarray(np.asarray(x, dtype=dt))
            self.keep.append(a)
            return a

        m = _Mask()
        m.kind, m.B, m.H, m.N, m.d = spec.kind, spec.B, spec.H, spec.N, d
        m.bq, m.bk = spec.bq, spec.bk
        blocks = arr(spec.blocks, np.uint8)
        m.blocks = _ptr(blocks)
        qb, kb = arr(spec.q_bounds, np.int32), arr(spec.k_bounds, np.int32)
        m.q_bounds, m.k_bounds = _ptr(qb), _ptr(kb)
        m.n_qseg = len(qb) - 1 if qb is not None else 0
        m.n_kseg = len(kb) - 1 if kb is not None else 0
        hk = arr(spec.head_kind, np.int8)
        m.head_kind = _ptr(hk)
        m.n_frames, m.frame_size = spec.n_frames, spec.frame_size
        m.slice_m = spec.slice_m
        ip = arr(spec.indptr, np.int64)
        ix = arr(spec.indices if spec.indices is None or len(spec.indices) else np.zeros(1),
                 np.int32)
        m.indptr, m.indices = _ptr(ip), _ptr(ix)
        m.temporal_radius = int(getattr(spec, "temporal_radius", 0))
        self.m = m

    @property
    def ref(self):
        return ctypes.byref(self.m)


def as_u16(t) -> np.ndarray:
    """bf16 torch tensor (any device) or uint16 array -> contiguous uint16 numpy."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def attention(spec, q, k, v, nthreads: int = 0):
    """Full fp64 output: (O [B,H,N,d], lse [B,H,N])."""
    qa, ka, va = as_u16(q), as_u16(k), as_u16(v)
    B, H, N, d = qa.shape
    bm = _Bound(spec, d)
    out = np.zeros((B, H, N, d), dtype=np.float64)
    lse = np.zeros((B, H, N), dtype=np.float64)
    rc = lib().oracle_attention(bm.ref, _ptr(qa), _ptr(ka), _ptr(va), _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle: invalid mask or inputs")
    return out, lse


def attention_rows(spec, q, k, v, rows, nthreads: int = 0):
    """Selected rows, rows[r] = (b*H + h)*N + i: (O [n,d], lse [n], counts [n])."""
    qa, ka, va = as_u16(q), as_u16(k), as_u16(v)
    d = qa.shape[-1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    bm = _Bound(spec, d)
    out = np.zeros((len(rows), d), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    cnt = np.zeros(len(rows), dtype=np.int64)
    rc = lib().oracle_attention_rows(bm.ref, _ptr(qa), _ptr(ka), _ptr(va), _ptr(rows), len(rows),
                                     _ptr(out), _ptr(lse), _ptr(cnt), nthreads)
    if rc != 0:
        raise ValueError("oracle: invalid mask, inputs or row ids")
    return out, lse, cnt


def probs_row(spec, q, k, v, b: int, h: int, i: int):
    """(keys, probabilities, O row, lse) of one row, keys ascending."""
    qa, ka, va = as_u16(q), as_u16(k), as_u16(v)
    d = qa.shape[-1]
    bm = _Bound(spec, d)
    keys = np.zeros(max(spec.N, 1), dtype=np.int32)
    probs = np.zeros(max(spec.N, 1), dtype=np.float64)
    out = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    n = lib().oracle_probs_row(bm.ref, _ptr(qa), _ptr(ka), _ptr(va), b, h, i,
                               _ptr(keys), _ptr(probs), _ptr(out), _ptr(lse))
    if n < 0:
        raise ValueError("oracle: invalid mask")
    return keys[:n].copy(), probs[:n].copy(), out, float(lse[0])


def row_keys(spec, b: int, h: int, i: int) -> np.ndarray:
    bm = _Bound(spec, 1)
    keys = np.zeros(max(spec.N, 1), dtype=np.int32)
    n = lib().oracle_row_keys(bm.ref, b, h, i, _ptr(keys))
    if n < 0:
        raise ValueError("oracle: invalid mask")
    return keys[:n].copy()


def count_allowed(spec, nthreads: int = 0) -> np.ndarray:
    """|E| per (b, h) as int64 [B*H]."""
    bm = _Bound(spec, 1)
    per = np.zeros(spec.B * spec.H, dtype=np.int64)
    n = lib().oracle_count_allowed(bm.ref, _ptr(per), nthreads)
    if n < 0:
        raise ValueError("oracle: invalid mask")
    return per


def coverage(spec, plan_bytes: bytes, nthreads: int = 0, max_report: int = 16):
    """Check an exported tile plan against the oracle's allowed set.

    Returns (n_errors, report, stats): report lists up to ``max_report`` failures
    as (code, b, h, i, j) tuples (codes in ``coverage.c``); stats is a dict with
    tile counts and element counts (computed / covered / allowed).
    """
    bm = _Bound(spec, 1)
    buf = np.frombuffer(plan_bytes, dtype=np.uint8)
    rep = np.zeros((max_report, 5), dtype=np.int64)
    st = np.zeros(8, dtype=np.int64)
    n = lib().coverage_check(bm.ref, _ptr(buf), len(buf), _ptr(rep), max_report, _ptr(st),
                             nthreads)
    if n < 0:
        raise ValueError(f"coverage: malformed plan export (code {n})")
    stats = dict(zip(("tiles", "full", "boundary", "computed", "covered", "allowed", "items"),
                     (int(x) for x in st[:7])))
    return int(n), [tuple(int(x) for x in r) for r in rep[: min(n, max_report)]], stats
