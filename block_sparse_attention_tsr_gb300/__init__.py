"""GB300 block-sparse attention forward -- Python binding of ``libtsr_gb300.so``.

Argument marshalling only: every step (planning, permutation, attention) runs
in the library's CUDA kernels, reached through the C ABI of ``include/tsr.h``.
There is no CPU path; without the built library every call raises.

The names follow the C ABI:

    mask = make_mask(kind, B, H, N, d, blocks=..., bq=64, bk=64)   # device tensors
    plan = tsr_plan(mask)                                            # physical tile plan
    out, lse = tsr_bsa_forward(q, k, v, plan)                        # bf16 O, fp32 lse
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "TsrError", "build", "lib", "make_mask", "Mask", "Plan", "tsr_plan", "tsr_plan_update",
    "tsr_bsa_forward",
    "tsr_bsa_forward_batch", "tsr_plan_device_status", "tsr_temporal_permute", "tsr_svg_route",
    "tsr_attention_host",
    "tsr_regime_load",
    "tsr_regime_lookup", "tsr_abi_version", "UNIFORM", "SEGMENTS", "SVG", "KEYLIST",
    "ORIENT_ROWS", "ORIENT_KEYS",
    "PLAN_SYNC_CHECK", "PLAN_NO_LPT", "PLAN_TEST_STALL", "PLAN_DEBUG_CHECKS",
    "PLAN_TEMPORAL_TILES",
]

UNIFORM, SEGMENTS, SVG, KEYLIST = 0, 1, 2, 3
ORIENT_ROWS, ORIENT_KEYS = 1, 2
PLAN_SYNC_CHECK, PLAN_NO_LPT, PLAN_TEST_STALL, PLAN_DEBUG_CHECKS = 1, 2, 4, 8
PLAN_TEMPORAL_TILES = 16
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "out of memory",
           5: "device wait timed out", 6: "internal error"}

REGIME_TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "regimes_gb300.txt")


class TsrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


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


class _Request(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("plan", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class _Opts(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("orient", ctypes.c_int32), ("kv_split", ctypes.c_int32)]


class _Stats(ctypes.Structure):
    _fields_ = [("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("gathered", ctypes.c_int32),
                ("n_temporal_heads", ctypes.c_int32), ("n_items", ctypes.c_int64),
                ("n_entries", ctypes.c_int64), ("n_boundary", ctypes.c_int64),
                ("n_logical_on", ctypes.c_int64), ("n_logical_total", ctypes.c_int64),
                ("max_item_len", ctypes.c_int64), ("regime_id", ctypes.c_int32),
                ("orient", ctypes.c_int32), ("kv_split", ctypes.c_int32),
                ("temporal_band", ctypes.c_int32)]


class _Regime(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("id", ctypes.c_int32), ("orient", ctypes.c_int32)]


_LIB = None
EXPORTS = ("tsr_abi_version", "tsr_status_string", "tsr_last_error", "tsr_plan", "tsr_plan_update",
           "tsr_bsa_forward", "tsr_bsa_forward_batch", "tsr_plan_device_status", "tsr_plan_destroy", "tsr_plan_get_stats",
           "tsr_plan_export", "tsr_temporal_permute", "tsr_svg_route", "tsr_attention_host",
           "tsr_release_host_buffers", "tsr_regime_load", "tsr_regime_lookup")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (sm_103a) and return its path."""
    return _build.build(force=force, verbose=verbose)


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"the CUDA library is not built ({_build.LIB} missing): "
                           "call block_sparse_attention_tsr_gb300.build() first")
    L = ctypes.CDLL(_build.LIB)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "tsr_abi_version": ([], I32),
        "tsr_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "tsr_last_error": ([], ctypes.c_char_p),
        "tsr_plan": ([P, P, P, P], ctypes.c_int),
        "tsr_plan_update": ([P, P, P], ctypes.c_int),
        "tsr_bsa_forward": ([P, P, P, P, P, P, P], ctypes.c_int),
        "tsr_bsa_forward_batch": ([P, I32, P], ctypes.c_int),
        "tsr_plan_device_status": ([P, P], ctypes.c_int),
        "tsr_plan_destroy": ([P], ctypes.c_int),
        "tsr_plan_get_stats": ([P, P], ctypes.c_int),
        "tsr_plan_export": ([P, P, P], ctypes.c_int),
        "tsr_temporal_permute": ([P, P, I32, I32, I32, I32, I32, P, I32, P], ctypes.c_int),
        "tsr_svg_route": ([P, P, P, I32, I32, I32, I32, I32, I32, P, I32, P, P, P], ctypes.c_int),
        "tsr_attention_host": ([P, P, P, P, P, P, P], ctypes.c_int),
        "tsr_release_host_buffers": ([], None),
        "tsr_regime_load": ([ctypes.c_char_p], ctypes.c_int),
        "tsr_regime_lookup": ([I32, I32, I32, I32, ctypes.c_double, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _LIB = L
    if os.path.exists(REGIME_TABLE):
        _check(L.tsr_regime_load(REGIME_TABLE.encode()))
    return _LIB


def _check(status: int) -> None:
    if status != 0:
        msg = _LIB.tsr_last_error().decode(errors="replace") if _LIB is not None else ""
        raise TsrError(status, msg)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dptr(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError("mask and tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


class Mask:
    """A tsr_mask struct plus the device tensors it points into (kept alive)."""

    def __init__(self, kind: int, B: int, H: int, N: int, d: int, *, bq: int = 0, bk: int = 0,
                 blocks=None, q_bounds=None, k_bounds=None, head_kind=None, n_frames: int = 0,
                 frame_size: int = 0, slice_m: int = 0, indptr=None, indices=None,
                 temporal_radius: int = 0):
        self.tensors = dict(blocks=blocks, q_bounds=q_bounds, k_bounds=k_bounds,
                            head_kind=head_kind, indptr=indptr, indices=indices)
        s = _Mask()
        s.kind, s.B, s.H, s.N, s.d = kind, B, H, N, d
        s.bq, s.bk = bq, bk
        s.blocks = _dptr(blocks)
        s.q_bounds, s.k_bounds = _dptr(q_bounds), _dptr(k_bounds)
        s.n_qseg = q_bounds.numel() - 1 if q_bounds is not None else 0
        s.n_kseg = k_bounds.numel() - 1 if k_bounds is not None else 0
        s.head_kind = _dptr(head_kind)
        s.n_frames, s.frame_size = n_frames, frame_size
        s.slice_m = slice_m
        s.indptr, s.indices = _dptr(indptr), _dptr(indices)
        s.temporal_radius = int(temporal_radius)
        self.struct = s
        self.kind, self.B, self.H, self.N, self.d = kind, B, H, N, d


def make_mask(kind: int, B: int, H: int, N: int, d: int, **kw) -> Mask:
    return Mask(kind, B, H, N, d, **kw)


class Plan:
    """Owner of a tsr_plan_t; released by destroy() or garbage collection."""

    def __init__(self, handle: int, mask: Mask):
        self.handle = handle
        self.mask = mask
        self.B, self.H, self.N, self.d = mask.B, mask.H, mask.N, mask.d

    def update(self, mask: "Mask", stream=None) -> "Plan":
        """Re-plan for a new mask of the same shape, reusing the plan's storage."""
        _check(lib().tsr_plan_update(self.handle, ctypes.byref(mask.struct), _stream_ptr(stream)))
        self.mask = mask
        return self

    def stats(self) -> dict:
        st = _Stats()
        _check(lib().tsr_plan_get_stats(self.handle, ctypes.byref(st)))
        return {f: getattr(st, f) for f, _ in st._fields_}

    def export(self) -> bytes:
        n = ctypes.c_size_t(0)
        _check(lib().tsr_plan_export(self.handle, None, ctypes.byref(n)))
        buf = (ctypes.c_uint8 * n.value)()
        _check(lib().tsr_plan_export(self.handle, buf, ctypes.byref(n)))
        return bytes(buf)[: n.value]

    def destroy(self) -> None:
        if self.handle:
            lib().tsr_plan_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _opts(opts) -> Optional[_Opts]:
    if opts is None:
        return None
    unknown = set(opts) - {"bn", "stages", "ctas_per_sm", "flags", "orient", "kv_split"}
    if unknown:
        raise ValueError(f"unknown plan option(s): {sorted(unknown)}")
    o = _Opts()
    o.bn = int(opts.get("bn", 0))
    o.stages = int(opts.get("stages", 0))
    o.ctas_per_sm = int(opts.get("ctas_per_sm", 0))
    o.flags = int(opts.get("flags", 0))
    o.orient = int(opts.get("orient", 0))
    o.kv_split = int(opts.get("kv_split", 0))
    return o


def tsr_plan(mask: Mask, opts: Optional[dict] = None, stream=None) -> Plan:
    """Physical tile plan of `mask` (see tsr_plan in include/tsr.h)."""
    L = lib()
    h = ctypes.c_void_p(0)
    o = _opts(opts)
    _check(L.tsr_plan(ctypes.byref(mask.struct), ctypes.byref(o) if o is not None else None,
                      ctypes.byref(h), _stream_ptr(stream)))
    return Plan(h.value, mask)


def tsr_plan_update(plan: Plan, mask: Mask, stream=None) -> Plan:
    return plan.update(mask, stream)


def tsr_bsa_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, plan: Plan,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    stream=None):
    """Attention over `plan`: returns (out bf16 [B,H,N,d], lse fp32 [B,H,N])."""
    shape = (plan.B, plan.H, plan.N, plan.d)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != shape:
            raise ValueError(f"q, k, v must be bf16 of shape {shape}")
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(shape[:3], dtype=torch.float32, device=q.device)
    _check(lib().tsr_bsa_forward(_dptr(q), _dptr(k), _dptr(v), plan.handle, _dptr(out),
                                 _dptr(lse), _stream_ptr(stream)))
    return out, lse


def tsr_plan_device_status(plan: Plan, stream=None) -> None:
    _check(lib().tsr_plan_device_status(plan.handle, _stream_ptr(stream)))


def tsr_temporal_permute(src: torch.Tensor, dst: torch.Tensor, n_frames: int, frame_size: int,
                         head_kind=None, inverse: bool = False, stream=None) -> torch.Tensor:
    """Temporal-major permutation of [B, H, F*S, row] tensors (see include/tsr.h)."""
    B, H, N = src.shape[:3]
    row_bytes = src[0, 0, 0].numel() * src.element_size()
    hk = None
    if head_kind is not None:
        hk_arr = (ctypes.c_int8 * H)(*[int(x) for x in head_kind])
        hk = ctypes.cast(hk_arr, ctypes.c_void_p)
    _check(lib().tsr_temporal_permute(_dptr(src), _dptr(dst), B, H, n_frames, frame_size,
                                      row_bytes, hk, 1 if inverse else 0, _stream_ptr(stream)))
    return dst


def tsr_bsa_forward_batch(requests, stream=None):
    """Several requests in one launch (see include/tsr.h).  ``requests``: a
    sequence of (q, k, v, plan) or (q, k, v, plan, out, lse); returns the list
    of (out, lse)."""
    n = len(requests)
    arr = (_Request * max(1, n))()
    outs = []
    for i, rq in enumerate(requests):
        q, k, v, plan = rq[:4]
        out = rq[4] if len(rq) > 4 and rq[4] is not None else torch.empty_like(q)
        lse = (rq[5] if len(rq) > 5 and rq[5] is not None else
               torch.empty(q.shape[:3], dtype=torch.float32, device=q.device))
        arr[i].q, arr[i].k, arr[i].v = _dptr(q), _dptr(k), _dptr(v)
        arr[i].plan = plan.handle
        arr[i].out, arr[i].lse = _dptr(out), _dptr(lse)
        outs.append((out, lse))
    _check(lib().tsr_bsa_forward_batch(ctypes.cast(arr, ctypes.c_void_p), n, _stream_ptr(stream)))
    return outs


def tsr_svg_route(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_frames: int,
                  frame_size: int, samples, temporal_radius: int = 0, stats=None,
                  head_kind=None, stream=None):
    """Route each head to the spatial or temporal SVG pattern from sampled query
    rows (see include/tsr.h).  Returns (stats fp32 [B, H, 3], head_kind int8 [H]),
    both on q's device; ``samples`` is a host sequence of row indices."""
    B, H, N, d = q.shape
    if N != n_frames * frame_size or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [B, H, n_frames * frame_size, d] alike")
    if stats is None:
        stats = torch.empty((B, H, 3), dtype=torch.float32, device=q.device)
    if head_kind is None:
        head_kind = torch.empty((H,), dtype=torch.int8, device=q.device)
    smp = [int(x) for x in samples]
    arr = (ctypes.c_int32 * max(1, len(smp)))(*smp)
    _check(lib().tsr_svg_route(_dptr(q), _dptr(k), _dptr(v), B, H, n_frames, frame_size, d,
                               temporal_radius, ctypes.cast(arr, ctypes.c_void_p), len(smp),
                               _dptr(stats), _dptr(head_kind), _stream_ptr(stream)))
    return stats, head_kind


def tsr_attention_host(kind: int, B: int, H: int, N: int, d: int, q, k, v, out, lse,
                       opts: Optional[dict] = None, **mask_arrays):
    """One whole call from host memory.  q, k, v, out: CPU bf16 tensors (pinned for
    speed), lse: CPU fp32; mask arrays are CPU tensors / NumPy arrays."""
    import numpy as np
    keep = []

    def hptr(x):
        if x is None:
            return 0
        if isinstance(x, torch.Tensor):
            if x.is_cuda or not x.is_contiguous():
                raise ValueError("host tensors must be contiguous CPU tensors")
            keep.append(x)
            return x.data_ptr()
        a = np.ascontiguousarray(x)
        keep.append(a)
        return a.ctypes.data

    s = _Mask()
    s.kind, s.B, s.H, s.N, s.d = kind, B, H, N, d
    s.bq, s.bk = mask_arrays.get("bq", 0), mask_arrays.get("bk", 0)
    s.blocks = hptr(mask_arrays.get("blocks"))
    qb, kb = mask_arrays.get("q_bounds"), mask_arrays.get("k_bounds")
    s.q_bounds, s.k_bounds = hptr(qb), hptr(kb)
    s.n_qseg = len(qb) - 1 if qb is not None else 0
    s.n_kseg = len(kb) - 1 if kb is not None else 0
    s.head_kind = hptr(mask_arrays.get("head_kind"))
    s.n_frames, s.frame_size = mask_arrays.get("n_frames", 0), mask_arrays.get("frame_size", 0)
    s.slice_m = mask_arrays.get("slice_m", 0)
    s.indptr, s.indices = hptr(mask_arrays.get("indptr")), hptr(mask_arrays.get("indices"))
    s.temporal_radius = int(mask_arrays.get("temporal_radius", 0))
    o = _opts(opts)
    _check(lib().tsr_attention_host(ctypes.byref(s), ctypes.byref(o) if o is not None else None,
                                    hptr(q), hptr(k), hptr(v), hptr(out), hptr(lse)))
    return out, lse


def tsr_regime_load(path: Optional[str]) -> None:
    _check(lib().tsr_regime_load(path.encode() if path else None))


def tsr_regime_lookup(kind: int, bq: int, bk: int, N: int, density: float) -> dict:
    r = _Regime()
    _check(lib().tsr_regime_lookup(kind, bq, bk, N, density, ctypes.byref(r)))
    return {"bn": r.bn, "stages": r.stages, "ctas_per_sm": r.ctas_per_sm, "id": r.id,
            "orient": r.orient}


def tsr_abi_version() -> int:
    return int(lib().tsr_abi_version())
