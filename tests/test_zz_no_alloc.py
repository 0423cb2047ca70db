"""tsr_attention_noalloc: attention for callers that cannot allocate device memory.

Callers whose device memory all comes from their own pool, or who cannot afford
cudaMalloc / cudaFree on their path, get one entry point that plans into and
runs over a fixed 32 MiB scratch array inside the library.  These tests call it
through the C ABI and check it against the allocating path (tsr_plan +
tsr_bsa_forward) and against the CPU oracle with the parity tolerances, on two
calls in a row with
different masks (the shared scratch keeps the previous call's contents), and
check that a plan too large for the scratch is refused with a clear error.

This file is collected last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_REL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def L():
    tsr.build()
    lib = tsr.lib()
    f = lib.tsr_attention_noalloc
    f.argtypes = [ctypes.c_void_p] * 7
    f.restype = ctypes.c_int
    return lib


def _noalloc(L, mask, q, k, v, out, lse):
    return L.tsr_attention_noalloc(ctypes.byref(mask.struct), q.data_ptr(), k.data_ptr(),
                                   v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)


def _close(o_a, l_a, o_b, l_b):
    """o_a, l_a: the call under test; o_b, l_b: the reference (tensors or arrays)."""
    as_np = lambda t, f: t if isinstance(t, np.ndarray) else f(t).cpu().numpy()
    o_a, o_b = as_np(o_a, lambda t: t.float()), as_np(o_b, lambda t: t.float())
    l_a, l_b = as_np(l_a, lambda t: t.double()), as_np(l_b, lambda t: t.double())
    fin = np.isfinite(l_b)
    assert np.array_equal(np.isfinite(l_a), fin)
    assert np.all(o_a[~fin] == 0.0)
    d = np.abs(o_a[fin] - o_b[fin])
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS
    assert (np.abs(l_a[fin] - l_b[fin]) / np.maximum(1.0, np.abs(l_b[fin]))).max() <= LSE_REL


def _case(spec, d, seed):
    q, k, v = (x.cuda() for x in W.qkv(spec.B, spec.H, spec.N, d, seed))
    mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, d, **W.mask_tensors(spec))
    return mask, q, k, v


def test_noalloc_matches_allocating_path_two_calls(L):
    cases = [
        (W.tiny_block_mask(seed=3, H=4, N=2048), 128, 1),    # larger plan first
        (W.segment_mask(5, 1, 2, 1500, lo=16, hi=300), 64, 2),  # then a smaller, different one
    ]
    for spec, d, seed in cases:
        mask, q, k, v = _case(spec, d, seed)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((spec.B, spec.H, spec.N), float("nan"), device="cuda")
        st = _noalloc(L, mask, q, k, v, out, lse)
        assert st == 0, L.tsr_last_error()
        plan = tsr.tsr_plan(mask)
        o_ref, l_ref = tsr.tsr_bsa_forward(q, k, v, plan)
        torch.cuda.synchronize()
        _close(out, lse, o_ref, l_ref)
        o_or, l_or = oracle.attention(spec, q.cpu(), k.cpu(), v.cpu())
        _close(out, lse, o_or, l_or)


def test_noalloc_refuses_plans_beyond_the_scratch(L):
    spec = W.video_block_mask(seed=2)          # 24 heads x 32,760 tokens: plan ~38 MB
    mask, q, k, v = _case(spec, 128, 2)
    out = torch.empty_like(q)
    lse = torch.empty((1, 24, spec.N), device="cuda")
    st = _noalloc(L, mask, q, k, v, out, lse)
    assert st == 2
    assert b"32 MiB" in L.tsr_last_error()
    # the library stays usable after the refusal
    small = W.tiny_block_mask(seed=4)
    mask, q, k, v = _case(small, 64, 3)
    out = torch.empty_like(q)
    lse = torch.empty((1, 2, small.N), device="cuda")
    assert _noalloc(L, mask, q, k, v, out, lse) == 0


def test_noalloc_rejects_other_mask_kinds(L):
    spec = W.svg_mask(1, 2, n_frames=16, frame_size=48, kinds=np.array([0, 1], np.int8))
    mask, q, k, v = _case(spec, 64, 1)
    out = torch.empty_like(q)
    lse = torch.empty((1, 2, spec.N), device="cuda")
    assert _noalloc(L, mask, q, k, v, out, lse) == 2
