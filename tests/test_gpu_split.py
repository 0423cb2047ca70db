"""Split-KV on the GPU: each work item's key tiles cut into 2 or 4 parts, each
part writing its normalised partial O and lse, the last part of an item merging
them in the attention kernel (lse = log sum_p e^lse_p, O = sum_p e^(lse_p - lse)
O_p; all parts empty gives O = 0, lse = -inf).  Against the CPU oracle at the
stated tolerances, in both tile orientations and every mask form, with parts
that hold no tile, empty rows, the rescale path, plan updates, the automatic
rule (few work items per CTA slot), the batched launch, the debug checks and
the host entry point.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W
from test_gpu_parity import _sample_rows, check_coverage, compare, run

pytestmark = pytest.mark.gpu

ORIENTS = {"rows": tsr.ORIENT_ROWS, "keys": tsr.ORIENT_KEYS}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def parity(spec, d, seed, opts, scale=1.0, qkv=None):
    (q, k, v), plan, O, L = run(spec, d, seed=seed, opts=opts, scale=scale, qkv=qkv)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"split {opts}")
    check_coverage(spec, plan)
    return (q, k, v), plan, O, L


@pytest.mark.parametrize("orient", ORIENTS)
@pytest.mark.parametrize("s", [2, 4])
def test_tiny_block_mask(orient, s):
    spec = W.tiny_block_mask(seed=1)                 # one fully masked query block per head
    _, plan, O, L = parity(spec, 128, 1, {"orient": ORIENTS[orient], "kv_split": s})
    assert plan.stats()["kv_split"] == s
    assert np.sum(~np.isfinite(L)) == 2 * 64


UNIFORM = [
    # (N, H, bq, bk, p)
    (1000, 2, 64, 64, 0.3),
    (4096, 1, 64, 64, 0.9),                          # long lists: many tiles per part
    (900, 1, 64, 256, 0.5),
    (1100, 1, 16, 48, 0.3),
]


@pytest.mark.parametrize("orient", ORIENTS)
@pytest.mark.parametrize("s", [2, 4])
@pytest.mark.parametrize("case", UNIFORM, ids=[str(i) for i in range(len(UNIFORM))])
def test_uniform(case, s, orient):
    N, H, bq, bk, p = case
    r = np.random.Generator(np.random.PCG64(N + bq + 11))
    blocks = (r.random((1, H, -(-N // bq), -(-N // bk))) < p).astype(np.uint8)
    blocks[0, 0, 1, :] = 0                           # an empty query block
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=bq, bk=bk, blocks=blocks)
    parity(spec, 128, N, {"orient": ORIENTS[orient], "kv_split": s}, scale=1.5)


def test_d64_rows():
    r = np.random.Generator(np.random.PCG64(64))
    blocks = (r.random((1, 2, 18, 18)) < 0.4).astype(np.uint8)
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, 2, 1100, bq=64, bk=64, blocks=blocks)
    parity(spec, 64, 5, {"kv_split": 4})


@pytest.mark.parametrize("orient", ORIENTS)
def test_parts_without_tiles(orient):
    """Query block i lists i + 1 key tiles, cut into 4 parts: the short items'
    first parts hold no tile (lse -inf, O 0) and the merge must ignore them."""
    N, nb = 64 * 12, 12
    blocks = np.zeros((1, 1, nb, nb), np.uint8)
    for i in range(nb):
        blocks[0, 0, i, :i + 1] = 1
    blocks[0, 0, 5, :] = 0                           # and one empty row block
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=64, bk=64, blocks=blocks)
    _, _, O, L = parity(spec, 128, 3, {"orient": ORIENTS[orient], "kv_split": 4})
    assert np.all(L[0, 0, 5 * 64:6 * 64] == -np.inf) and np.all(O[0, 0, 5 * 64:6 * 64] == 0)


@pytest.mark.parametrize("orient", ORIENTS)
@pytest.mark.parametrize("F,S,kinds,r", [(16, 48, [0, 1, 1, 0], 0), (5, 130, [1, 1, 0], 40)])
def test_svg(F, S, kinds, r, orient):
    """Temporal heads gather their rows through the temporal-major permutation
    and the merged rows are stored back in frame-major order (radius-0 heads
    kept on the tiles by TSR_PLAN_TEMPORAL_TILES)."""
    spec = W.svg_mask(2, len(kinds), n_frames=F, frame_size=S, kinds=np.array(kinds, np.int8),
                      temporal_radius=r)
    parity(spec, 128, 21 + F, {"orient": ORIENTS[orient], "kv_split": 2,
                               "flags": tsr.PLAN_TEMPORAL_TILES})


KEYLIST = [
    # (N, H, slice_m, lo, hi)
    (1000, 2, 64, 0, 400),
    (1024, 1, 128, 0, 300),
    (300, 1, 64, 0, 0),                              # every list empty
]


@pytest.mark.parametrize("orient", ORIENTS)
@pytest.mark.parametrize("s", [2, 4])
@pytest.mark.parametrize("case", KEYLIST, ids=[str(i) for i in range(len(KEYLIST))])
def test_keylist(case, s, orient):
    N, H, M, lo, hi = case
    spec = W.random_keylist(N + M + 3, 1, H, N, slice_m=M, lo=lo, hi=hi)
    parity(spec, 128, N + 1, {"orient": ORIENTS[orient], "kv_split": s})


@pytest.mark.parametrize("orient", ORIENTS)
def test_rescale_path_large_logits(orient):
    """Large, growing logits: every part raises its running maximum many times,
    and the parts' maxima differ widely before the merge."""
    N = 4096
    spec = W.tiny_block_mask(seed=6, N=N)
    q, k, v = W.qkv(1, 2, N, 128, 3)
    q = (q.float() * 4.0).to(torch.bfloat16)
    ramp = torch.linspace(0.1, 4.0, N).view(1, 1, -1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    parity(spec, 128, 0, {"orient": ORIENTS[orient], "kv_split": 4}, qkv=(q, k, v))


@pytest.mark.parametrize("orient", ORIENTS)
def test_plan_update_keeps_splitting(orient):
    N, H = 1500, 2
    q, k, v = W.qkv(1, H, N, 128, 21)
    r = np.random.Generator(np.random.PCG64(23))
    specs = [W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=64, bk=64,
                        blocks=(r.random((1, H, 24, 24)) < 0.3).astype(np.uint8)),
             W.segment_mask(9, 1, H, N, lo=16, hi=200),
             W.random_keylist(22, 1, H, N, slice_m=64, lo=0, hi=500)]
    plan = None
    for spec in specs:
        mask = tsr.make_mask(spec.kind, 1, H, N, 128, **W.mask_tensors(spec))
        opts = {"orient": ORIENTS[orient], "kv_split": 2}
        plan = tsr.tsr_plan(mask, opts) if plan is None else plan.update(mask)
        assert plan.stats()["kv_split"] == 2
        out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().double().numpy(), "update")
    tsr.tsr_plan_device_status(plan)


def test_automatic_rule():
    """128-row plans are split automatically only when their work items are
    fewer than the CTA slots: a one-head 8,192-token layer (64 items on two
    CTAs per SM, 304 slots) into four parts, a one-head 480p layer (256 items)
    into two, a 24-head one not at all; key-major plans are not split
    automatically; kv_split = 1 turns it off.  The split small layer is checked
    against the oracle."""
    small = W.video_block_mask(seed=2, H=1, N=8192)
    rows2 = {"orient": tsr.ORIENT_ROWS, "bn": 64, "stages": 2, "ctas_per_sm": 2}
    (q, k, v), plan, O, L = parity(small, 128, 2, rows2)
    assert plan.stats()["kv_split"] == 4
    (q, k, v), plan, O, L = parity(small, 128, 2, {"orient": tsr.ORIENT_KEYS})
    assert plan.stats()["kv_split"] == 1
    mask = tsr.make_mask(small.kind, 1, 1, small.N, 128, **W.mask_tensors(small))
    assert tsr.tsr_plan(mask, dict(rows2, kv_split=1)).stats()["kv_split"] == 1
    for H in (1, 24):
        spec = W.video_block_mask(seed=2, H=H)
        mask = tsr.make_mask(spec.kind, 1, H, spec.N, 128, **W.mask_tensors(spec))
        assert tsr.tsr_plan(mask, {"orient": tsr.ORIENT_KEYS}).stats()["kv_split"] == 1
        assert tsr.tsr_plan(mask, {"orient": tsr.ORIENT_ROWS, "bn": 64, "stages": 2,
                                   "ctas_per_sm": 2}).stats()["kv_split"] == (2 if H == 1 else 1)


def test_one_head_480p_split_sampled():
    """A one-head 480p layer cut into four parts, on sampled rows."""
    one = W.video_block_mask(seed=2, H=1)
    (q, k, v), plan, O, L = run(one, 128, seed=2, opts={"kv_split": 4})
    assert plan.stats()["kv_split"] == 4
    rows = _sample_rows(one, 64, 2)
    O_ref, L_ref, _ = oracle.attention_rows(one, q, k, v, rows)
    compare(O_ref, L_ref, O.reshape(-1, 128)[rows], L.reshape(-1)[rows], "480p one head, split")


@pytest.mark.parametrize("orient", ORIENTS)
def test_batched_launch_matches_single_launches(orient):
    specs = [W.video_block_mask(seed=31, H=2, N=3000), W.tiny_block_mask(seed=32, H=3, N=1024)]
    # batched launches are compiled for the default 128-row regime
    regime = {"bn": 64, "stages": 2, "ctas_per_sm": 2} if orient == "rows" else {}
    reqs, singles = [], []
    for i, spec in enumerate(specs):
        (q, k, v), plan, O, L = parity(spec, 128, 40 + i,
                                       dict(regime, orient=ORIENTS[orient], kv_split=2 + 2 * i))
        reqs.append((q.cuda(), k.cuda(), v.cuda(), plan))
        singles.append((O, L))
    outs = tsr.tsr_bsa_forward_batch(reqs)
    torch.cuda.synchronize()
    for (o, l), (O, L) in zip(outs, singles):
        assert np.array_equal(o.float().cpu().numpy(), O)
        assert np.array_equal(l.cpu().double().numpy(), L)


@pytest.mark.parametrize("orient", ORIENTS)
def test_debug_checks(orient):
    """The device plan checks pass on split plans, every launch computes each
    tile exactly once over all parts, and the results are unchanged."""
    spec = W.random_keylist(15, 1, 2, 900, slice_m=64, lo=0, hi=300)
    opts = {"orient": ORIENTS[orient], "kv_split": 4}
    (q, k, v), plan, O, L = run(spec, 128, seed=13, opts=dict(opts, flags=tsr.PLAN_DEBUG_CHECKS))
    _, _, O2, L2 = run(spec, 128, seed=13, opts=opts, qkv=(q, k, v))
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


@pytest.mark.parametrize("which", ["uniform", "keylist"])
def test_host_entry_point_with_split(which):
    """An explicit split is honoured by the host entry point (one plan over all
    heads, or one plan per head group for key lists); a part's result depends
    only on its item and the number of parts, so the output equals the device
    path bit for bit."""
    opts = {"kv_split": 2}
    if which == "uniform":
        spec = W.video_block_mask(seed=5, H=6, N=8192)
        kw = dict(bq=64, bk=64, blocks=spec.blocks)
    else:
        spec = W.keylist_mask(seed=6, H=4, N=8192)
        kw = dict(slice_m=64, indptr=spec.indptr, indices=spec.indices)
    q, k, v = W.qkv(spec.B, spec.H, spec.N, 128, 17)
    _, plan, O, L = run(spec, 128, seed=0, opts=opts, qkv=(q, k, v))
    assert plan.stats()["kv_split"] == 2
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
    for _ in range(2):
        tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, 128, q.pin_memory(),
                               k.pin_memory(), v.pin_memory(), out, lse, opts=opts, **kw)
        assert np.array_equal(out.float().numpy(), O)
        assert np.array_equal(lse.double().numpy(), L)
