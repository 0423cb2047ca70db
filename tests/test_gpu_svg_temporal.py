"""SVG temporal heads of radius 0 by spatial position: with n_frames <= 32 each
temporal head is frame_size independent F x F blocks, computed by their own
kernel (on a stream the plan owns, forked from the call's stream and joined
back), while the attention kernel runs the spatial heads' items only.  Against the CPU oracle at the stated tolerances: frame counts 1 to 32,
frame sizes that leave a ragged last CTA of positions, d = 64 and 128, both tile
orientations, split-KV, plan updates that change the head kinds, every head
temporal, the batched launch and the host entry point.  The attention-tile
path for the same heads (TSR_PLAN_TEMPORAL_TILES) stays correct, and plans
that cannot use the kernel (radius > 0, more than 32 frames, debug checks)
keep the tiles.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W
from test_gpu_parity import check_coverage, compare, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def parity(spec, d, seed, opts=None, band=1):
    (q, k, v), plan, O, L = run(spec, d, seed=seed, opts=opts)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"svg temporal {spec.meta.get('workload')} {opts}")
    check_coverage(spec, plan)                       # the plan keeps the temporal items
    assert plan.stats()["temporal_band"] == band
    return (q, k, v), plan, O, L


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("F,S", [(1, 37), (5, 130), (13, 50), (16, 41), (21, 78), (32, 19)])
def test_band_against_oracle(F, S, d):
    spec = W.svg_mask(2, 3, n_frames=F, frame_size=S, kinds=np.array([1, 0, 1], np.int8))
    parity(spec, d, seed=F * 7 + S)


@pytest.mark.parametrize("orient", [tsr.ORIENT_ROWS, tsr.ORIENT_KEYS])
def test_band_with_either_orientation(orient):
    spec = W.svg_mask(1, 4, n_frames=21, frame_size=60, kinds=np.array([0, 1, 0, 1], np.int8))
    _, plan, _, _ = parity(spec, 128, seed=3, opts={"orient": orient})
    assert plan.stats()["orient"] == orient


def test_band_matches_tiles():
    """The same inputs through the per-position kernel and through the
    attention tiles: both within tolerance of the oracle, and close to each
    other (the sums run in another order; both round P to bf16)."""
    spec = W.svg_mask(2, 2, n_frames=16, frame_size=48, kinds=np.array([1, 0], np.int8))
    qkv, _, O1, L1 = parity(spec, 128, seed=9, opts={"kv_split": 1})
    _, _, O2, L2 = parity(spec, 128, seed=9, opts={"flags": tsr.PLAN_TEMPORAL_TILES, "kv_split": 1},
                          band=0)
    # spatial heads take the same tiles either way (no split: the launch lists
    # differ in length, which could change an automatic split)
    assert np.array_equal(O1[:, 1], O2[:, 1]) and np.array_equal(L1[:, 1], L2[:, 1])
    assert np.abs(O1 - O2).max() <= 2e-2
    assert np.abs(L1 - L2).max() <= 1e-3 * max(1.0, np.abs(L1).max())


@pytest.mark.parametrize("opts,r,F,why", [
    ({"flags": tsr.PLAN_TEMPORAL_TILES}, 0, 16, "flag"),
    (None, 1, 16, "radius"),
    (None, 0, 33, "frames"),
    ({"flags": tsr.PLAN_DEBUG_CHECKS}, 0, 16, "debug checks"),
])
def test_tiles_where_the_kernel_does_not_apply(opts, r, F, why):
    spec = W.svg_mask(1, 3, n_frames=F, frame_size=24, kinds=np.array([1, 0, 1], np.int8),
                      temporal_radius=r)
    parity(spec, 128, seed=F + r, opts=opts, band=0)


def test_every_head_temporal():
    """No spatial item at all: the attention launch is empty, the per-position
    kernel writes every row."""
    spec = W.svg_mask(2, 2, n_frames=8, frame_size=100, kinds=np.array([1, 1], np.int8))
    parity(spec, 128, seed=4)


@pytest.mark.parametrize("orient", [tsr.ORIENT_ROWS, tsr.ORIENT_KEYS])
@pytest.mark.parametrize("s", [2, 4])
def test_band_with_split_kv(s, orient):
    """Split-KV cuts the launch list (spatial items only): units, partial
    results and arrival counters are indexed in that list."""
    spec = W.svg_mask(2, 3, n_frames=16, frame_size=48, kinds=np.array([0, 1, 0], np.int8))
    _, plan, _, _ = parity(spec, 128, seed=5 + s, opts={"orient": orient, "kv_split": s})
    assert plan.stats()["kv_split"] == s


def test_plan_update_changes_head_kinds():
    """Re-planning with other head kinds rebuilds the launch list; an update to
    a radius-1 mask falls back to the tiles, and back again."""
    F, S, H, d = 16, 41, 3, 128
    q, k, v = W.qkv(1, H, F * S, d, 77)
    plan = None
    for kinds, r in (([1, 0, 1], 0), ([0, 1, 1], 0), ([0, 1, 1], 1), ([1, 1, 0], 0)):
        spec = W.svg_mask(1, H, n_frames=F, frame_size=S, kinds=np.array(kinds, np.int8),
                          temporal_radius=r)
        mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, d, **W.mask_tensors(spec))
        if plan is None:
            plan = tsr.tsr_plan(mask)
        else:
            plan.update(mask)
        assert plan.stats()["temporal_band"] == (1 if r == 0 else 0)
        out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
        torch.cuda.synchronize()
        tsr.tsr_plan_device_status(plan)
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().numpy().astype(np.float64),
                f"update {kinds} r={r}")
        check_coverage(spec, plan)


def test_batched_launch():
    """Two SVG requests and a block mask in one attention launch; each SVG
    request's temporal heads then run on their own."""
    specs = [W.svg_mask(1, 3, n_frames=16, frame_size=41, kinds=np.array([1, 0, 1], np.int8)),
             W.tiny_block_mask(seed=3),
             W.svg_mask(2, 2, n_frames=21, frame_size=30, kinds=np.array([0, 1], np.int8))]
    d = 128
    opts = {"orient": tsr.ORIENT_ROWS, "bn": 64, "stages": 2, "ctas_per_sm": 2, "kv_split": 1}
    reqs, keep = [], []
    for i, spec in enumerate(specs):
        q, k, v = W.qkv(spec.B, spec.H, spec.N, d, 50 + i)
        mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, d, **W.mask_tensors(spec))
        plan = tsr.tsr_plan(mask, opts)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        out = torch.empty_like(qd)
        lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32, device="cuda")
        reqs.append((qd, kd, vd, plan, out, lse))
        keep.append((spec, q, k, v, plan))
    tsr.tsr_bsa_forward_batch(reqs)
    torch.cuda.synchronize()
    for (spec, q, k, v, plan), (_, _, _, _, out, lse) in zip(keep, reqs):
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().numpy().astype(np.float64),
                f"batch {spec.meta.get('workload')}")
        if spec.kind == W.MASK_SVG:
            assert plan.stats()["temporal_band"] == 1


def test_host_entry_point():
    """tsr_attention_host takes one plan over all heads and launches each head
    group's range: the spatial items of the group's heads, then the group's
    temporal heads.  B = 3, H = 3 puts groups across batches."""
    spec = W.svg_mask(3, 3, n_frames=21, frame_size=120, kinds=np.array([1, 0, 1], np.int8))
    opts = {"kv_split": 1}
    q, k, v = W.qkv(spec.B, spec.H, spec.N, 128, 17)
    _, plan, O, L = run(spec, 128, seed=0, opts=opts, qkv=(q, k, v))
    assert plan.stats()["temporal_band"] == 1
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
    tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, 128, q.pin_memory(), k.pin_memory(),
                           v.pin_memory(), out, lse, opts=opts, n_frames=21, frame_size=120,
                           head_kind=spec.head_kind)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, out.float().numpy(), lse.double().numpy(), "host")
    # the temporal heads are computed by the same kernel either way
    for b in range(3):
        for h in (0, 2):
            assert np.array_equal(out[b, h].float().numpy(), O[b, h])
            assert np.array_equal(lse[b, h].double().numpy(), L[b, h])
