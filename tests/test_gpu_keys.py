"""GPU parity of the key-major (transposed) tile orientation, TSR_ORIENT_KEYS.

Plans with 64-row query tiles and 64 x 64 tiles, computed two tiles per step as
S^T = K Q^T (128 keys x 64 queries) with the softmax per key lane, against the
CPU oracle at the stated tolerances (max |dO| <= 2e-2, mean |dO| <= 2e-3, lse
within 1e-3 * max(1, |lse|), empty rows exactly 0 / -inf), and the plans checked
bit-exactly against the oracle's allowed set.  Cases cover every mask form,
ragged N, empty query blocks, odd tile counts (the second tile of a step
missing), the running-maximum fix-up path, plan updates, the batched launch and
the host entry point; full-size 480p and 720p cases are sampled.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W
from test_gpu_parity import _sample_rows, check_coverage, compare, run

pytestmark = pytest.mark.gpu

KEYS = {"orient": tsr.ORIENT_KEYS}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def full_parity(spec, seed, opts=None, scale=1.0):
    (q, k, v), plan, O, L = run(spec, 128, seed=seed, opts=dict(KEYS, **(opts or {})), scale=scale)
    st = plan.stats()
    assert st["orient"] == tsr.ORIENT_KEYS and st["bm"] == 64 and st["bn"] == 64
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"keys {spec.meta.get('workload', spec.kind)}")
    cov = check_coverage(spec, plan)
    return plan, cov


def test_tiny_block_mask():
    spec = W.tiny_block_mask(seed=1)                 # one fully masked query block per head
    plan, _ = full_parity(spec, seed=1)


UNIFORM = [
    # (N, H, bq, bk, p)
    (1000, 2, 64, 64, 0.3),
    (777, 1, 32, 32, 0.4),
    (1024, 2, 128, 128, 0.5),
    (900, 1, 64, 256, 0.5),
    (900, 1, 256, 64, 0.5),
    (200, 1, 64, 64, 1.0),
    (129, 1, 16, 16, 0.5),
    (1100, 1, 16, 48, 0.3),
    (4096, 1, 64, 64, 0.9),                          # long lists: many steps per item
]


@pytest.mark.parametrize("case", UNIFORM, ids=[str(i) for i in range(len(UNIFORM))])
def test_uniform(case):
    N, H, bq, bk, p = case
    r = np.random.Generator(np.random.PCG64(N + bq + 7))
    blocks = (r.random((1, H, -(-N // bq), -(-N // bk))) < p).astype(np.uint8)
    if blocks.shape[2] > 2:
        blocks[0, 0, 2, :] = 0
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=bq, bk=bk, blocks=blocks)
    full_parity(spec, seed=N, scale=1.5)


def test_odd_and_even_tile_counts():
    """Query blocks whose lists hold 1, 2, 3, ... key tiles: steps whose second
    tile is missing (odd counts) load zero-filled rows and mask the whole lane."""
    N, nb = 64 * 12, 12
    blocks = np.zeros((1, 1, nb, nb), np.uint8)
    for i in range(nb):
        blocks[0, 0, i, :i + 1] = 1                  # block i lists i + 1 key tiles
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=64, bk=64, blocks=blocks)
    _, cov = full_parity(spec, seed=3)
    assert cov["tiles"] == nb * (nb + 1) // 2


def test_segments():
    spec = W.segment_mask(3, 1, 2, 1500, lo=16, hi=300)
    full_parity(spec, seed=5)


@pytest.mark.parametrize("F,S,kinds,r", [(16, 48, [0, 1, 1, 0], 0), (13, 50, [1, 0, 1], 0),
                                         (16, 41, [1, 0, 1], 2), (5, 130, [1, 1, 0], 40),
                                         (1, 700, [0, 1, 0], 0)])
def test_svg(F, S, kinds, r):
    """Spatial heads (TMA) and temporal heads (rows gathered through the
    temporal-major permutation, band descriptors) in one launch; ragged N.
    Radius-0 heads are kept on the tiles here (TSR_PLAN_TEMPORAL_TILES)."""
    spec = W.svg_mask(2, len(kinds), n_frames=F, frame_size=S, kinds=np.array(kinds, np.int8),
                      temporal_radius=r)
    plan, _ = full_parity(spec, seed=21 + F, opts={"flags": tsr.PLAN_TEMPORAL_TILES})
    assert plan.stats()["temporal_band"] == 0
    assert plan.stats()["n_temporal_heads"] == sum(kinds)


KEYLIST = [
    # (N, H, slice_m, lo, hi)
    (1000, 2, 64, 0, 400),
    (777, 2, 64, 1, 777),
    (1024, 1, 128, 0, 300),
    (1100, 2, 64, 5, 200),
    (640, 1, 64, 640, 640),                          # every key listed: full tiles only
    (300, 1, 64, 0, 0),                              # every list empty
]


@pytest.mark.parametrize("case", KEYLIST, ids=[str(i) for i in range(len(KEYLIST))])
def test_keylist(case):
    N, H, M, lo, hi = case
    spec = W.random_keylist(N + M + 1, 1, H, N, slice_m=M, lo=lo, hi=hi)
    plan, cov = full_parity(spec, seed=N + 1)
    assert plan.stats()["gathered"] == 1
    if lo == hi == N:
        assert cov["full"] == cov["tiles"]


def test_keylist_clustered_runs():
    spec = W.keylist_mask(seed=4, H=2, N=4096)
    full_parity(spec, seed=4)


def test_rescale_path_large_logits():
    """Large, growing logits: the reference maximum is raised (with O^T and the
    row sums rescaled) in many steps after the first."""
    N = 4096
    spec = W.tiny_block_mask(seed=6, N=N)
    q, k, v = W.qkv(1, 2, N, 128, 3)
    q = (q.float() * 4.0).to(torch.bfloat16)
    ramp = torch.linspace(0.1, 4.0, N).view(1, 1, -1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    _, _, O, L = run(spec, 128, seed=0, opts=KEYS, qkv=(q, k, v))
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "keys rescale")


def test_q_zero_closed_form():
    """Q = 0: lse_i = ln |A_i| exactly; every allowed key counted once."""
    spec = W.video_block_mask(seed=7, H=2, N=2000)
    _, k, v = W.qkv(1, 2, 2000, 128, 9)
    q = torch.zeros_like(k)
    _, _, O, L = run(spec, 128, seed=0, opts=KEYS, qkv=(q, k, v))
    cnt = oracle.count_allowed(spec)
    rows = np.array([[len(oracle.row_keys(spec, 0, h, i)) for i in range(spec.N)]
                     for h in range(spec.H)])
    assert rows.sum() == cnt.sum()
    fin = rows > 0
    assert np.all(L[0][~fin] == -np.inf)
    assert np.abs(L[0][fin] - np.log(rows[fin])).max() <= 1e-5


def test_plan_update_switches_orientation_and_masks():
    """One plan re-planned for masks of different kind and block shape, the
    orientation forced both ways: every result and plan matches the oracle."""
    N, H = 1500, 2
    q, k, v = W.qkv(1, H, N, 128, 21)
    r = np.random.Generator(np.random.PCG64(21))
    specs = [
        W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=64, bk=64,
                   blocks=(r.random((1, H, 24, 24)) < 0.2).astype(np.uint8)),
        W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=32, bk=32,
                   blocks=(r.random((1, H, 47, 47)) < 0.6).astype(np.uint8)),
        W.segment_mask(9, 1, H, N, lo=16, hi=200),
        W.random_keylist(22, 1, H, N, slice_m=64, lo=0, hi=500),
    ]
    for orient in (tsr.ORIENT_KEYS, tsr.ORIENT_ROWS):
        plan = None
        for spec in specs:
            mask = tsr.make_mask(spec.kind, 1, H, N, 128, **W.mask_tensors(spec))
            plan = tsr.tsr_plan(mask, {"orient": orient}) if plan is None else plan.update(mask)
            assert plan.stats()["orient"] == orient
            out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
            O_ref, L_ref = oracle.attention(spec, q, k, v)
            compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().double().numpy(),
                    f"update orient {orient}")
            check_coverage(spec, plan)
        tsr.tsr_plan_device_status(plan)


@pytest.mark.parametrize("which", ["uniform", "svg", "keylist"])
def test_debug_checks_pass(which):
    if which == "uniform":
        spec = W.tiny_block_mask(seed=13, N=1000)
    elif which == "svg":
        spec = W.svg_mask(2, 3, n_frames=16, frame_size=41, kinds=np.array([1, 0, 1], np.int8),
                          temporal_radius=1)
    else:
        spec = W.random_keylist(15, 1, 2, 900, slice_m=64, lo=0, hi=300)
    (q, k, v), plan, O, L = run(spec, 128, seed=13, opts=dict(KEYS, flags=tsr.PLAN_DEBUG_CHECKS))
    _, _, O2, L2 = run(spec, 128, seed=13, opts=KEYS, qkv=(q, k, v))
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def test_batched_launch_matches_single_launches():
    specs = [W.video_block_mask(seed=31, H=2, N=3000), W.svg_mask(1, 2, n_frames=8, frame_size=200),
             W.tiny_block_mask(seed=32, H=3, N=1024)]
    reqs, singles = [], []
    for i, spec in enumerate(specs):
        (q, k, v), plan, O, L = run(spec, 128, seed=40 + i, opts=KEYS)
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        compare(O_ref, L_ref, O, L, f"batch member {i}")
        reqs.append((q.cuda(), k.cuda(), v.cuda(), plan))
        singles.append((O, L))
    outs = tsr.tsr_bsa_forward_batch(reqs)
    torch.cuda.synchronize()
    for (o, l), (O, L) in zip(outs, singles):
        assert np.array_equal(o.float().cpu().numpy(), O)
        assert np.array_equal(l.cpu().double().numpy(), L)


@pytest.mark.parametrize("which", ["uniform", "keylist"])
def test_host_entry_point(which):
    if which == "uniform":
        spec = W.video_block_mask(seed=5, H=10)
        kw = dict(bq=64, bk=64, blocks=spec.blocks)
    else:
        spec = W.keylist_mask(seed=6, H=4, N=8192)
        kw = dict(slice_m=64, indptr=spec.indptr, indices=spec.indices)
    q, k, v = W.qkv(spec.B, spec.H, spec.N, 128, 17)
    # the host entry point does not split work items automatically
    _, _, O, L = run(spec, 128, seed=0, opts=dict(KEYS, kv_split=1), qkv=(q, k, v))
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
    for _ in range(2):
        tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, 128, q.pin_memory(),
                               k.pin_memory(), v.pin_memory(), out, lse, opts=KEYS, **kw)
        assert np.array_equal(out.float().numpy(), O)
        assert np.array_equal(lse.double().numpy(), L)


def test_d64_refused_and_table_falls_back():
    spec = W.tiny_block_mask(seed=1)
    mask = tsr.make_mask(spec.kind, 1, 2, spec.N, 64, **W.mask_tensors(spec))
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_plan(mask, KEYS)
    assert e.value.status == 2


# -------------------------------------------------------- full-size configs
def _sampled(spec, seed, rows_per_head=24):
    (q, k, v), plan, O, L = run(spec, 128, seed=seed, opts=KEYS)
    rows = _sample_rows(spec, rows_per_head, seed)
    O_ref, L_ref, _ = oracle.attention_rows(spec, q, k, v, rows)
    compare(O_ref, L_ref, O.reshape(-1, 128)[rows], L.reshape(-1)[rows],
            "keys " + spec.meta.get("workload", ""))
    return plan


@pytest.mark.slow
def test_video_480p_full_size():
    spec = W.video_block_mask(seed=2)
    plan = _sampled(spec, seed=2)
    one = W.MaskSpec(W.MASK_UNIFORM, 1, 2, spec.N, bq=64, bk=64,
                     blocks=np.ascontiguousarray(spec.blocks[:, :2]))
    p1 = tsr.tsr_plan(tsr.make_mask(one.kind, 1, 2, one.N, 128, **W.mask_tensors(one)), KEYS)
    check_coverage(one, p1)


@pytest.mark.slow
def test_svg_480p_full_size():
    spec = W.svg_mask(1, 24, n_frames=21, frame_size=1560)
    _sampled(spec, seed=3)


@pytest.mark.slow
def test_keylist_720p_two_heads_coverage():
    spec = W.keylist_mask(seed=4, H=2)
    (q, k, v), plan, O, L = run(spec, 128, seed=40, opts=KEYS)
    check_coverage(spec, plan)
    rows = _sample_rows(spec, 32, 40)
    O_ref, L_ref, _ = oracle.attention_rows(spec, q, k, v, rows)
    compare(O_ref, L_ref, O.reshape(-1, 128)[rows], L.reshape(-1)[rows], "keys keylist 720p H2")


@pytest.mark.slow
def test_keylist_720p_full_size():
    spec = W.keylist_mask(seed=4)
    _sampled(spec, seed=4, rows_per_head=12)
