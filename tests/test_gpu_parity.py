"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (bf16 output of fp32 arithmetic against fp64): max |dO| <= 2e-2 and
mean |dO| <= 2e-3 over the non-empty rows, |dlse| <= 1e-3 * max(1, |lse|),
rows with no allowed key exactly O = 0 and lse = -inf.  Plans are checked
bit-exactly against the oracle's allowed set by ``oracle.coverage``.
"""
import math

import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_REL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def run(spec, d, seed, opts=None, scale=1.0, qkv=None):
    """Plan and run on the GPU.  `scale` multiplies Q and K only (sharper
    softmax); V stays N(0, 1), the distribution the tolerances are stated for."""
    if qkv is None:
        q, k, v = W.qkv(spec.B, spec.H, spec.N, d, seed)
        if scale != 1.0:
            q = (q.float() * scale).to(torch.bfloat16)
            k = (k.float() * scale).to(torch.bfloat16)
    else:
        q, k, v = qkv
    mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, d, **W.mask_tensors(spec))
    plan = tsr.tsr_plan(mask, opts)
    out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
    torch.cuda.synchronize()
    tsr.tsr_plan_device_status(plan)
    return (q, k, v), plan, out.float().cpu().numpy(), lse.cpu().numpy().astype(np.float64)


def compare(O_ref, L_ref, O, L, where=""):
    O_ref = O_ref.reshape(-1, O_ref.shape[-1])
    O = O.reshape(-1, O.shape[-1])
    L_ref, L = L_ref.reshape(-1), L.reshape(-1)
    empty = ~np.isfinite(L_ref)
    assert np.all(L[empty] == -np.inf), f"{where}: empty rows must have lse = -inf"
    assert np.all(O[empty] == 0.0), f"{where}: empty rows must have O = 0"
    assert np.all(np.isfinite(L[~empty])), f"{where}: non-empty rows must have finite lse"
    if (~empty).any():
        d = np.abs(O[~empty] - O_ref[~empty])
        assert d.max() <= MAX_ABS, f"{where}: max |dO| = {d.max():.3e}"
        assert d.mean() <= MEAN_ABS, f"{where}: mean |dO| = {d.mean():.3e}"
        dl = np.abs(L[~empty] - L_ref[~empty]) / np.maximum(1.0, np.abs(L_ref[~empty]))
        assert dl.max() <= LSE_REL, f"{where}: lse rel err = {dl.max():.3e}"


def check_coverage(spec, plan):
    n, rep, st = oracle.coverage(spec, plan.export())
    assert n == 0, f"plan coverage failures: {rep}"
    assert st["covered"] == st["allowed"]
    return st


# ------------------------------------------------------------------ tiny config
def test_tiny_config_full_parity():
    spec = W.tiny_block_mask(seed=1)               # B=1 H=2 N=1024 d=64, 64x64 blocks
    (q, k, v), plan, O, L = run(spec, 64, seed=1)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "tiny")
    check_coverage(spec, plan)
    assert np.sum(~np.isfinite(L)) == 2 * 64       # one masked query block per head


UNIFORM_CASES = [
    # (N, H, d, bq, bk, p, opts)
    (1000, 2, 128, 64, 64, 0.3, None),
    (777, 1, 128, 32, 32, 0.4, {"bn": 64, "stages": 4, "ctas_per_sm": 1}),
    (1024, 2, 128, 128, 128, 0.5, {"bn": 128, "stages": 2}),
    (900, 1, 128, 64, 256, 0.5, {"bn": 64, "stages": 2, "ctas_per_sm": 2}),
    (900, 1, 128, 256, 64, 0.5, None),
    (1100, 2, 64, 64, 64, 0.3, {"bn": 128, "stages": 4}),
    (1100, 1, 64, 16, 48, 0.3, {"bn": 64, "stages": 4}),
    (1100, 1, 64, 64, 64, 0.3, {"bn": 64, "stages": 3, "ctas_per_sm": 2}),
    (200, 1, 128, 64, 64, 1.0, None),
    (129, 1, 64, 16, 16, 0.5, {"bn": 64, "stages": 4}),
]


@pytest.mark.parametrize("case", UNIFORM_CASES, ids=[str(i) for i in range(len(UNIFORM_CASES))])
def test_uniform_masks(case):
    N, H, d, bq, bk, p, opts = case
    r = np.random.Generator(np.random.PCG64(N + bq))
    blocks = (r.random((1, H, -(-N // bq), -(-N // bk))) < p).astype(np.uint8)
    if blocks.shape[2] > 2:
        blocks[0, 0, 2, :] = 0                       # a fully masked query block
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=bq, bk=bk, blocks=blocks)
    (q, k, v), plan, O, L = run(spec, d, seed=N, opts=opts, scale=1.5)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"uniform {case}")
    check_coverage(spec, plan)


def test_segments_mask():
    spec = W.segment_mask(3, 1, 2, 1500, lo=16, hi=300)
    (q, k, v), plan, O, L = run(spec, 128, seed=5)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "segments")
    check_coverage(spec, plan)


@pytest.mark.parametrize("d", [64, 128])
def test_svg_small(d):
    spec = W.svg_mask(1, 4, n_frames=16, frame_size=48, kinds=np.array([0, 1, 1, 0], np.int8))
    (q, k, v), plan, O, L = run(spec, d, seed=7)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "svg")
    st = check_coverage(spec, plan)
    assert plan.stats()["n_temporal_heads"] == 2
    assert st["allowed"] == 2 * 48 * 48 * 31 + 2 * 768 * 16


@pytest.mark.parametrize("opts,F,S", [(None, 16, 41), ({"bn": 128, "stages": 3}, 24, 27),
                                      ({"bn": 64, "stages": 2, "ctas_per_sm": 2}, 16, 41),
                                      ({"bn": 64, "stages": 3, "ctas_per_sm": 2}, 24, 27),
                                      (None, 13, 50), ({"bn": 128, "stages": 3}, 5, 130),
                                      ({"bn": 64, "stages": 2, "ctas_per_sm": 2}, 1, 700)])
def test_svg_ragged_temporal_gather(opts, F, S):
    """Temporal-major heads load Q, K and V rows through the inverse permutation
    inside the kernel; N = F x S leaves a ragged last query and key tile whose
    rows past N must neither be read as keys nor written as outputs.  Two
    batches and mixed head kinds put spatial (TMA) and temporal (gathered)
    items in one launch.  Frame counts below 16 (13, 5, 1) put more than 8
    temporal segments in a 128-token tile: those tiles are masked by the band
    rule, which has no segment limit.  TSR_PLAN_TEMPORAL_TILES keeps these
    radius-0 heads on the tiles."""
    d = 64 if opts and opts.get("stages") == 3 and opts.get("ctas_per_sm") == 2 else 128
    spec = W.svg_mask(2, 3, n_frames=F, frame_size=S, kinds=np.array([1, 0, 1], np.int8))
    opts = dict(opts or {}, flags=tsr.PLAN_TEMPORAL_TILES)
    (q, k, v), plan, O, L = run(spec, d, seed=21, opts=opts)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"svg ragged {opts}")
    check_coverage(spec, plan)
    assert plan.stats()["n_temporal_heads"] == 2
    assert plan.stats()["temporal_band"] == 0


@pytest.mark.parametrize("r,opts", [(1, None), (4, {"bn": 128, "stages": 3}),
                                     (2, {"bn": 64, "stages": 3, "ctas_per_sm": 2}), (40, None)])
def test_svg_temporal_radius(r, opts):
    """Temporal heads with a spatial radius: a band of (2r + 1) F-token
    segments in temporal-major order; r = 40 >= S - 1 makes those heads dense.
    N = 16 x 41 = 656 leaves ragged tiles."""
    d = 64 if opts and opts.get("ctas_per_sm") == 2 else 128
    spec = W.svg_mask(1, 3, n_frames=16, frame_size=41, kinds=np.array([1, 0, 1], np.int8),
                      temporal_radius=r)
    (q, k, v), plan, O, L = run(spec, d, seed=31 + r, opts=opts)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"svg radius {r}")
    st = check_coverage(spec, plan)
    F, S = 16, 41
    temporal = F * F * (S * (2 * r + 1) - r * (r + 1)) if r < S else (F * S) ** 2
    assert st["allowed"] == 2 * temporal + S * S * (2 * F - 1)


def test_q_zero_closed_form_on_gpu():
    """Q = 0: lse_i = ln |A_i| exactly in fp64; the GPU must reproduce the count
    of allowed keys, so a tile computed twice or skipped shows up here."""
    spec = W.tiny_block_mask(seed=4, N=1000)
    _, k, v = W.qkv(spec.B, spec.H, spec.N, 64, 9)
    q = torch.zeros_like(k)
    _, _, O, L = run(spec, 64, seed=0, qkv=(q, k, v))
    cnt = np.array([[len(oracle.row_keys(spec, 0, h, i)) for i in range(spec.N)]
                    for h in range(spec.H)])
    fin = cnt > 0
    assert np.all(np.isfinite(L[0][fin])) and np.all(L[0][~fin] == -np.inf)
    assert np.abs(L[0][fin] - np.log(cnt[fin])).max() <= 1e-5


def test_rescale_path_large_logits():
    """Large, growing logits force many running-maximum rescales."""
    spec = W.tiny_block_mask(seed=6, N=1024)
    q, k, v = W.qkv(1, 2, 1024, 64, 3)
    q = (q.float() * 4.0).to(torch.bfloat16)
    ramp = torch.linspace(0.1, 3.0, 1024).view(1, 1, -1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    _, _, O, L = run(spec, 64, seed=0, qkv=(q, k, v))
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "rescale")


def test_plan_reuse_and_lpt_off():
    spec = W.tiny_block_mask(seed=8, N=2048)
    q, k, v = W.qkv(1, 2, 2048, 128, 8)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    mask = tsr.make_mask(spec.kind, 1, 2, 2048, 128, **W.mask_tensors(spec))
    for opts in (None, {"flags": tsr.PLAN_NO_LPT}, {"flags": tsr.PLAN_SYNC_CHECK}):
        plan = tsr.tsr_plan(mask, opts)
        for _ in range(2):
            out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
            compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().double().numpy(), str(opts))
        tsr.tsr_plan_device_status(plan)


def test_temporal_permute_roundtrip_bit_exact():
    F, S, H = 21, 40, 3
    x = torch.randn(2, H, F * S, 128, device="cuda").to(torch.bfloat16)
    y = torch.zeros_like(x)
    z = torch.zeros_like(x)
    kinds = [1, 0, 1]
    tsr.tsr_temporal_permute(x, y, F, S, head_kind=kinds)
    tsr.tsr_temporal_permute(y, z, F, S, head_kind=kinds, inverse=True)
    torch.cuda.synchronize()
    for h, kd in enumerate(kinds):
        if kd:
            assert torch.equal(z[:, h], x[:, h])
            # t' = s*F + f holds token t = f*S + s
            perm = torch.tensor([(tp % F) * S + tp // F for tp in range(F * S)], device="cuda")
            assert torch.equal(y[:, h], x[:, h, perm])
        else:
            assert torch.count_nonzero(y[:, h]) == 0


def test_host_entry_point_matches_device_path():
    spec = W.tiny_block_mask(seed=2, N=1024)
    q, k, v = W.qkv(1, 2, 1024, 64, 2)
    # the host entry point does not split work items automatically
    _, _, O, L = run(spec, 64, seed=0, qkv=(q, k, v), opts={"kv_split": 1})
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((1, 2, 1024), dtype=torch.float32).pin_memory()
    tsr.tsr_attention_host(spec.kind, 1, 2, 1024, 64, q.pin_memory(), k.pin_memory(),
                           v.pin_memory(), out, lse, bq=64, bk=64, blocks=spec.blocks)
    assert np.array_equal(out.float().numpy(), O)
    assert np.array_equal(lse.double().numpy(), L)


# -------------------------------------------------------- full-size configs
def _sample_rows(spec, n_per_head, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    rows = []
    for bh in range(spec.B * spec.H):
        idx = np.concatenate([r.integers(0, spec.N, n_per_head - 2), [spec.N - 1, 0]])
        rows.append(bh * spec.N + idx)
    return np.concatenate(rows)


def _sampled_parity(spec, d, seed, opts=None, rows_per_head=24):
    (q, k, v), plan, O, L = run(spec, d, seed=seed, opts=opts)
    rows = _sample_rows(spec, rows_per_head, seed)
    O_ref, L_ref, _ = oracle.attention_rows(spec, q, k, v, rows)
    compare(O_ref, L_ref, O.reshape(-1, d)[rows], L.reshape(-1)[rows], spec.meta.get("workload", ""))
    return plan


@pytest.mark.slow
def test_video_480p_block_mask_full_size():
    spec = W.video_block_mask(seed=2)              # 24 heads x 32,760 tokens, 64x64 blocks
    plan = _sampled_parity(spec, 128, seed=2)
    check_coverage(spec, plan)


@pytest.mark.slow
def test_video_480p_block_mask_bn128():
    spec = W.video_block_mask(seed=2, H=4)
    _sampled_parity(spec, 128, seed=12, opts={"bn": 128, "stages": 3})


@pytest.mark.slow
@pytest.mark.parametrize("flags", [0, tsr.PLAN_TEMPORAL_TILES])
def test_svg_480p_full_size(flags):
    """Temporal heads by spatial position (the default), or on the tiles."""
    spec = W.svg_mask(1, 24, n_frames=21, frame_size=1560)
    plan = _sampled_parity(spec, 128, seed=3, opts={"flags": flags} if flags else None)
    st = plan.stats()
    assert st["n_temporal_heads"] == 12
    assert st["temporal_band"] == (0 if flags else 1)
    cov = check_coverage(spec, plan)                   # every head, every row, bit-exact
    assert cov["allowed"] == 12 * (99_777_600 + 687_960)


@pytest.mark.slow
@pytest.mark.parametrize("m", [0, 1, 2, 3])
def test_sweep_members(m):
    spec = W.sweep_mask(m, H=4)
    plan = _sampled_parity(spec, 128, seed=100 + m, rows_per_head=16)
    check_coverage(spec, plan)


def test_plan_update_across_masks():
    """One plan re-planned for masks of different density, block shape and kind
    (storage grows and is reused); every result and plan matches the oracle."""
    N, H, d = 1500, 2, 128
    q, k, v = W.qkv(1, H, N, d, 21)
    r = np.random.Generator(np.random.PCG64(21))
    specs = [
        W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=64, bk=64,
                   blocks=(r.random((1, H, 24, 24)) < 0.1).astype(np.uint8)),
        W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=32, bk=32,
                   blocks=(r.random((1, H, 47, 47)) < 0.7).astype(np.uint8)),
        W.segment_mask(9, 1, H, N, lo=16, hi=200),
        W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=128, bk=64,
                   blocks=(r.random((1, H, 12, 24)) < 0.3).astype(np.uint8)),
    ]
    plan = None
    for spec in specs:
        mask = tsr.make_mask(spec.kind, 1, H, N, d, **W.mask_tensors(spec))
        plan = tsr.tsr_plan(mask) if plan is None else plan.update(mask)
        out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        compare(O_ref, L_ref, out.float().cpu().numpy(), lse.cpu().double().numpy(), "update")
        check_coverage(spec, plan)
    tsr.tsr_plan_device_status(plan)


# ------------------------------------------------------- KEYLIST (gathered)
KEYLIST_CASES = [
    # (N, H, d, slice_m, lo, hi, opts)
    (1000, 2, 128, 64, 0, 400, None),
    (777, 2, 128, 64, 1, 777, {"bn": 128, "stages": 3, "ctas_per_sm": 1}),
    (1024, 1, 64, 128, 0, 300, None),
    (1100, 2, 64, 64, 5, 200, {"bn": 128, "stages": 4, "ctas_per_sm": 1}),
    (640, 1, 128, 128, 640, 640, None),          # every key listed: full gathered tiles
]


@pytest.mark.parametrize("case", KEYLIST_CASES, ids=[str(i) for i in range(len(KEYLIST_CASES))])
def test_keylist_masks(case):
    N, H, d, M, lo, hi, opts = case
    spec = W.random_keylist(N + M, 1, H, N, slice_m=M, lo=lo, hi=hi)
    (q, k, v), plan, O, L = run(spec, d, seed=N + 1, opts=opts)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, f"keylist {case}")
    st = check_coverage(spec, plan)
    assert plan.stats()["gathered"] == 1
    if lo == hi == N:
        assert st["full"] == st["tiles"]


def test_keylist_clustered_runs():
    """FG-Attn-shaped lists: clustered runs (Geometric lengths) covering 15% of keys."""
    spec = W.keylist_mask(seed=4, H=2, N=4096)
    (q, k, v), plan, O, L = run(spec, 128, seed=4)
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "keylist clustered")
    check_coverage(spec, plan)


def test_keylist_invalid_lists_rejected():
    spec = W.random_keylist(3, 1, 1, 512, slice_m=64, lo=4, hi=20)
    bad = spec.indices.copy()
    bad[2] = bad[1]                                  # a repeated key
    spec.indices = bad
    mask = tsr.make_mask(spec.kind, 1, 1, 512, 64, **W.mask_tensors(spec))
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_plan(mask)
    assert e.value.status == 1
    spec.indices = np.where(np.arange(len(bad)) == 0, 600, spec.indices).astype(np.int32)  # out of range
    mask = tsr.make_mask(spec.kind, 1, 1, 512, 64, **W.mask_tensors(spec))
    with pytest.raises(tsr.TsrError):
        tsr.tsr_plan(mask)
    # a negative key in the second list of a query tile, a decreasing indptr,
    # and an indptr that does not start at 0
    good = W.random_keylist(3, 1, 1, 512, slice_m=64, lo=4, hi=20)
    neg = good.indices.copy()
    neg[good.indptr[1]] = -1
    bad_ptr = good.indptr.copy()
    bad_ptr[3] = bad_ptr[2] - 1
    off_ptr = good.indptr.copy()
    off_ptr[0] = 1                                   # every offset stays inside the array
    for ind, ptr in ((neg, good.indptr), (good.indices, bad_ptr), (good.indices, off_ptr)):
        t = W.mask_tensors(good)
        t["indices"] = torch.as_tensor(np.asarray(ind, np.int32)).cuda()
        t["indptr"] = torch.as_tensor(np.asarray(ptr, np.int64)).cuda()
        with pytest.raises(tsr.TsrError) as e:
            tsr.tsr_plan(tsr.make_mask(good.kind, 1, 1, 512, 64, **t))
        assert e.value.status == 1
    # the valid lists still plan and run after the refusals
    (q, k, v), plan, O, L = run(good, 64, seed=4)
    O_ref, L_ref = oracle.attention(good, q, k, v)
    compare(O_ref, L_ref, O, L, "keylist after refusals")


@pytest.mark.slow
def test_keylist_720p_coverage_two_heads():
    spec = W.keylist_mask(seed=4, H=2)               # 75,600 tokens, 11,340 keys per block
    (q, k, v), plan, O, L = run(spec, 128, seed=40)
    check_coverage(spec, plan)
    rows = _sample_rows(spec, 32, 40)
    O_ref, L_ref, _ = oracle.attention_rows(spec, q, k, v, rows)
    compare(O_ref, L_ref, O.reshape(-1, 128)[rows], L.reshape(-1)[rows], "keylist 720p H2")


@pytest.mark.slow
def test_keylist_720p_full_size():
    spec = W.keylist_mask(seed=4)                     # 24 heads x 75,600 tokens
    _sampled_parity(spec, 128, seed=4, rows_per_head=12)


def test_host_entry_point_keylist():
    spec = W.random_keylist(8, 1, 2, 900, slice_m=64, lo=0, hi=300)
    q, k, v = W.qkv(1, 2, 900, 128, 8)
    _, _, O, L = run(spec, 128, seed=0, qkv=(q, k, v), opts={"kv_split": 1})
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((1, 2, 900), dtype=torch.float32).pin_memory()
    tsr.tsr_attention_host(spec.kind, 1, 2, 900, 128, q.pin_memory(), k.pin_memory(),
                           v.pin_memory(), out, lse, slice_m=64, indptr=spec.indptr,
                           indices=spec.indices)
    assert np.array_equal(out.float().numpy(), O)
    assert np.array_equal(lse.double().numpy(), L)


@pytest.mark.parametrize("which", ["uniform", "uniform_debug", "svg", "keylist"])
def test_host_entry_point_in_head_groups(which):
    """Heads are copied in, attended and copied out in groups (growing from one
    head, ending with two and one); with the regime forced the result is
    bit-identical to one device call over all heads.  The SVG case has B = 3, H = 3, so a group spans two
    batches and its head kinds come from the flattened (b, h) order; the
    key-list case rebases each group's slice of indptr.  Block masks and SVG
    take one plan over all heads and launch each group over its item range;
    with the debug checks (every plan checked on the device, every launch's
    tile count compared) and for key lists each group has its own plan."""
    opts = {"bn": 64, "stages": 2, "ctas_per_sm": 2, "kv_split": 1}
    if which == "uniform_debug":
        opts = dict(opts, flags=tsr.PLAN_DEBUG_CHECKS)
    if which in ("uniform", "uniform_debug"):
        spec = W.video_block_mask(seed=5, H=16)      # groups of 1, 2, 2, 2, 3, 3, 2, 1 heads
        kw = dict(bq=64, bk=64, blocks=spec.blocks)
    elif which == "svg":
        spec = W.svg_mask(3, 3, n_frames=21, frame_size=1560, kinds=np.array([1, 0, 1], np.int8))
        kw = dict(n_frames=21, frame_size=1560, head_kind=spec.head_kind)
    else:
        spec = W.keylist_mask(seed=6, H=4)
        kw = dict(slice_m=64, indptr=spec.indptr, indices=spec.indices)
    q, k, v = W.qkv(spec.B, spec.H, spec.N, 128, 17)
    _, _, O, L = run(spec, 128, seed=0, opts=opts, qkv=(q, k, v))
    out = torch.empty_like(q).pin_memory()
    lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
    for _ in range(2):      # the second call reuses the cached group plans
        tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, 128, q.pin_memory(),
                               k.pin_memory(), v.pin_memory(), out, lse, opts=opts, **kw)
        assert np.array_equal(out.float().numpy(), O)
        assert np.array_equal(lse.double().numpy(), L)


def test_host_entry_point_alternating_shapes():
    """Host calls that change shape and mask form from call to call: every
    call re-plans into (or replaces) the cached plans and re-zeroes the work
    counters of its head-group launches, so each result equals one device call
    over all heads bit for bit (regime forced).  The block-mask, segment and
    SVG calls take the one-plan path (one plan, one launch per head group over
    its item range); the key-list call plans group by group."""
    opts = {"bn": 64, "stages": 2, "ctas_per_sm": 2, "kv_split": 1}
    cases = [
        (W.video_block_mask(seed=31, H=12, N=16384), dict(bq=64, bk=64)),
        (W.segment_mask(32, 2, 5, 8000, lo=16, hi=300), {}),
        (W.svg_mask(2, 3, n_frames=8, frame_size=512, kinds=np.array([0, 1, 1], np.int8)),
         dict(n_frames=8, frame_size=512)),
        (W.video_block_mask(seed=33, H=12, N=16384), dict(bq=64, bk=64)),
        (W.keylist_mask(seed=34, H=9, N=8192), dict(slice_m=64)),
        (W.video_block_mask(seed=31, H=12, N=16384), dict(bq=64, bk=64)),
    ]
    for i, (spec, kw) in enumerate(cases):
        arrays = {k: getattr(spec, k) for k in ("blocks", "q_bounds", "k_bounds", "head_kind",
                                                "indptr", "indices")
                  if getattr(spec, k) is not None}
        q, k, v = W.qkv(spec.B, spec.H, spec.N, 128, 40 + i)
        _, _, O, L = run(spec, 128, seed=0, opts=opts, qkv=(q, k, v))
        out = torch.empty_like(q).pin_memory()
        lse = torch.empty((spec.B, spec.H, spec.N), dtype=torch.float32).pin_memory()
        tsr.tsr_attention_host(spec.kind, spec.B, spec.H, spec.N, 128, q.pin_memory(),
                               k.pin_memory(), v.pin_memory(), out, lse, opts=opts, **kw,
                               **arrays)
        assert np.array_equal(out.float().numpy(), O), f"call {i}"
        assert np.array_equal(lse.double().numpy(), L), f"call {i}"


@pytest.mark.parametrize("which", ["uniform", "segments", "svg", "keylist"])
def test_debug_checks_pass_on_valid_plans(which):
    """With TSR_PLAN_DEBUG_CHECKS every plan is checked index by index on the
    device and every launch's computed tile count is compared with the plan;
    valid plans of every mask form pass, and the results are unchanged."""
    if which == "uniform":
        spec = W.tiny_block_mask(seed=13, N=1000)
    elif which == "segments":
        spec = W.segment_mask(14, 1, 2, 1500, lo=16, hi=300)
    elif which == "svg":
        spec = W.svg_mask(2, 3, n_frames=16, frame_size=41, kinds=np.array([1, 0, 1], np.int8),
                          temporal_radius=1)
    else:
        spec = W.random_keylist(15, 1, 2, 900, slice_m=64, lo=0, hi=300)
    (q, k, v), plan, O, L = run(spec, 128, seed=13, opts={"flags": tsr.PLAN_DEBUG_CHECKS})
    _, _, O2, L2 = run(spec, 128, seed=13, qkv=(q, k, v))
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, 128, **W.mask_tensors(spec))
    plan.update(mask)                                   # re-plan: checked again
    out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
    torch.cuda.synchronize()
    assert np.array_equal(out.float().cpu().numpy(), O)


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection without a GPU fault: with the test-only stall flag the
    MMA issuer waits on a barrier nothing signals; the kernel gives up after its
    bound, reports TSR_ERR_TIMEOUT through the error word, and the next normal
    call on the same context is correct."""
    spec = W.tiny_block_mask(seed=12)
    q, k, v = W.qkv(1, 2, 1024, 64, 12)
    mask = tsr.make_mask(spec.kind, 1, 2, 1024, 64, **W.mask_tensors(spec))
    plan = tsr.tsr_plan(mask, {"flags": tsr.PLAN_TEST_STALL})
    tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_plan_device_status(plan)
    assert e.value.status == 5
    tsr.tsr_plan_device_status(plan)                 # the error word was cleared
    (q, k, v), plan2, O, L = run(spec, 64, seed=0, qkv=(q, k, v))
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    compare(O_ref, L_ref, O, L, "after timeout")
