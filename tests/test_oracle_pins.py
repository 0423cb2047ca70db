"""Pins of the CPU oracle to things other than itself (CPU only).

The pages print no worked example, so the oracle is pinned by:
  * an independent dense brute force (``oracle/brute.py``) on tiny inputs of every
    mask form;
  * a library routine: with an all-ones mask the result is plain dense attention
    (``torch.nn.functional.scaled_dot_product_attention`` in fp64);
  * block-diagonal masks equal independent per-block dense attention;
  * closed forms: Q = 0 gives lse = ln|A_i| and O = mean of the allowed values
    (this pins the allowed-set size of each mask form); one allowed key gives
    O = v_j and lse = s_ij; constant V gives O = c; a two-key case by hand;
  * counted densities of the SVG patterns;
  * permutation invariance of the temporal pattern (the temporal-major reading);
  * the empty-row rule (O = 0, lse = -inf exactly);
  * probabilities of a row summing to one and reproducing O.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads as W


def _qkv(B, H, N, d, seed, scale=1.0):
    return W.qkv(B, H, N, d, seed, scale)


def _masks_small(N=200, H=2):
    """One small mask of every form (N not a multiple of the block sizes)."""
    out = []
    r = np.random.Generator(np.random.PCG64(7))
    for bq, bk in ((32, 32), (64, 64), (16, 48), (64, 16)):
        nqb, nkb = -(-N // bq), -(-N // bk)
        blk = (r.random((1, H, nqb, nkb)) < 0.4).astype(np.uint8)
        blk[0, 0, 1, :] = 0          # a fully masked query block
        out.append(W.MaskSpec(W.MASK_UNIFORM, 1, H, N, bq=bq, bk=bk, blocks=blk))
    out.append(W.segment_mask(3, 1, H, N, lo=16, hi=60))
    out.append(W.svg_mask(1, H, n_frames=5, frame_size=N // 5, kinds=np.array([0, 1][:H], np.int8)))
    out.append(W.random_keylist(5, 1, H, N, slice_m=64, lo=0, hi=N // 2))
    out.append(W.random_keylist(6, 1, H, N, slice_m=128, lo=1, hi=N))
    out.append(W.svg_mask(1, H, n_frames=5, frame_size=N // 5, kinds=np.array([1, 0][:H], np.int8),
                          temporal_radius=3))
    return out


@pytest.mark.parametrize("idx", range(9))
@pytest.mark.parametrize("d", [64, 128])
def test_brute_force_agrees(idx, d):
    spec = _masks_small()[idx]
    q, k, v = _qkv(spec.B, spec.H, spec.N, d, seed=idx + 11)
    O, L = oracle.attention(spec, q, k, v)
    Ob, Lb = brute.attention(spec, q, k, v)
    fin = np.isfinite(Lb)
    assert np.array_equal(fin, np.isfinite(L))
    assert np.all(L[~fin] == -np.inf)
    assert np.abs(O - Ob).max() <= 1e-12
    assert np.abs(L[fin] - Lb[fin]).max() <= 1e-12
    assert np.all(O[~fin] == 0.0)


def test_all_ones_is_dense_attention():
    B, H, N, d = 1, 2, 192, 64
    q, k, v = _qkv(B, H, N, d, seed=21)
    spec = W.MaskSpec(W.MASK_UNIFORM, B, H, N, bq=64, bk=64,
                      blocks=np.ones((B, H, 3, 3), np.uint8))
    O, L = oracle.attention(spec, q, k, v)
    qd, kd, vd = (x.double() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd)
    assert np.abs(O - ref.numpy()).max() <= 1e-12
    lse_ref = torch.logsumexp(qd @ kd.transpose(-1, -2) / math.sqrt(d), dim=-1)
    assert np.abs(L - lse_ref.numpy()).max() <= 1e-12


def test_block_diagonal_is_per_block_attention():
    B, H, N, d, blk = 1, 1, 250, 64, 64
    q, k, v = _qkv(B, H, N, d, seed=22)
    nb = -(-N // blk)
    spec = W.MaskSpec(W.MASK_UNIFORM, B, H, N, bq=blk, bk=blk,
                      blocks=np.eye(nb, dtype=np.uint8)[None, None])
    O, _ = oracle.attention(spec, q, k, v)
    for s in range(0, N, blk):
        e = min(N, s + blk)
        sl = [x[:, :, s:e].double() for x in (q, k, v)]
        ref = torch.nn.functional.scaled_dot_product_attention(*sl)
        assert np.abs(O[:, :, s:e] - ref.numpy()).max() <= 1e-12


@pytest.mark.parametrize("idx", range(8))
def test_q_zero_closed_form(idx):
    """Q = 0: every allowed logit is 0, so lse_i = ln|A_i| and O_i = mean v_j."""
    spec = _masks_small()[idx]
    d = 64
    _, k, v = _qkv(spec.B, spec.H, spec.N, d, seed=31 + idx)
    q = torch.zeros_like(k)
    O, L = oracle.attention(spec, q, k, v)
    vd = brute.bf16_to_f64(oracle.as_u16(v))
    for h in range(spec.H):
        for i in range(0, spec.N, 7):
            keys = oracle.row_keys(spec, 0, h, i)
            if len(keys) == 0:
                assert L[0, h, i] == -np.inf and np.all(O[0, h, i] == 0)
                continue
            assert abs(L[0, h, i] - math.log(len(keys))) <= 1e-12
            assert np.abs(O[0, h, i] - vd[0, h, keys].mean(axis=0)).max() <= 1e-12


def test_uniform_row_counts_closed_form():
    """|A_i| = sum over allowed key blocks of the block width, truncated at N."""
    N, bq, bk = 300, 64, 48
    r = np.random.Generator(np.random.PCG64(3))
    blk = (r.random((1, 1, -(-N // bq), -(-N // bk))) < 0.5).astype(np.uint8)
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=bq, bk=bk, blocks=blk)
    widths = np.array([min(bk, N - c * bk) for c in range(blk.shape[3])])
    for i in range(N):
        assert len(oracle.row_keys(spec, 0, 0, i)) == int((blk[0, 0, i // bq] * widths).sum())
    assert oracle.count_allowed(spec)[0] == sum(
        int((blk[0, 0, i // bq] * widths).sum()) for i in range(N))


@pytest.mark.parametrize("F,S", [(21, 1560), (5, 40), (16, 17)])
def test_svg_counted_densities(F, S):
    """Spatial: frame 0 rows see S keys, other rows 2S, so |E| = S^2 (2F - 1);
    temporal: every row sees F keys, |E| = N F."""
    spec = W.svg_mask(1, 2, n_frames=F, frame_size=S, kinds=np.array([0, 1], np.int8))
    per = oracle.count_allowed(spec)
    assert per[0] == S * S * (2 * F - 1)
    assert per[1] == F * S * F
    if (F, S) == (21, 1560):
        assert per[0] == 99_777_600 and per[1] == 687_960


@pytest.mark.parametrize("F,S,r", [(21, 1560, 1), (5, 40, 3), (16, 17, 16), (4, 10, 25)])
def test_svg_temporal_radius_counted(F, S, r):
    """Temporal head with radius r: a row with spatial index s sees F keys for
    each index in [max(0, s - r), min(S - 1, s + r)], so summed over the S
    indices |E| = F^2 (S (2r + 1) - r (r + 1)) while r < S, and N^2 beyond."""
    spec = W.svg_mask(1, 1, n_frames=F, frame_size=S, kinds=np.array([1], np.int8),
                      temporal_radius=r)
    per = oracle.count_allowed(spec)
    want = F * F * (S * (2 * r + 1) - r * (r + 1)) if r < S else (F * S) ** 2
    assert per[0] == want
    for i in (0, S - 1, S // 2, F * S - 1):
        s_i = i % S
        assert len(oracle.row_keys(spec, 0, 0, i)) == F * (min(S - 1, s_i + r) - max(0, s_i - r) + 1)


def test_temporal_radius_covering_frame_is_dense():
    """r >= S - 1 allows every key: dense attention (library fp64 routine)."""
    F, S, d = 4, 24, 64
    N = F * S
    q, k, v = _qkv(1, 1, N, d, seed=23)
    spec = W.svg_mask(1, 1, n_frames=F, frame_size=S, kinds=np.array([1], np.int8),
                      temporal_radius=S - 1)
    O, L = oracle.attention(spec, q, k, v)
    qd, kd, vd = (x.double() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd)
    assert np.abs(O - ref.numpy()).max() <= 1e-12


def test_temporal_radius_is_a_band_in_temporal_major_order():
    """In temporal-major order t' = s F + f, the radius-r temporal pattern is
    the band |i - j| <= r of F x F blocks."""
    F, S, d, r = 6, 40, 64, 2
    N = F * S
    q, k, v = _qkv(1, 1, N, d, seed=73)
    spec = W.svg_mask(1, 1, n_frames=F, frame_size=S, kinds=np.array([1], np.int8),
                      temporal_radius=r)
    O, L = oracle.attention(spec, q, k, v)
    perm = np.array([(tp % F) * S + tp // F for tp in range(N)])
    qp, kp, vp = (x[:, :, perm].contiguous() for x in (q, k, v))
    idx = np.arange(S)
    blk = (np.abs(idx[:, None] - idx[None, :]) <= r).astype(np.uint8)[None, None]
    spec_p = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=F, bk=F, blocks=blk)
    Op, Lp = oracle.attention(spec_p, qp, kp, vp)
    assert np.abs(Op - O[:, :, perm]).max() <= 1e-12
    assert np.abs(Lp - L[:, :, perm]).max() <= 1e-12


def test_one_key_closed_form():
    """A single allowed key: O = v_j exactly and lse = q.k_j / sqrt(d)."""
    B, H, N, d, M = 1, 2, 256, 128, 64
    q, k, v = _qkv(B, H, N, d, seed=41)
    r = np.random.Generator(np.random.PCG64(9))
    nqb = N // M
    keys = r.integers(0, N, size=B * H * nqb).astype(np.int32)
    spec = W.MaskSpec(W.MASK_KEYLIST, B, H, N, slice_m=M,
                      indptr=np.arange(B * H * nqb + 1, dtype=np.int64), indices=keys)
    O, L = oracle.attention(spec, q, k, v)
    qd, kd, vd = (brute.bf16_to_f64(oracle.as_u16(x)) for x in (q, k, v))
    for h in range(H):
        for i in range(N):
            j = keys[h * nqb + i // M]
            assert np.array_equal(O[0, h, i], vd[0, h, j])
            assert abs(L[0, h, i] - qd[0, h, i] @ kd[0, h, j] / math.sqrt(d)) <= 1e-12


def test_constant_v_closed_form():
    spec = _masks_small()[1]
    q, k, _ = _qkv(spec.B, spec.H, spec.N, 64, seed=51, scale=3.0)
    v = torch.full_like(q, 1.5)
    O, L = oracle.attention(spec, q, k, v)
    fin = np.isfinite(L)
    assert np.abs(O[fin] - 1.5).max() <= 1e-12
    assert np.all(O[~fin] == 0)


def test_two_keys_by_hand():
    """d = 64, q = 8 e0, k0 = 0, k1 = e0: scores 0 and 1, so
    p = (1, e) / (1 + e), lse = ln(1 + e), O = (v0 + e v1) / (1 + e)."""
    B, H, N, d = 1, 1, 2, 64
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    q[0, 0, :, 0] = 8.0
    k[0, 0, 1, 0] = 1.0
    v[0, 0, 0, 0] = 1.0
    v[0, 0, 1, 0] = 2.0
    v[0, 0, 1, 5] = -0.5
    spec = W.MaskSpec(W.MASK_UNIFORM, B, H, N, bq=16, bk=16, blocks=np.ones((1, 1, 1, 1), np.uint8))
    O, L = oracle.attention(spec, q, k, v)
    e = math.e
    assert abs(L[0, 0, 0] - math.log(1 + e)) <= 1e-14
    assert abs(O[0, 0, 0, 0] - (1 + 2 * e) / (1 + e)) <= 1e-14
    assert abs(O[0, 0, 0, 5] - (-0.5 * e) / (1 + e)) <= 1e-14
    keys, probs, _, _ = oracle.probs_row(spec, q, k, v, 0, 0, 1)
    assert list(keys) == [0, 1]
    assert np.allclose(probs, [1 / (1 + e), e / (1 + e)], rtol=0, atol=1e-15)


@pytest.mark.parametrize("idx", [0, 4, 5, 6])
def test_probabilities_sum_to_one(idx):
    spec = _masks_small()[idx]
    q, k, v = _qkv(spec.B, spec.H, spec.N, 64, seed=61, scale=2.0)
    vd = brute.bf16_to_f64(oracle.as_u16(v))
    for h in range(spec.H):
        for i in (0, 3, spec.N // 2, spec.N - 1):
            keys, probs, out, lse = oracle.probs_row(spec, q, k, v, 0, h, i)
            if len(keys) == 0:
                assert lse == -np.inf and np.all(out == 0)
                continue
            assert abs(probs.sum() - 1.0) <= 1e-12
            assert np.abs(probs @ vd[0, h, keys] - out).max() <= 1e-12


def test_temporal_permutation_invariance():
    """The temporal pattern in frame-major order equals block-diagonal attention
    (blocks of F tokens) on the temporal-major permutation t' = s F + f."""
    F, S, d = 6, 40, 64
    N = F * S
    q, k, v = _qkv(1, 1, N, d, seed=71)
    spec = W.svg_mask(1, 1, n_frames=F, frame_size=S, kinds=np.array([1], np.int8))
    O, L = oracle.attention(spec, q, k, v)
    # t' = s*F + f holds token t = f*S + s
    perm = np.array([(tp % F) * S + tp // F for tp in range(N)])
    qp, kp, vp = (x[:, :, perm].contiguous() for x in (q, k, v))
    blk = np.eye(S, dtype=np.uint8)[None, None]
    spec_p = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=F, bk=F, blocks=blk)
    Op, Lp = oracle.attention(spec_p, qp, kp, vp)
    assert np.abs(Op - O[:, :, perm]).max() <= 1e-12
    assert np.abs(Lp - L[:, :, perm]).max() <= 1e-12


def test_empty_rows_exact():
    spec = W.tiny_block_mask(seed=1, N=512)
    q, k, v = _qkv(spec.B, spec.H, spec.N, 64, seed=81)
    O, L = oracle.attention(spec, q, k, v)
    for h in range(spec.H):
        empty = np.nonzero(spec.blocks[0, h].sum(axis=1) == 0)[0]
        assert len(empty) == 1
        rows = slice(empty[0] * 64, (empty[0] + 1) * 64)
        assert np.all(L[0, h, rows] == -np.inf)
        assert np.all(O[0, h, rows] == 0.0)
    assert np.isfinite(L).sum() == spec.H * (512 - 64)


def test_rows_api_matches_full():
    spec = _masks_small()[6]
    q, k, v = _qkv(spec.B, spec.H, spec.N, 64, seed=91)
    O, L = oracle.attention(spec, q, k, v)
    rows = np.array([0, 5, spec.N + 3, 2 * spec.N - 1])
    Or, Lr, cnt = oracle.attention_rows(spec, q, k, v, rows)
    flatO, flatL = O.reshape(-1, 64), L.reshape(-1)
    assert np.array_equal(Or, flatO[rows]) and np.array_equal(Lr, flatL[rows])
    for r, c in zip(rows, cnt):
        assert c == len(oracle.row_keys(spec, 0, r // spec.N, r % spec.N))


def test_invalid_keylist_rejected():
    spec = W.random_keylist(5, 1, 1, 128, slice_m=64, lo=3, hi=10)
    bad = spec.indices.copy()
    bad[1] = bad[0]                      # a repeated key
    spec.indices = bad
    q, k, v = _qkv(1, 1, 128, 64, seed=1)
    with pytest.raises(ValueError):
        oracle.attention(spec, q, k, v)


def test_generators_are_seeded():
    a = W.video_block_mask(seed=2, H=2, N=2048)
    b = W.video_block_mask(seed=2, H=2, N=2048)
    assert np.array_equal(a.blocks, b.blocks)
    r1 = W.clustered_keys(1000, 150, np.random.Generator(np.random.PCG64(1)))
    r2 = W.clustered_keys(1000, 150, np.random.Generator(np.random.PCG64(1)))
    assert np.array_equal(r1, r2) and len(r1) == 150 and np.all(np.diff(r1) > 0)
    q1, _, _ = W.qkv(1, 1, 16, 64, seed=3)
    q2, _, _ = W.qkv(1, 1, 16, 64, seed=3)
    assert torch.equal(q1, q2)
