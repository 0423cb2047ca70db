"""The seeded input generators produce the workloads the benchmark and the
parity tests claim: shapes, sizes, densities, list lengths and value
distributions (CPU only; these generators draw numbers and hold no attention
arithmetic)."""
import numpy as np
import pytest
import torch

import workloads as W


def test_qkv_is_seeded_standard_normal_bf16():
    q, k, v = W.qkv(1, 2, 4096, 64, seed=3)
    assert q.dtype == torch.bfloat16 and q.shape == (1, 2, 4096, 64)
    q2, _, _ = W.qkv(1, 2, 4096, 64, seed=3)
    assert torch.equal(q, q2)                        # same seed, same draw
    x = torch.cat([q.float().flatten(), k.float().flatten(), v.float().flatten()])
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    assert not torch.equal(q, k) and not torch.equal(k, v)


def test_video_block_mask_recipe():
    """480p layer: 21 frames x 30 x 52 latents, 64 x 64 logical blocks, per-head
    density in [0.10, 0.40], every block on the token diagonal kept."""
    spec = W.video_block_mask(seed=2, H=4)
    assert spec.N == 21 * 30 * 52 == 32760 and spec.bq == spec.bk == 64
    nb = W.cdiv(32760, 64)
    assert spec.blocks.shape == (1, 4, nb, nb) and spec.blocks.dtype == np.uint8
    dens = spec.blocks.reshape(4, -1).mean(axis=1)
    want = spec.meta["densities"].reshape(-1)
    assert np.all((want >= 0.10) & (want <= 0.40))
    assert np.all(np.abs(dens - want) < 0.01)        # Bernoulli draws around the target
    assert np.all(spec.blocks[0, :, np.arange(nb), np.arange(nb)] == 1)
    # banded: blocks near the diagonal are on more often than far ones
    i, j = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    near = spec.blocks[0][:, np.abs(i - j) <= 4].mean()
    far = spec.blocks[0][:, np.abs(i - j) >= 64].mean()
    assert near > 2 * far


def test_tiny_block_mask_has_empty_query_block_rows():
    spec = W.tiny_block_mask(seed=1)
    blocks = spec.blocks[0]
    assert spec.N == 1024 and blocks.shape == (2, 16, 16)
    assert all((blocks[h].sum(axis=1) == 0).sum() == 1 for h in range(2))


@pytest.mark.parametrize("m", [0, 1, 2, 3, 7])
def test_sweep_members(m):
    spec = W.sweep_mask(m, H=2)
    assert (spec.bq, spec.bk) in W.SWEEP_SHAPES
    assert 0.05 <= spec.meta["rho"] <= 0.60
    assert spec.blocks.shape == (1, 2, W.cdiv(spec.N, spec.bq), W.cdiv(spec.N, spec.bk))
    assert np.all(np.abs(spec.meta["densities"] / spec.meta["rho"] - 1.0) <= 0.2 + 1e-12)


def test_svg_mask_recipe():
    spec = W.svg_mask()
    assert spec.N == 21 * 1560 and spec.n_frames == 21 and spec.frame_size == 1560
    assert list(spec.head_kind) == [W.HEAD_SPATIAL] * 12 + [W.HEAD_TEMPORAL] * 12


def test_keylist_mask_recipe():
    """720p: 21 x 45 x 80 = 75,600 tokens, 64-query blocks, each listing exactly
    ceil(0.15 N) = 11,340 sorted, unique keys in [0, N), built from runs."""
    spec = W.keylist_mask(seed=4, H=1)
    N = spec.N
    assert N == 21 * 45 * 80 == 75600 and spec.slice_m == 64
    nqb = W.cdiv(N, 64)
    assert spec.indptr.shape == (nqb + 1,) and spec.indptr[0] == 0
    lens = np.diff(spec.indptr)
    assert np.all(lens == 11340) and spec.meta["target"] == 11340
    for b in (0, 1, nqb // 2, nqb - 1):
        keys = spec.indices[spec.indptr[b]:spec.indptr[b + 1]]
        assert np.all(np.diff(keys) > 0) and keys[0] >= 0 and keys[-1] < N
        # clustered: mean run of consecutive keys well above 1 (mean run 8 drawn)
        runs = np.split(keys, np.nonzero(np.diff(keys) != 1)[0] + 1)
        assert np.mean([len(r) for r in runs]) > 4


def test_random_keylist_allows_empty_lists():
    spec = W.random_keylist(9, 1, 2, 900, slice_m=64, lo=0, hi=300)
    lens = np.diff(spec.indptr)
    assert lens.min() >= 0 and lens.max() <= 300
    assert np.all(spec.indices >= 0) and np.all(spec.indices < 900)


def test_segment_mask_bounds():
    spec = W.segment_mask(32, 2, 5, 8000, lo=16, hi=300)
    for bd in (spec.q_bounds, spec.k_bounds):
        assert bd[0] == 0 and bd[-1] == 8000 and np.all(np.diff(bd) > 0)
        assert np.all(np.diff(bd)[:-1] >= 16) and np.all(np.diff(bd) <= 300)
    assert spec.blocks.shape == (2, 5, len(spec.q_bounds) - 1, len(spec.k_bounds) - 1)
