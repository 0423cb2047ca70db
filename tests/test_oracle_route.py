"""Pins of the routing oracle (oracle/route.py), CPU only.

  * K = 0 (every score equal): each pattern's output is the plain mean of V
    over its allowed keys, so the three error sums are computed here directly;
  * a temporal radius covering the frame makes the temporal pattern dense:
    zero temporal error;
  * an independent NumPy brute force (oracle/brute.py) of the three patterns;
  * heads built to be spatial or temporal are routed to that pattern.
"""
import numpy as np
import torch

from oracle import brute
from oracle import route as R
import workloads as W


def _f64(x):
    return x.float().double().numpy()


def test_zero_keys_reduce_to_means():
    B, H, F, S, d, r = 1, 2, 4, 24, 64, 2
    N = F * S
    q, _, v = W.qkv(B, H, N, d, seed=3)
    k = torch.zeros_like(q)
    samples = np.array([0, 5, S + 3, 2 * S, N - 1])
    stats, kinds = R.route(q, k, v, F, S, samples, temporal_radius=r)
    V = _f64(v)
    t = np.arange(N)
    want = np.zeros((B, H, 3))
    for b in range(B):
        for h in range(H):
            dense = V[b, h].mean(axis=0)
            for i in samples:
                sp = V[b, h][(t // S == i // S) | (t // S == 0)].mean(axis=0)
                tp = V[b, h][np.abs(t % S - i % S) <= r].mean(axis=0)
                want[b, h] += [((sp - dense) ** 2).sum(), ((tp - dense) ** 2).sum(),
                               (dense ** 2).sum()]
    assert np.abs(stats - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
    assert list(kinds) == [int(want[0, h, 1] < want[0, h, 0]) for h in range(H)]


def test_radius_covering_frame_has_no_temporal_error():
    F, S, d = 4, 16, 64
    q, k, v = W.qkv(1, 2, F * S, d, seed=5)
    stats, kinds = R.route(q, k, v, F, S, np.arange(0, F * S, 7), temporal_radius=S - 1)
    assert np.all(stats[..., 1] <= 1e-24)
    assert np.all(stats[..., 0] > 0) and np.all(kinds == 1)


def test_brute_force_agrees():
    F, S, d, r = 4, 20, 64, 1
    N = F * S
    q, k, v = W.qkv(2, 2, N, d, seed=9)
    samples = np.array([1, 19, 20, 47, 79])
    stats, _ = R.route(q, k, v, F, S, samples, temporal_radius=r)
    dense = W.MaskSpec(W.MASK_UNIFORM, 2, 2, N, bq=N, bk=N, blocks=np.ones((2, 2, 1, 1), np.uint8))
    sp = W.svg_mask(2, 2, n_frames=F, frame_size=S, kinds=np.zeros(2, np.int8))
    tp = W.svg_mask(2, 2, n_frames=F, frame_size=S, kinds=np.ones(2, np.int8), temporal_radius=r)
    O, _ = brute.attention(dense, q, k, v)
    Os, _ = brute.attention(sp, q, k, v)
    Ot, _ = brute.attention(tp, q, k, v)
    want = np.stack([((Os - O)[:, :, samples] ** 2).sum(axis=(2, 3)),
                     ((Ot - O)[:, :, samples] ** 2).sum(axis=(2, 3)),
                     (O[:, :, samples] ** 2).sum(axis=(2, 3))], axis=-1)
    assert np.abs(stats - want).max() <= 1e-10 * max(1.0, np.abs(want).max())


def test_structured_heads_are_routed_to_their_pattern():
    F, S, d = 8, 32, 64
    kinds = np.array([0, 1, 1, 0, 1], np.int8)
    q, k, v = W.svg_routing_heads(1, kinds, F, S, d, seed=11)
    samples = np.random.Generator(np.random.PCG64(4)).choice(F * S, size=24, replace=False)
    stats, routed = R.route(q, k, v, F, S, samples)
    assert list(routed) == list(kinds)
    rel = stats[0, :, :2] / stats[0, :, 2:3]
    for h, kd in enumerate(kinds):
        assert rel[h, kd] < 0.5 * rel[h, 1 - kd]
