"""GPU parity of SVG head routing (tsr_svg_route) against the routing oracle.

Tolerance: the per-head error sums, divided by the dense norm sum, agree with
the fp64 oracle within 1e-4 + 1e-3 x the oracle's value (fp32 attention over up
to 32,760 keys).  The routing decision is integer output decided by floating
point: the GPU's head_kind must equal the argmin of its own sums, and the
oracle's decision wherever the two patterns' errors differ by more than 5%.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
from oracle import route as R
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def _samples(N, n, seed):
    return np.sort(np.random.Generator(np.random.PCG64(seed)).choice(N, size=n, replace=False))


def _check(q, k, v, F, S, samples, r=0):
    stats, kinds = tsr.tsr_svg_route(q.cuda(), k.cuda(), v.cuda(), F, S, samples, temporal_radius=r)
    torch.cuda.synchronize()
    stats = stats.cpu().numpy().astype(np.float64)
    kinds = kinds.cpu().numpy()
    ref, ref_kinds = R.route(q, k, v, F, S, samples, temporal_radius=r)
    rel = stats[..., :2] / ref[..., 2:3]
    rel_ref = ref[..., :2] / ref[..., 2:3]
    assert np.all(np.abs(rel - rel_ref) <= 1e-4 + 1e-3 * rel_ref), (rel, rel_ref)
    assert np.all(np.abs(stats[..., 2] - ref[..., 2]) <= 1e-3 * ref[..., 2])
    tot = stats.sum(axis=0)
    assert list(kinds) == [int(tot[h, 1] < tot[h, 0]) for h in range(q.shape[1])]
    tot_ref = ref.sum(axis=0)
    clear = np.abs(tot_ref[:, 1] - tot_ref[:, 0]) > 0.05 * np.maximum(tot_ref[:, 0], tot_ref[:, 1])
    assert np.array_equal(kinds[clear], ref_kinds[clear])
    return kinds


@pytest.mark.parametrize("d,r", [(128, 0), (128, 2), (64, 1)])
def test_route_random_heads(d, r):
    F, S = 16, 64
    q, k, v = W.qkv(2, 3, F * S, d, seed=40 + r)
    _check(q, k, v, F, S, _samples(F * S, 40, seed=d + r), r)


@pytest.mark.parametrize("d", [64, 128])
def test_route_structured_heads_then_attention(d):
    """Heads generated to be spatial or temporal are routed to that pattern; the
    routed head_kind (still on the device) drives an SVG plan whose output
    matches the oracle with those kinds."""
    F, S = 16, 48
    kinds_true = np.array([0, 1, 1, 0, 1, 0], np.int8)
    q, k, v = W.svg_routing_heads(1, kinds_true, F, S, d, seed=5)
    kinds = _check(q, k, v, F, S, _samples(F * S, 64, seed=3))
    assert list(kinds) == list(kinds_true)
    _, head_kind = tsr.tsr_svg_route(q.cuda(), k.cuda(), v.cuda(), F, S, _samples(F * S, 64, seed=3))
    spec = W.svg_mask(1, len(kinds_true), n_frames=F, frame_size=S, kinds=kinds_true)
    mt = W.mask_tensors(spec)
    mt["head_kind"] = head_kind
    mask = tsr.make_mask(spec.kind, 1, spec.H, spec.N, d, **mt)
    plan = tsr.tsr_plan(mask)
    out, lse = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attention(spec, q, k, v)
    O = out.float().cpu().numpy()
    assert np.abs(O - O_ref).max() <= 2e-2 and np.abs(O - O_ref).mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - L_ref).max() <= 1e-3 * max(1.0, np.abs(L_ref).max())


@pytest.mark.slow
def test_route_480p_shape():
    """21 frames of 1,560 tokens (N = 32,760), two spatial and two temporal heads
    built as such, 64 sampled rows."""
    F, S = 21, 1560
    kinds_true = np.array([0, 1, 0, 1], np.int8)
    q, k, v = W.svg_routing_heads(1, kinds_true, F, S, 128, seed=8)
    kinds = _check(q, k, v, F, S, _samples(F * S, 64, seed=8))
    assert list(kinds) == list(kinds_true)


def test_route_rejects_bad_arguments():
    q, k, v = (x.cuda() for x in W.qkv(1, 2, 256, 64, seed=1))
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_svg_route(q, k, v, 4, 64, [0, 256])          # row outside [0, N)
    assert e.value.status == 1
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_svg_route(q, k, v, 4, 64, list(range(256)) * 5)   # more than 1024 rows
    assert e.value.status == 2
    with pytest.raises(ValueError):
        tsr.tsr_svg_route(q, k, v, 4, 60, [0])               # N != n_frames * frame_size
