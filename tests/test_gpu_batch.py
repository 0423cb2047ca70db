"""One launch over several requests of different shapes (tsr_bsa_forward_batch).

Each batched request must equal the same request run alone with the same
regime (bit for bit: same kernel arithmetic per tile) and the oracle within the
parity tolerances; mismatched batches are refused before any launch.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

OPTS = {"bn": 64, "stages": 2, "ctas_per_sm": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tsr.build()
    tsr.lib()


def _request(spec, d, seed, opts=OPTS):
    q, k, v = W.qkv(spec.B, spec.H, spec.N, d, seed)
    mask = tsr.make_mask(spec.kind, spec.B, spec.H, spec.N, d, **W.mask_tensors(spec))
    plan = tsr.tsr_plan(mask, opts)
    return spec, (q, k, v), plan


def _check(reqs, d):
    outs = tsr.tsr_bsa_forward_batch([(q.cuda(), k.cuda(), v.cuda(), plan)
                                      for _, (q, k, v), plan in reqs])
    torch.cuda.synchronize()
    tsr.tsr_plan_device_status(reqs[0][2])
    for (spec, (q, k, v), plan), (out, lse) in zip(reqs, outs):
        alone, lse_alone = tsr.tsr_bsa_forward(q.cuda(), k.cuda(), v.cuda(), plan)
        torch.cuda.synchronize()
        assert torch.equal(out, alone) and torch.equal(lse, lse_alone)
        O_ref, L_ref = oracle.attention(spec, q, k, v)
        O = out.float().cpu().numpy()
        fin = np.isfinite(L_ref)
        assert np.all(O[~fin] == 0) and np.all(lse.cpu().numpy()[~fin] == -np.inf)
        assert np.abs(O - O_ref)[fin].max() <= 2e-2 and np.abs(O - O_ref)[fin].mean() <= 2e-3


@pytest.mark.parametrize("d", [64, 128])
def test_mixed_shapes_and_mask_kinds(d):
    opts = OPTS if d == 128 else {"bn": 64, "stages": 3, "ctas_per_sm": 2}
    r = np.random.Generator(np.random.PCG64(3))
    blocks = (r.random((1, 2, 16, 16)) < 0.35).astype(np.uint8)
    reqs = [
        _request(W.MaskSpec(W.MASK_UNIFORM, 1, 2, 1000, bq=64, bk=64, blocks=blocks), d, 1, opts),
        _request(W.svg_mask(1, 3, n_frames=16, frame_size=41, kinds=np.array([1, 0, 1], np.int8)),
                 d, 2, opts),
        _request(W.segment_mask(4, 2, 1, 1500, lo=16, hi=300), d, 3, opts),
        _request(W.tiny_block_mask(seed=5, N=300), d, 4, opts),
    ]
    _check(reqs, d)


def test_key_list_requests():
    reqs = [_request(W.random_keylist(9, 1, 2, 900, slice_m=64, lo=0, hi=300), 128, 5),
            _request(W.random_keylist(10, 1, 1, 2048, slice_m=128, lo=1, hi=700), 128, 6)]
    _check(reqs, 128)


def test_batch_with_debug_checks():
    """The tile count of a batched launch is compared with all its plans."""
    opts = dict(OPTS, flags=tsr.PLAN_DEBUG_CHECKS)
    reqs = [_request(W.tiny_block_mask(seed=16, N=1024), 128, 16, opts),
            _request(W.svg_mask(1, 2, n_frames=16, frame_size=48, kinds=np.array([0, 1], np.int8)),
                     128, 17, opts)]
    _check(reqs, 128)


def test_single_request_batch_equals_forward():
    reqs = [_request(W.tiny_block_mask(seed=7, N=1024), 128, 7)]
    _check(reqs, 128)


def test_batch_refusals():
    a = _request(W.tiny_block_mask(seed=8, N=512), 128, 8)
    b = _request(W.tiny_block_mask(seed=9, N=512), 128, 9, opts={"bn": 128, "stages": 3})
    c = _request(W.random_keylist(11, 1, 1, 512, slice_m=64, lo=1, hi=100), 128, 10)
    req = lambda x: (x[1][0].cuda(), x[1][1].cuda(), x[1][2].cuda(), x[2])
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_bsa_forward_batch([req(a), req(b)])          # different regimes
    assert e.value.status == 2
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_bsa_forward_batch([req(a), req(c)])          # key lists with block masks
    assert e.value.status == 2
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_bsa_forward_batch([req(a), req(a)])          # one plan twice
    assert e.value.status == 1
    with pytest.raises(tsr.TsrError) as e:
        tsr.tsr_bsa_forward_batch([req(a)] * 17)              # too many
    assert e.value.status == 1
