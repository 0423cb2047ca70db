"""The 256-mask sweep through the regime table, against the oracle (GPU).

Every member m = 0..255 of the seeded sweep (N = 32,760 tokens, H = 24,
d = 128, logical blocks of 32 x 32, 64 x 64, 128 x 128, 64 x 256 or 256 x 64,
density U(0.05, 0.60)) is planned with the regime the lookup table picks and
run at full size.  Parity is sampled: 2 seeded heads x 8 seeded 64-query blocks
of whole rows (1,024 rows) against ``oracle.attention_rows``, at the stated
tolerances.  The tile plan of one seeded head per mask, planned with the same
regime, is checked bit-exactly against the oracle's allowed set.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_tsr_gb300 as tsr
import oracle
import workloads as W
from test_gpu_parity import check_coverage, compare

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N, H, D = 32760, 24, 128


@pytest.fixture(scope="module")
def inputs():
    tsr.build()
    tsr.lib()
    q, k, v = W.qkv(1, H, N, D, seed=10)
    return (q, k, v), tuple(x.cuda() for x in (q, k, v))


def sampled_rows(m: int):
    """Rows (b*H + h)*N + i of 2 seeded heads x 8 seeded 64-query blocks (the
    last block is cut at N), and the first sampled head."""
    r = np.random.Generator(np.random.PCG64(5000 + m))
    heads = r.choice(H, size=2, replace=False)
    blocks = r.choice(-(-N // 64), size=8, replace=False)
    rows = []
    for h in heads:
        for b in blocks:
            i = b * 64 + np.arange(64)
            rows.append(h * N + i[i < N])
    return np.concatenate(rows), int(heads[0])


def regime_opts(st):
    return {"bn": st["bn"], "stages": st["stages"], "ctas_per_sm": st["ctas_per_sm"],
            "orient": st["orient"]}


@pytest.mark.parametrize("chunk", range(8))
def test_sweep_members_sampled_parity_and_coverage(inputs, chunk):
    (q, k, v), (qd, kd, vd) = inputs
    out = torch.empty_like(qd)
    lse = torch.empty((1, H, N), dtype=torch.float32, device="cuda")
    picked = {}
    for m in range(32 * chunk, 32 * chunk + 32):
        spec = W.sweep_mask(m, H=H, N=N)
        mask = tsr.make_mask(spec.kind, 1, H, N, D, **W.mask_tensors(spec))
        plan = tsr.tsr_plan(mask)                       # the table's regime
        tsr.tsr_bsa_forward(qd, kd, vd, plan, out, lse)
        torch.cuda.synchronize()
        tsr.tsr_plan_device_status(plan)
        st = plan.stats()
        picked[m] = (spec.bq, spec.bk, st["bn"], st["stages"], st["ctas_per_sm"])
        rows, h = sampled_rows(m)
        O_ref, L_ref, _ = oracle.attention_rows(spec, q, k, v, rows)
        O = out.float().cpu().numpy().reshape(-1, D)[rows]
        L = lse.double().cpu().numpy().reshape(-1)[rows]
        compare(O_ref, L_ref, O, L, f"sweep member {m} ({spec.bq}x{spec.bk}, rho {spec.meta['rho']:.2f})")
        # coverage of one head, planned alone with the same regime
        one = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N, bq=spec.bq, bk=spec.bk,
                         blocks=np.ascontiguousarray(spec.blocks[:, h:h + 1]))
        plan1 = tsr.tsr_plan(tsr.make_mask(one.kind, 1, 1, N, D, **W.mask_tensors(one)),
                             regime_opts(st))
        check_coverage(one, plan1)
        plan1.destroy()
        plan.destroy()
    assert len(picked) == 32
