"""Host logic of bench.py's multi-rank path (one process per GPU, no data-path
collective): rank r runs heads [r*H/N, (r+1)*H/N) of the one request (or, with
--replicas, a whole request of its own); the job's step time is the slowest
rank's, and the value is the work of all ranks over that time.  Run with two
gloo ranks on the CPU, plus the per-step launch count claimed in the JSON line."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                   # rank 1 is the slow one
        dist.barrier()
        m = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, m, bench.whole_job_rate(1e12, m, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in got:
        assert m == 5.0
        # two ranks of 1e12 flops per 5 ms step: 400 TFLOP/s for the job
        assert rate == pytest.approx(400.0)


def test_one_rank_is_its_own_time():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(4e12, 2.0, 1) == pytest.approx(2000.0)


def test_launches_per_step_match_the_planner():
    """count, [logical count,] schedule, emit, attention; key lists: count,
    schedule, emit (+ a validation pass above 196,608 tokens), attention; no
    permutation kernels (SVG temporal heads on the tiles are permuted inside
    the loads; by spatial position they add the launch-list compaction and
    their own kernel); a split plan adds the unit cut."""
    assert bench.launches_per_step(W.tiny_block_mask(), {}) == 5
    assert bench.launches_per_step(W.tiny_block_mask(), {"kv_split": 2}) == 6
    assert bench.launches_per_step(W.segment_mask(1, 1, 1, 2048), {}) == 5
    assert bench.launches_per_step(W.svg_mask(1, 4, 4, 64), {"n_temporal_heads": 2}) == 4
    assert bench.launches_per_step(W.svg_mask(1, 4, 4, 64),
                                   {"n_temporal_heads": 2, "temporal_band": 1}) == 6
    kl = W.random_keylist(1, 1, 1, 1024, hi=10)
    assert bench.launches_per_step(kl, {}) == 4
    kl.N = 200000
    assert bench.launches_per_step(kl, {}) == 5


class _FakePlan:
    """A plan whose export is built by hand in the tsr_plan_export layout: an
    80-byte header (n_items at byte 48) and 32-byte items (bh, q_tile, begin,
    end, layout, 0, 0, 0)."""

    def __init__(self, items):
        hdr = np.zeros(80, np.uint8)
        hdr[:4] = np.frombuffer(b"TSRP", np.uint8)
        hdr[48:56] = np.frombuffer(np.int64(len(items)).tobytes(), np.uint8)
        self.buf = hdr.tobytes() + np.asarray(items, np.int32).reshape(-1, 8).tobytes()

    def export(self):
        return self.buf


def test_fill_counts_only_the_spatial_tiles_when_temporal_heads_run_apart():
    """With the SVG temporal heads on their own kernel, the fill is the spatial
    heads' allowed pairs over their tiles' elements (items of layout 0 from the
    export); temporal items (layout 1) are left out."""
    spec = W.svg_mask(1, 2, n_frames=4, frame_size=64, kinds=np.array([0, 1], np.int8))
    # head 0 spatial: 2 query tiles of 128 rows, 3 + 2 tiles of 64 keys;
    # head 1 temporal: 2 items, 7 tiles, ignored
    items = [[0, 0, 0, 3, 0, 0, 0, 0], [0, 1, 3, 5, 0, 0, 0, 0],
             [1, 0, 5, 9, 1, 0, 0, 0], [1, 1, 9, 12, 1, 0, 0, 0]]
    stats = {"temporal_band": 1, "bm": 128, "bn": 64, "n_entries": 12}
    allowed = 64 * 64 * (2 * 4 - 1)                     # S^2 (2F - 1) for the spatial head
    assert bench.fill_of(spec, stats, _FakePlan(items)) == pytest.approx(allowed / (5 * 128 * 64))
    # on the tiles every item counts
    stats = dict(stats, temporal_band=0)
    assert bench.fill_of(spec, stats, _FakePlan(items)) == pytest.approx(
        bench.allowed_pairs(spec) / (12 * 128 * 64))


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 24, 30])
def test_head_ranges_cover_every_head_once(world):
    H = 24
    seen = np.zeros(H, dtype=int)
    sizes = []
    for r in range(world):
        lo, hi = bench.head_range(H, world, r)
        assert 0 <= lo <= hi <= H
        seen[lo:hi] += 1
        sizes.append(hi - lo)
    assert np.all(seen == 1)
    assert max(sizes) - min(sizes) <= 1               # balanced to within one head
    if world <= H:
        assert min(sizes) >= 1


def _masks_for_split():
    return [W.video_block_mask(seed=5, B=2, H=6, N=1000),
            W.segment_mask(2, 2, 6, 900, lo=16, hi=100),
            W.svg_mask(2, 6, n_frames=4, frame_size=50, kinds=np.array([0, 1, 1, 0, 1, 0], np.int8)),
            W.random_keylist(3, 2, 6, 700, slice_m=64, lo=0, hi=200)]


def _reassemble(spec, parts):
    """Concatenate per-rank head slices back into one request."""
    out = {}
    if spec.blocks is not None:
        out["blocks"] = np.concatenate([p.blocks for p in parts], axis=1)
    if spec.head_kind is not None:
        out["head_kind"] = np.concatenate([p.head_kind for p in parts])
    if spec.indptr is not None:
        nqb = -(-spec.N // spec.slice_m)
        lists = [[] for _ in range(spec.B)]
        for p in parts:
            for b in range(spec.B):
                for row in range(b * p.H * nqb, (b + 1) * p.H * nqb):
                    lists[b].append(p.indices[p.indptr[row]:p.indptr[row + 1]])
        flat = [x for b in range(spec.B) for x in lists[b]]
        out["indptr"] = np.concatenate([[0], np.cumsum([len(x) for x in flat])])
        out["indices"] = np.concatenate(flat)
    return out


def _split_rank(rank: int, world: int, port: int, q) -> None:
    """One gloo rank: slice every mask form and Q, K, V to this rank's heads,
    gather all ranks' slices (plain arrays) and check that, put back in rank
    order, they equal the whole request.  Reports (rank, failures)."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bad = []
    try:
        specs = _masks_for_split()
        mine = []
        for spec in specs:
            lo, hi = bench.head_range(spec.H, world, rank)
            part = bench.slice_heads(spec, lo, hi)
            qkv = W.qkv(spec.B, spec.H, spec.N, 64, seed=9)
            mine.append((lo, hi, part, [x[:, lo:hi].contiguous().float().numpy() for x in qkv]))
        got = [None] * world
        dist.all_gather_object(got, mine)
        for i, spec in enumerate(specs):
            per = [got[r][i] for r in range(world)]
            if per[0][0] != 0 or per[-1][1] != spec.H or any(
                    per[r][1] != per[r + 1][0] for r in range(world - 1)):
                bad.append((i, "ranges"))
            parts = [x[2] for x in per]
            for key, val in _reassemble(spec, parts).items():
                if not np.array_equal(val, getattr(spec, key)):
                    bad.append((i, key))
            qkv = W.qkv(spec.B, spec.H, spec.N, 64, seed=9)
            for t in range(3):
                if not np.array_equal(np.concatenate([x[3][t] for x in per], axis=1),
                                      qkv[t].float().numpy()):
                    bad.append((i, "qkv", t))
    except Exception as e:                      # reported, not raised: the parent asserts
        bad.append(repr(e))
    finally:
        dist.destroy_process_group()
    q.put((rank, bad))


def test_two_gloo_ranks_split_heads_and_reassemble():
    """Two gloo ranks each slice every mask form (block grid, segments, SVG head
    kinds, key lists with rebased indptr) and Q, K, V to their heads; gathered,
    the slices in rank order equal the whole request."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = [q.get(timeout=180) for _ in range(2)]
    finally:
        for p in procs:
            p.join(30)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, bad in results:
        assert bad == [], (rank, bad)
