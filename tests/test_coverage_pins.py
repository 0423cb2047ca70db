"""Pins of the plan checker ``oracle.coverage`` (``oracle/coverage.c``), CPU only.

Every claim that a GPU plan covers exactly the oracle's allowed set rests on
this checker, so it is pinned here against tile plans written out by hand in
the export layout of ``include/tsr.h`` (header, items, entries, descriptors,
gathered keys, head layouts), not produced by the library.  For each form of
boundary descriptor (grid, list, band) and for temporal-major items, a correct
hand-built plan must pass with no failure, and the same plan with one planted
mistake must fail with the code that names the mistake:

  1 an allowed pair no tile computes      2 a computed pair the mask forbids
  3 a pair computed twice                 4 a "full" tile over a forbidden pair
  5 a "boundary" tile that is all allowed 6 a kept tile that computes nothing
  7 a query tile with no item, or two     8 an item or entry out of range

The grid descriptor's bit index (row segment * 8 + column segment) is pinned
by an asymmetric case whose transpose is a different element set, and the
band and list decodes by off-by-one radii and single flipped bits.
"""
import struct

import numpy as np
import pytest

import oracle
import workloads as W

HDR = struct.Struct("<4s11i4q")          # 80 bytes
ITEM = struct.Struct("<8i")              # 32 bytes
ENTRY = struct.Struct("<2i")             # 8 bytes
GRID = struct.Struct("<BB8s9s5sQ")       # 32 bytes
LIST = struct.Struct("<8I")              # 32 bytes
assert HDR.size == 80 and ITEM.size == 32 and GRID.size == 32 and LIST.size == 32


def grid(r_start, c_start, bits):
    """Grid-form descriptor: row segments start at r_start, column segments at
    c_start[:-1] (c_start[-1] = first out-of-range column), allowed cells set in
    `bits` as (row segment, column segment) pairs."""
    n_r, n_c = len(r_start), len(c_start) - 1
    b = 0
    for r, c in bits:
        b |= 1 << (r * 8 + c)
    return GRID.pack(n_r, n_c, bytes(r_start).ljust(8, b"\0"), bytes(c_start).ljust(9, b"\0"),
                     b"\0" * 5, b)


def band(F, R):
    return GRID.pack(0, 0, b"\0" * 8, b"\0" * 9, b"\0" * 5, (F << 32) | R)


def colmask(seg_bits):
    """List-form descriptor: seg_bits[r] = allowed columns of row segment r."""
    words = [0] * 8
    for r, cols in enumerate(seg_bits):
        for c in cols:
            words[r * 4 + c // 32] |= 1 << (c % 32)
    return LIST.pack(*words)


def export(B, H, N, d, bm, bn, items, entries, descs, gidx=(), head_layout=None, gathered=0,
           n_frames=0, frame_size=0, slice_m=0):
    hl = bytes(head_layout if head_layout is not None else [0] * H)
    out = [HDR.pack(b"TSRP", 1, B, H, N, d, bm, bn, gathered, n_frames, frame_size, slice_m,
                    len(items), len(entries), len(descs), len(gidx))]
    out += [ITEM.pack(*(list(it) + [0] * (8 - len(it)))) for it in items]
    out += [ENTRY.pack(*e) for e in entries]
    out += list(descs)
    out += [struct.pack("<i", g) for g in gidx]
    out.append(hl)
    return b"".join(out)


def codes(spec, buf):
    n, rep, _ = oracle.coverage(spec, buf, nthreads=2, max_report=1 << 16)
    assert n <= 1 << 16
    return n, {r[0] for r in rep}


# ---------------------------------------------------------------------------
# Grid form: UNIFORM 64 x 64 blocks, N = 200 (ragged last block of 8 tokens),
# physical tiles of 128 query rows x 64 keys.
BLOCKS = np.array([[1, 0, 1, 0],
                   [1, 1, 0, 0],
                   [0, 0, 0, 0],          # an empty query block
                   [0, 1, 0, 1]], np.uint8)
N_G = 200
SPEC_G = W.MaskSpec(W.MASK_UNIFORM, 1, 1, N_G, bq=64, bk=64, blocks=BLOCKS[None, None])


def grid_plan(items=None, entries=None, descs=None):
    """The exact plan of SPEC_G, written by hand from the block grid:
    query tile 0 (rows 0..127 = blocks 0, 1) against key tiles 0 (both blocks
    allowed: full), 1 (only block 1) and 2 (only block 0); key tile 3 is
    empty for it.  Query tile 1 (rows 128..199 = block 2 and the 8 rows of
    block 3) against key tile 1 (block 3 only) and key tile 3 (block 3, whose
    last 8 keys 192..199 are the only ones in range)."""
    d = [grid([0, 64], [0, 64], [(1, 0)]),          # kt 1 for qt 0
         grid([0, 64], [0, 64], [(0, 0)]),          # kt 2 for qt 0
         grid([0, 64], [0, 64], [(1, 0)]),          # kt 1 for qt 1
         grid([0, 64], [0, 8], [(1, 0)])]           # kt 3 for qt 1: 8 keys in range
    e = [(0, -1), (64, 0), (128, 1), (64, 2), (192, 3)]
    it = [(0, 0, 0, 3), (0, 1, 3, 5)]
    return export(1, 1, N_G, 64, 128, 64, items if items is not None else it,
                  entries if entries is not None else e, descs if descs is not None else d)


def test_hand_built_grid_plan_is_exact():
    n, rep, st = oracle.coverage(SPEC_G, grid_plan())
    assert n == 0, rep
    allowed = sum(len(oracle.row_keys(SPEC_G, 0, 0, i)) for i in range(N_G))
    assert st["allowed"] == st["covered"] == allowed
    assert st["tiles"] == 5 and st["full"] == 1 and st["boundary"] == 4


def test_dropped_tile_is_code_1():
    e = [(0, -1), (128, 1), (64, 2), (192, 3)]
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 2), (0, 1, 2, 4)], entries=e))
    assert n > 0 and c == {1}


def test_extra_pair_is_code_2():
    d = [grid([0, 64], [0, 64], [(0, 0), (1, 0)]),  # block (0, 1) is not allowed
         grid([0, 64], [0, 64], [(0, 0)]), grid([0, 64], [0, 64], [(1, 0)]),
         grid([0, 64], [0, 8], [(1, 0)])]
    n, c = codes(SPEC_G, grid_plan(descs=d))
    assert n > 0 and 2 in c and 1 not in c


def test_duplicated_tile_is_code_3():
    e = [(0, -1), (0, -1), (64, 0), (128, 1), (64, 2), (192, 3)]
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 4), (0, 1, 4, 6)], entries=e))
    assert n > 0 and c == {3}


def test_full_tile_over_masked_pair_is_code_4():
    e = [(0, -1), (64, -1), (128, 1), (64, 2), (192, 3)]   # kt 1 of qt 0 marked full
    n, c = codes(SPEC_G, grid_plan(entries=e))
    assert n > 0 and 4 in c


def test_all_allowed_boundary_tile_is_code_5():
    d = [grid([0, 64], [0, 64], [(1, 0)]), grid([0, 64], [0, 64], [(0, 0)]),
         grid([0, 64], [0, 64], [(1, 0)]), grid([0, 64], [0, 8], [(1, 0)]),
         grid([0, 64], [0, 64], [(0, 0), (1, 0)])]     # kt 0 of qt 0 as a boundary tile
    e = [(0, 4), (64, 0), (128, 1), (64, 2), (192, 3)]
    n, c = codes(SPEC_G, grid_plan(entries=e, descs=d))
    assert n > 0 and c == {5}


def test_kept_empty_tile_is_code_6():
    d = [grid([0, 64], [0, 64], [(1, 0)]), grid([0, 64], [0, 64], [(0, 0)]),
         grid([0, 64], [0, 64], [(1, 0)]), grid([0, 64], [0, 8], [(1, 0)]),
         grid([0, 64], [0, 8], [])]                      # kt 3 of qt 0: nothing selected
    e = [(0, -1), (64, 0), (128, 1), (192, 4), (64, 2), (192, 3)]
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 4), (0, 1, 4, 6)], entries=e, descs=d))
    assert n > 0 and c == {6}


def test_missing_or_repeated_query_tile_is_code_7():
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 3)]))
    assert n > 0 and c == {7}
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 3), (0, 0, 0, 3), (0, 1, 3, 5)]))
    assert n > 0 and c == {7}


def test_out_of_range_entry_or_item_is_code_8():
    e = [(0, -1), (64, 0), (128, 1), (64, 2), (400, 3)]    # key start past N
    n, c = codes(SPEC_G, grid_plan(entries=e))
    assert n > 0 and 8 in c
    e = [(0, -1), (64, 9), (128, 1), (64, 2), (192, 3)]    # descriptor index past n_desc
    n, c = codes(SPEC_G, grid_plan(entries=e))
    assert n > 0 and 8 in c
    n, c = codes(SPEC_G, grid_plan(items=[(0, 0, 0, 3), (0, 1, 3, 9)]))   # end past n_entries
    assert n > 0 and 8 in c


def test_grid_bit_index_is_row_times_8_plus_column():
    """Blocks of 64 query rows x 32 keys; in the tile (rows 0..127, keys 0..63)
    only (row segment 0, column segment 1) is allowed, i.e. bit 0*8 + 1.  A
    checker that read bit c*8 + r would see (row segment 1, column segment 0)."""
    blocks = np.zeros((1, 1, 2, 4), np.uint8)      # N = 128: 2 query x 4 key blocks
    blocks[0, 0, 0, 1] = 1
    spec = W.MaskSpec(W.MASK_UNIFORM, 1, 1, 128, bq=64, bk=32, blocks=blocks)
    good = export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 1)], [(0, 0)],
                  [grid([0, 64], [0, 32, 64], [(0, 1)])])
    n, rep, st = oracle.coverage(spec, good)
    assert n == 0, rep
    assert st["covered"] == 64 * 32
    swapped = export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 1)], [(0, 0)],
                     [grid([0, 64], [0, 32, 64], [(1, 0)])])
    n, c = codes(spec, swapped)
    assert n > 0 and c == {1, 2}


def test_grid_segment_starts_are_decoded_exactly():
    """Row segments [0, 40) and [40, 128), column segments [0, 24) and
    [24, 64): the same block pattern with a start moved by one token is
    caught (a boundary off by one row or one column)."""
    qb = np.array([0, 40, 128], np.int32)
    kb = np.array([0, 24, 64, 128], np.int32)
    blocks = np.array([[[[1, 0, 0], [0, 1, 0]]]], np.uint8)
    spec = W.MaskSpec(W.MASK_SEGMENTS, 1, 1, 128, q_bounds=qb, k_bounds=kb, blocks=blocks)
    good = export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 1)], [(0, 0)],
                  [grid([0, 40], [0, 24, 64], [(0, 0), (1, 1)])])
    n, rep, _ = oracle.coverage(spec, good)
    assert n == 0, rep
    for rs, cs in (([0, 41], [0, 24, 64]), ([0, 39], [0, 24, 64]), ([0, 40], [0, 25, 64]),
                   ([0, 40], [0, 23, 64]), ([0, 40], [0, 24, 63])):
        bad = export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 1)], [(0, 0)],
                     [grid(rs, cs, [(0, 0), (1, 1)])])
        n, c = codes(spec, bad)
        assert n > 0 and c & {1, 2}, (rs, cs)


# ---------------------------------------------------------------------------
# Band form and temporal-major items: an SVG temporal head with radius R.
F_B, S_B = 4, 8                              # N = 32 tokens, one 128-row tile


@pytest.mark.parametrize("R", [0, 1, 2])
def test_band_plan_is_exact_and_radius_is_pinned(R):
    spec = W.svg_mask(1, 1, n_frames=F_B, frame_size=S_B, kinds=np.array([1], np.int8),
                      temporal_radius=R)
    N = F_B * S_B

    def plan(r, layout=1):
        return export(1, 1, N, 64, 128, 64, [(0, 0, 0, 1, layout)], [(0, 0)], [band(F_B, r)],
                      head_layout=[1], n_frames=F_B, frame_size=S_B)

    n, rep, st = oracle.coverage(spec, plan(R))
    assert n == 0, rep
    assert st["covered"] == F_B * F_B * (S_B * (2 * R + 1) - R * (R + 1))
    n, c = codes(spec, plan(R + 1))          # one segment too wide: extra pairs
    assert n > 0 and c == {2}
    if R > 0:
        n, c = codes(spec, plan(R - 1))      # one too narrow: missed pairs
        assert n > 0 and c == {1}
    n, c = codes(spec, plan(R, layout=0))    # caller order instead of temporal-major
    assert n > 0 and c & {1, 2}


def test_temporal_major_item_on_a_caller_order_head_is_code_8():
    """The malformed item is refused (8), so its query tile has no item (7)."""
    spec = W.svg_mask(1, 1, n_frames=F_B, frame_size=S_B, kinds=np.array([1], np.int8))
    buf = export(1, 1, 32, 64, 128, 64, [(0, 0, 0, 1, 1)], [(0, 0)], [band(F_B, 0)],
                 head_layout=[0], n_frames=F_B, frame_size=S_B)
    n, c = codes(spec, buf)
    assert n > 0 and c == {7, 8}


def test_temporal_major_grid_plan_with_permuted_rows():
    """A temporal head planned with a grid descriptor in temporal-major order
    (F = 16 tokens per segment, radius 0: blocks on the diagonal of 16 x 16
    blocks): rows and keys are mapped back to caller order by the checker."""
    F, S = 16, 8
    spec = W.svg_mask(1, 1, n_frames=F, frame_size=S, kinds=np.array([1], np.int8))
    # 128 temporal-major tokens = 8 segments of 16; the tile of keys 0..63 holds
    # segments 0..3, keys 64..127 segments 4..7
    d0 = grid(list(range(0, 128, 16)), [0, 16, 32, 48, 64], [(s, s) for s in range(4)])
    d1 = grid(list(range(0, 128, 16)), [0, 16, 32, 48, 64], [(s + 4, s) for s in range(4)])
    buf = export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 2, 1)], [(0, 0), (64, 1)], [d0, d1],
                 head_layout=[1], n_frames=F, frame_size=S)
    n, rep, st = oracle.coverage(spec, buf)
    assert n == 0, rep
    assert st["covered"] == 128 * F
    d1_bad = grid(list(range(0, 128, 16)), [0, 16, 32, 48, 64], [(s + 4, (s + 1) % 4) for s in range(4)])
    n, c = codes(spec, export(1, 1, 128, 64, 128, 64, [(0, 0, 0, 2, 1)], [(0, 0), (64, 1)],
                              [d0, d1_bad], head_layout=[1], n_frames=F, frame_size=S))
    assert n > 0 and c == {1, 2}


# ---------------------------------------------------------------------------
# List form: KEYLIST with 64-query slices, one 128-row tile holding two slices.
def test_list_plan_is_exact_and_bits_are_pinned():
    N = 100
    lists = [[1, 5, 70], [5, 99]]
    spec = W.MaskSpec(W.MASK_KEYLIST, 1, 1, N, slice_m=64,
                      indptr=np.array([0, 3, 5], np.int64),
                      indices=np.array(lists[0] + lists[1], np.int32))
    union = [1, 5, 70, 99]
    gidx = union + [0] * 60

    def plan(bits, g=gidx, bm=128):
        return export(1, 1, N, 64, bm, 64, [(0, 0, 0, 1)], [(0, 0)], [colmask(bits)], gidx=g,
                      gathered=1, slice_m=64)

    good = [[0, 1, 2], [1, 3]]
    n, rep, st = oracle.coverage(spec, plan(good))
    assert n == 0, rep
    assert st["covered"] == 64 * 3 + 36 * 2
    n, c = codes(spec, plan([[0, 1, 2], [0, 1, 3]]))   # key 1 given to slice 1
    assert n > 0 and c == {2}
    n, c = codes(spec, plan([[0, 1], [1, 3]]))         # key 70 dropped from slice 0
    assert n > 0 and c == {1}
    n, c = codes(spec, plan(good, g=[1, 5, 71, 99] + [0] * 60))   # wrong gathered key
    assert n > 0 and c == {1, 2}
    n, c = codes(spec, plan([list(range(64)), list(range(64))]))  # all columns, padding included
    assert n > 0 and 2 in c


def test_list_plan_with_64_row_tiles():
    """One 64-query slice per tile (bm = 64): each tile's single row segment."""
    N = 100
    spec = W.MaskSpec(W.MASK_KEYLIST, 1, 1, N, slice_m=64,
                      indptr=np.array([0, 3, 5], np.int64),
                      indices=np.array([1, 5, 70, 5, 99], np.int32))
    gidx = [1, 5, 70] + [0] * 61 + [5, 99] + [0] * 62
    buf = export(1, 1, N, 64, 64, 64, [(0, 0, 0, 1), (0, 1, 1, 2)], [(0, 0), (64, 1)],
                 [colmask([[0, 1, 2]]), colmask([[0, 1]])], gidx=gidx, gathered=1, slice_m=64)
    n, rep, st = oracle.coverage(spec, buf)
    assert n == 0, rep
    assert st["covered"] == 64 * 3 + 36 * 2
    bad = export(1, 1, N, 64, 64, 64, [(0, 0, 0, 1), (0, 1, 1, 2)], [(0, 0), (64, 1)],
                 [colmask([[0, 1, 2]]), colmask([[0]])], gidx=gidx, gathered=1, slice_m=64)
    n, c = codes(spec, bad)                          # key 99 dropped from slice 1
    assert n > 0 and c == {1}
    bad = export(1, 1, N, 64, 64, 64, [(0, 0, 0, 1), (0, 1, 1, 2)], [(0, 0), (64, 1)],
                 [colmask([[0, 1, 2]]), colmask([[0, 1, 2]])], gidx=gidx, gathered=1, slice_m=64)
    n, c = codes(spec, bad)                          # a padding slot (key 0) selected
    assert n > 0 and c == {2}


def test_malformed_exports_are_refused():
    good = grid_plan()
    with pytest.raises(ValueError):
        oracle.coverage(SPEC_G, good[:60])                       # shorter than the header
    with pytest.raises(ValueError):
        oracle.coverage(SPEC_G, b"XXXX" + good[4:])              # bad magic
    with pytest.raises(ValueError):
        oracle.coverage(SPEC_G, good[:-10])                      # truncated body
    other = W.MaskSpec(W.MASK_UNIFORM, 1, 1, 256, bq=64, bk=64,
                       blocks=np.ones((1, 1, 4, 4), np.uint8))
    with pytest.raises(ValueError):
        oracle.coverage(other, good)                             # N differs from the mask
