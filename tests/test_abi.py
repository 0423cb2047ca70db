"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
entry point that include/tsr.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

import block_sparse_attention_tsr_gb300 as tsr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    tsr.build()
    return tsr.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "tsr.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(tsr_[a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_entry_points():
    names = _declared()
    assert "tsr_plan" in names and "tsr_bsa_forward" in names
    assert len(names) >= 12


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert set(tsr.EXPORTS) <= set(_declared())


def test_abi_version_and_strings(L):
    assert tsr.tsr_abi_version() == 3
    assert L.tsr_status_string(0) == b"ok"
    assert L.tsr_status_string(5) == b"device wait timed out"


def _mask(**kw):
    m = tsr._Mask()
    for k, v in kw.items():
        setattr(m, k, v)
    return m


@pytest.mark.parametrize("kw,code", [
    (dict(kind=0, B=1, H=1, N=128, d=96, bq=64, bk=64, blocks=16), 1),      # d not 64/128
    (dict(kind=0, B=1, H=1, N=128, d=64, bq=8, bk=64, blocks=16), 1),       # block < 16
    (dict(kind=0, B=1, H=1, N=128, d=64, bq=64, bk=64, blocks=0), 1),       # no blocks
    (dict(kind=0, B=0, H=1, N=128, d=64, bq=64, bk=64, blocks=16), 1),      # B = 0
    (dict(kind=2, B=1, H=2, N=100, d=64, n_frames=3, frame_size=30, head_kind=16), 1),  # F*S != N
    (dict(kind=9, B=1, H=1, N=128, d=64), 1),                               # unknown kind
])
def test_plan_rejects_bad_arguments_on_host(L, kw, code):
    h = ctypes.c_void_p(0)
    m = _mask(**kw)
    st = L.tsr_plan(ctypes.byref(m), None, ctypes.byref(h), None)
    assert st == code
    assert h.value is None or h.value == 0
    assert len(L.tsr_last_error()) > 0


@pytest.mark.parametrize("field,value", [("kv_split", 3), ("kv_split", -1), ("kv_split", 8),
                                         ("orient", 3), ("bn", 96)])
def test_plan_rejects_bad_options_on_host(L, field, value):
    h = ctypes.c_void_p(0)
    m = _mask(kind=0, B=1, H=1, N=128, d=128, bq=64, bk=64, blocks=16)
    o = tsr._Opts()
    setattr(o, field, value)
    assert L.tsr_plan(ctypes.byref(m), ctypes.byref(o), ctypes.byref(h), None) == 1
    assert h.value is None or h.value == 0
    assert field.encode() in L.tsr_last_error()


def test_forward_rejects_null_plan(L):
    assert L.tsr_bsa_forward(None, None, None, None, None, None, None) == 1


def test_regime_table_parsing(L, tmp_path):
    good = tmp_path / "good.txt"
    good.write_text("# comment\n0 64 64 * * 0 0.5 128 64 4 1\n* * * * * * * 128 128 3 1\n"
                    "* * * * * * * 64 128 4 1\n")
    tsr.tsr_regime_load(str(good))
    r = tsr.tsr_regime_lookup(0, 64, 64, 32760, 0.2)
    assert (r["bn"], r["stages"], r["ctas_per_sm"], r["id"]) == (64, 4, 1, 0)
    assert r["orient"] == tsr.ORIENT_ROWS
    r = tsr.tsr_regime_lookup(0, 64, 64, 32760, 0.7)
    assert (r["bn"], r["id"]) == (128, 1)
    # orientation column: key-major rows, and "*" / absent meaning 128-row tiles
    good.write_text("0 64 64 * * 0 0.5 128 64 2 1 2\n0 64 64 * * 0.5 1.01 128 64 4 1 *\n"
                    "* * * * * * * 128 128 3 1 1\n")
    tsr.tsr_regime_load(str(good))
    r = tsr.tsr_regime_lookup(0, 64, 64, 32760, 0.2)
    assert (r["bn"], r["stages"], r["ctas_per_sm"], r["id"], r["orient"]) == (64, 2, 1, 0, tsr.ORIENT_KEYS)
    r = tsr.tsr_regime_lookup(0, 64, 64, 32760, 0.7)
    assert (r["bn"], r["stages"], r["id"], r["orient"]) == (64, 4, 1, tsr.ORIENT_ROWS)
    r = tsr.tsr_regime_lookup(0, 32, 32, 32760, 0.7)
    assert (r["bn"], r["id"], r["orient"]) == (128, 2, tsr.ORIENT_ROWS)
    bad = tmp_path / "bad.txt"
    for row in ("* * * * * * * 128 128 3 1 2",            # key-major rows name the one kernel
                "* * * * * * * 64 64 2 1 2",              # key-major tiles need d = 128
                "* * * * * * * 128 64 2 1 3"):            # no such orientation
        bad.write_text(row + "\n")
        with pytest.raises(tsr.TsrError):
            tsr.tsr_regime_load(str(bad))
    r = tsr.tsr_regime_lookup(0, 64, 64, 32760, 0.2)       # a refused table leaves the last one
    assert r["orient"] == tsr.ORIENT_KEYS
    bad.write_text("* * * * * * * 128 96 3 1\n")            # no such kernel variant
    with pytest.raises(tsr.TsrError):
        tsr.tsr_regime_load(str(bad))
    bad.write_text("* * * 1\n")
    with pytest.raises(tsr.TsrError):
        tsr.tsr_regime_load(str(bad))
    tsr.tsr_regime_load(tsr.REGIME_TABLE if os.path.exists(tsr.REGIME_TABLE) else None)


def test_package_has_no_cpu_path():
    src = open(os.path.join(ROOT, "block_sparse_attention_tsr_gb300", "__init__.py")).read()
    assert "import oracle" not in src and "from oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "block_sparse_attention_tsr_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "block_sparse_attention_tsr_gb300", "csrc", f)).read()


def test_plan_flags_match_the_header():
    """The binding's flag values are the header's #defines."""
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "tsr.h")).read()
    defs = dict(re.findall(r"#define (TSR_PLAN_\w+)\s+(\d+)", hdr))
    assert int(defs["TSR_PLAN_SYNC_CHECK"]) == tsr.PLAN_SYNC_CHECK
    assert int(defs["TSR_PLAN_NO_LPT"]) == tsr.PLAN_NO_LPT
    assert int(defs["TSR_PLAN_TEST_STALL"]) == tsr.PLAN_TEST_STALL
    assert int(defs["TSR_PLAN_DEBUG_CHECKS"]) == tsr.PLAN_DEBUG_CHECKS
    assert int(defs["TSR_PLAN_TEMPORAL_TILES"]) == tsr.PLAN_TEMPORAL_TILES
    # every flag the header defines is a distinct bit the binding knows
    assert sorted(int(v) for v in defs.values()) == [1, 2, 4, 8, 16]


def test_plan_stats_layout_matches_the_header():
    """The binding's tsr_plan_stats fields are the header's, in order."""
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "tsr.h")).read()
    body = hdr[hdr.index("/* Statistics of a plan"):]
    body = body[body.index("{") + 1:body.index("} tsr_plan_stats;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = [n for decl in body.split(";") if decl.strip()
             for n in re.sub(r"^\s*\w+\s+", "", decl.strip()).replace(" ", "").split(",")]
    assert names == [f for f, _ in tsr._Stats._fields_]
