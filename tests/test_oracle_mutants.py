"""Planted mistakes in the oracle and in the plan checker are caught (CPU only).

Each case copies ``oracle/oracle.c`` and ``oracle/coverage.c``, plants ONE
plausible mistake in the copy (a dropped term, a wrong scale, an index off by
one, a transposed bit index, a report that never fires), compiles it and runs
the named pins of ``tests/test_oracle_pins.py`` and
``tests/test_coverage_pins.py`` on that build.  Every named pin must fail on
the mutant -- otherwise the pins would not detect that mistake in the real
oracle.  The unmodified sources pass the same pins (their own test files).
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_coverage_pins as CP
import test_oracle_pins as OP

HERE = os.path.dirname(os.path.abspath(oracle.__file__))

# name: (file, original text, replacement, [(pin, args), ...])
MUTANTS = {
    # --- oracle.c: the attention definition
    "scale_1_over_d": ("oracle.c", "const double scale = 1.0 / sqrt((double)d);",
                       "const double scale = 1.0 / (double)d;",
                       [(OP.test_all_ones_is_dense_attention, ()),
                        (OP.test_two_keys_by_hand, ())]),
    "no_frame0_rule": ("oracle.c", "if (j / S == fi || j / S == 0) keys[n++] = j;",
                       "if (j / S == fi) keys[n++] = j;",
                       [(OP.test_svg_counted_densities, (21, 1560))]),
    "block_row_uses_bk": ("oracle.c", "i / m->bq) * nkb;", "i / m->bk) * nkb;",
                          [(OP.test_uniform_row_counts_closed_form, ())]),
    "perturbed_exponent": ("oracle.c", "s[t] = exp(s[t] - mx);",
                           "s[t] = exp(1.001 * (s[t] - mx));",
                           [(OP.test_two_keys_by_hand, ()),
                            (OP.test_all_ones_is_dense_attention, ())]),
    "lse_without_max": ("oracle.c", "*lse = mx + log(l);", "*lse = log(l);",
                        [(OP.test_one_key_closed_form, ()), (OP.test_two_keys_by_hand, ())]),
    "empty_row_lse_zero": ("oracle.c", "*lse = -INFINITY;\n    return 0;",
                           "*lse = 0.0;\n    return 0;",
                           [(OP.test_empty_rows_exact, ())]),
    "radius_ignored": ("oracle.c", "const int32_t si = i % S, r = m->temporal_radius;",
                       "const int32_t si = i % S, r = 0;",
                       [(OP.test_svg_temporal_radius_counted, (5, 40, 3))]),
    "temporal_uses_frame": ("oracle.c", "keys[n++] = f * S + sj;", "keys[n++] = sj * S + f;",
                            [(OP.test_temporal_permutation_invariance, ())]),
    "keylist_block_off_by_one": ("oracle.c", "+ i / m->slice_m;", "+ (i + 1) / m->slice_m;",
                                 [(OP.test_one_key_closed_form, ())]),
    "probabilities_not_normalised": ("oracle.c", "const double p = s[t] / l;",
                                     "const double p = s[t];",
                                     [(OP.test_constant_v_closed_form, ())]),
    # --- coverage.c: the plan checker
    "grid_bit_transposed": ("coverage.c", "(d->bits >> (rs * 8 + cs))", "(d->bits >> (cs * 8 + rs))",
                            [(CP.test_grid_bit_index_is_row_times_8_plus_column, ())]),
    "band_radius_off_by_one": ("coverage.c", "return (dist <= R && -dist <= R) ? 1 : 0;",
                               "return (dist <= R + 1 && -dist <= R + 1) ? 1 : 0;",
                               [(CP.test_band_plan_is_exact_and_radius_is_pinned, (1,))]),
    "row_segment_start_off_by_one": ("coverage.c", "d->r_start[rs + 1] <= r", "d->r_start[rs + 1] < r",
                                     [(CP.test_grid_segment_starts_are_decoded_exactly, ())]),
    "code1_never_reported": ("coverage.c", "if (ar[j] && c == 0) report_add", "if (0) report_add",
                             [(CP.test_dropped_tile_is_code_1, ())]),
    "code3_never_reported": ("coverage.c", "else if (c > 1) report_add", "else if (c > 2) report_add",
                             [(CP.test_duplicated_tile_is_code_3, ())]),
    "full_tile_not_checked": ("coverage.c", "if (E->desc < 0 && full_bad) report_add",
                              "if (0 && full_bad) report_add",
                              [(CP.test_full_tile_over_masked_pair_is_code_4, ())]),
    "list_segment_ignored": ("coverage.c", "const int seg = r / p->h->slice_m;", "const int seg = 0;",
                             [(CP.test_list_plan_is_exact_and_bits_are_pinned, ())]),
    "unpermute_swapped": ("coverage.c", "return (tp % F) * S + tp / F;", "return (tp / F) * S + tp % F;",
                          [(CP.test_temporal_major_grid_plan_with_permuted_rows, ())]),
    "query_tile_count_unchecked": ("coverage.c", "if (seen[t] != 1) report_add", "if (seen[t] > 1) report_add",
                                   [(CP.test_missing_or_repeated_query_tile_is_code_7, ())]),
}


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


def build_mutant(workdir, name):
    fname, old, new, _ = MUTANTS[name]
    d = workdir / name
    d.mkdir()
    for f in ("oracle.c", "coverage.c", "oracle_mask.h"):
        shutil.copy(os.path.join(HERE, f), d / f)
    src = (d / fname).read_text()
    assert src.count(old) == 1, f"{name}: the text to mutate must occur exactly once"
    (d / fname).write_text(src.replace(old, new))
    so = d / f"liboracle_{name}.so"
    cmd = ["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(d / "oracle.c"),
           str(d / "coverage.c"), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_its_pins(workdir, name):
    so = build_mutant(workdir, name)
    with oracle.swapped_library(so):
        for pin, args in MUTANTS[name][3]:
            with pytest.raises((AssertionError, ValueError)):
                pin(*args)
    # the normal build is back and passes the same pins
    for pin, args in MUTANTS[name][3]:
        pin(*args)
