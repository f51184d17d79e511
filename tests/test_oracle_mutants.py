"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is a one-spot text change of oracle/okv_oracle.c (a dropped term, a wrong
sign or comparison, a wrong index or operand, an off-by-one), compiled on the CPU into a
temporary directory. The committed oracle itself is never modified.
"""
import os
import shutil
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "okv_oracle.c")

MUTANTS = {
    "kv_bytes_no_factor_2": ("return 2 * layers * kv_heads", "return layers * kv_heads"),
    "cap_ceil": ("double c = floor((double)cap * (double)budget_blocks);",
                 "double c = ceil((double)cap * (double)budget_blocks);"),
    "summary_skips_last_token": ("for (int32_t t = 1; t < nv; ++t) {", "for (int32_t t = 1; t < nv - 1; ++t) {"),
    "summary_reads_invalid_tokens": ("return n < 0 ? 0 : (n > bs ? bs : n);", "return n < 0 ? 0 : bs;"),
    "summary_min_max_swapped": ("if (load(host_unit, dtype, i) < load(host_unit, dtype, imin)) imin = i;",
                                "if (load(host_unit, dtype, i) > load(host_unit, dtype, imin)) imin = i;"),
    "score_drops_kmin": ("s += lo > hi ? lo : hi;", "s += hi;"),
    "score_min_not_max": ("s += lo > hi ? lo : hi;", "s += lo < hi ? lo : hi;"),
    "score_first_head_only": ("double x = load(q, dtype, (int64_t)h * d + c);", "double x = load(q, dtype, c);"),
    "score_transposed_summary": ("double lo = x * load(summ, dtype, ((int64_t)b * 2 + 0) * d + c);",
                                 "double lo = x * load(summ, dtype, ((int64_t)c * 2 + 0) * d + b);"),
    "topk_ascending": ("if (x->s > y->s) return -1;\n  if (x->s < y->s) return 1;",
                       "if (x->s < y->s) return -1;\n  if (x->s > y->s) return 1;"),
    "topk_ties_high_id": ("return (x->id > y->id) - (x->id < y->id);\n}\n\nint32_t oracle_topk",
                          "return (x->id < y->id) - (x->id > y->id);\n}\n\nint32_t oracle_topk"),
    "select_cap_ignored": ("const int32_t n_admit = n_miss < cap_blocks ? n_miss : cap_blocks;",
                           "const int32_t n_admit = n_miss;"),
    "select_hits_unprotected": ("      hit_slot[s] = 1;\n", "\n"),
    "select_most_recent_first": ("if (x->stamp != y->stamp) return (x->stamp > y->stamp) - (x->stamp < y->stamp);",
                                 "if (x->stamp != y->stamp) return (x->stamp < y->stamp) - (x->stamp > y->stamp);"),
    "select_ignores_stamp": ("if (x->stamp != y->stamp) return (x->stamp > y->stamp) - (x->stamp < y->stamp);", ""),
    "select_no_stamp_on_hit": ("      stamp[s] = step;\n      hit_slot[s] = 1;", "      hit_slot[s] = 1;"),
    "select_evicted_stays_mapped": ("if (old >= 0) resident[old] = -1;", ""),
    "local_ignores_capacity": ("if (*local_used < local_cap) {", "if (1) {"),
    "local_fill_marked_as_hit": ("route[i] = 2 * local_of[b] + 1;", "route[i] = 2 * local_of[b];"),
    "local_entry_off_by_one": ("local_of[b] = *local_used;", "local_of[b] = *local_used + 1;"),
    "local_full_reads_uncounted": ("    ++from_full;\n    if (*local_used", "    if (*local_used"),
    "attend_no_scale": ("z[k] = dot * scale;", "z[k] = dot;"),
    "attend_values_from_keys": ("z[k] * load(host_unit, dtype, v_off(b, t, c, bs, d));",
                                "z[k] * load(host_unit, dtype, k_off(b, t, c, bs, d));"),
    "attend_no_normalise": ("out[(int64_t)h * d + c] /= denom;", "out[(int64_t)h * d + c] /= 1.0;"),
    "attend_drops_last_slot": ("for (int32_t s = 0; s < kb; ++s)\n    if (slot_block[s] >= 0) blocks[n++] = slot_block[s];",
                               "for (int32_t s = 0; s < kb - 1; ++s)\n    if (slot_block[s] >= 0) blocks[n++] = slot_block[s];"),
    "append_no_new_block_reset": ("if (t == 0) {", "if (t == -1) {"),
    "append_v_into_k": ("copy_elem(host_unit, v_off(b, t, c, bs, d), v_new, c, dtype);",
                        "copy_elem(host_unit, k_off(b, t, c, bs, d), v_new, c, dtype);"),
}


@pytest.fixture(scope="module")
def tmpdir_mut():
    d = tempfile.mkdtemp(prefix="okv_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmpdir_mut):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name} is not unique in the oracle"
    path_c = os.path.join(tmpdir_mut, f"{name}.c")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.build(force=True, out_path=os.path.join(tmpdir_mut, f"{name}.so"), sources=[path_c])
    L = oracle.lib(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(L)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
