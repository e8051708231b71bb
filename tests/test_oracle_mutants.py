"""The oracle's pins are strong enough to catch plausible oracle bugs.

Each case plants one mistake in a private copy of the oracle's C source (a
wrong index, a dropped term, a swapped operand, an off-by-one), compiles it
to a temporary library, points the oracle's ctypes front end at it and runs
the pins of test_oracle.py.  At least one pin must fail for every mutant;
the unmodified source must pass them all (test_oracle.py itself).
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()

MUTANTS = {
    "gqa_modulo_grouping": ("h / group", "h % num_kv_heads"),
    "block_index_modulo": ("block_table[t / ORACLE_BLOCK]", "block_table[t % max_blocks]"),
    "offset_from_quotient": ("block * ORACLE_BLOCK + t % ORACLE_BLOCK", "block * ORACLE_BLOCK + t / ORACLE_BLOCK"),
    "causal_off_by_one": ("ctx - lq + (tok - t0) + 1", "ctx - lq + (tok - t0)"),
    "causal_top_left": ("ctx - lq + (tok - t0) + 1", "(tok - t0) + 1"),
    "scale_dropped": ("x[t] = scale * dot;", "x[t] = dot;"),
    "not_normalised": ("const double p = x[t] / z;", "const double p = x[t];"),
    "logit_reads_values": ("const double* k = K + (int64_t)t * row", "const double* k = V + (int64_t)t * row"),
    "head_offset_unscaled": ("const double* v = V + (int64_t)t * row + (int64_t)kv_head * head_dim;",
                             "const double* v = V + (int64_t)t * row + (int64_t)kv_head;"),
    "decode_misses_last_key": ("h / group, ctx, scale, dst, NULL", "h / group, ctx - 1, scale, dst, NULL"),
    "store_writes_v_into_k": ("k_cache[slot * row + e] = k[i * k_row_stride + e];",
                              "k_cache[slot * row + e] = v[i * v_row_stride + e];"),
    "store_skips_every_negative": ("if (slot == -1) continue;", "if (slot < 0) continue;"),
    "store_slot_off_by_one": ("v_cache[slot * row + e] = v[i * v_row_stride + e];",
                              "v_cache[(slot + 1 < num_slots ? slot + 1 : slot) * row + e] = v[i * v_row_stride + e];"),
}

PINS = [
    pins.test_golden_decode_block_boundary,
    pins.test_golden_prefill_bottom_right,
    pins.test_golden_gqa_grouping,
    pins.test_golden_store_rows,
    lambda: pins.test_decode_matches_library_sdpa(4, 2, 64),
    lambda: pins.test_prefill_matches_library_sdpa_lower_right(200, 100),
    pins.test_brute_force_tiny_decode,
    pins.test_brute_force_tiny_prefill,
    pins.test_single_key_returns_its_value_exactly,
    pins.test_zero_query_gives_mean_value,
    pins.test_dominant_key_selects_its_value,
    pins.test_softmax_rows_sum_to_one,
    pins.test_store_matches_indexed_assignment,
    pins.test_store_rejects_out_of_range_slot,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(src), "-o", str(so), "-lm"])
    saved = oracle._lib
    try:
        oracle._lib = None
        real_build = oracle.build
        oracle.build = lambda force=False: str(so)
        oracle.lib()
        caught = None
        for pin in PINS:
            try:
                pin()
            except (Exception, pytest.fail.Exception):
                caught = pin
                break
        assert caught is not None, f"no pin caught mutant {name}"
    finally:
        oracle.build = real_build
        oracle._lib = saved
