"""Planted mistakes: each broken copy of the oracle must fail at least one pin.

A mutant is the oracle's C source with one plausible mistake substituted in
(wrong start rank, reversed ring, dropped alignment, wrong rounding, signedness
slip, dropped term ...). It is compiled on the CPU into a temporary library and
the pins of oracle_pins.py are run against it. This shows the pins can tell a
correct oracle from a subtly wrong one.
"""
import os

import pytest

import oracle
from oracle import build as obuild
import oracle_pins as P

SRC = obuild.SRC

MUTANTS = {
    "start_at_c": ("acc = ((const T*)xs[(c + 1) % N])[i];",
                   "acc = ((const T*)xs[(c) % N])[i];"),
    "start_at_c_plus_2": ("acc = ((const T*)xs[(c + 1) % N])[i];",
                          "acc = ((const T*)xs[(c + 2) % N])[i];"),
    "ring_backwards": ("acc = COMBINE(op, acc, ((const T*)xs[(c + k) % N])[i]);",
                       "acc = COMBINE(op, acc, ((const T*)xs[(c + 2 * N + 2 - k) % N])[i]);"),
    "dropped_last_term": ("for (int k = 2; k <= N; ++k)", "for (int k = 2; k < N; ++k)"),
    "last_loop_no_align": ("? align_up(div_up(rem, (uint64_t)N), align)",
                           "? div_up(rem, (uint64_t)N)"),
    "channel_no_align": ("uint64_t per = align_up(div_up(count, (uint64_t)nChannels), align);",
                         "uint64_t per = div_up(count, (uint64_t)nChannels);"),
    "truncate_not_round": ("double r = nearbyint(n);", "double r = trunc(n);"),
    "ties_away": ("double r = nearbyint(n);", "double r = round(n);"),
    "no_overflow_to_inf": ("if (fabs(y) > maxf) return copysign(INFINITY, x);", ""),
    "unsigned_max_for_signed": ("COMBINE_INT(combine_i32, int32_t, uint32_t)",
                                "COMBINE_INT(combine_i32, uint32_t, uint32_t)"),
    "max_is_min": ("case OR_MAX: return a > b ? a : b;                                     \\",
                   "case OR_MAX: return a < b ? a : b;                                     \\"),
    "no_rounding_16bit": ("return encode16(round_fmt(combine_double(op, x, y), f), f);",
                          "return encode16(combine_double(op, x, y), f);"),
    "reduce_scatter_starts_at_b": ("fold(op, N, blk, outs[b], 0, recvcount, b);",
                                   "fold(op, N, blk, outs[b], 0, recvcount, (b + N - 1) % N);"),
    "all_gather_wrong_block": ("memcpy((char*)outs[b] + (size_t)k * bytes, xs[k], bytes);",
                               "memcpy((char*)outs[b] + (size_t)k * bytes, xs[(k + b) % N], bytes);"),
    "tree_parent_added_not_ored": ("int parent = (r - b) | (2 * b);",
                                   "int parent = (r - b) + (2 * b);"),
    "tree_children_swapped": ("if (d0[r] >= 0) acc = COMBINE(op, acc, val[d0[r]]);",
                              "if (d1[r] >= 0) acc = COMBINE(op, acc, val[d1[r]]);"
                              " if (d0[r] >= 0) acc = COMBINE(op, acc, val[d0[r]]); if (0)"),
    "tree_second_not_mirrored": ("if (tree == 0) {\n    btree_node(N, r, up, d0, d1);",
                                 "if (tree >= 0) {\n    btree_node(N, r, up, d0, d1);"),
    "tree_split_unaligned": ("uint64_t h = align_up(div_up(count, 2), 16 / (uint64_t)elemSize);",
                             "uint64_t h = div_up(count, 2);"),
    "avg_int_not_divided": ("  if (rc == 0 && !premul)\n    divide_by_n(",
                            "  if (rc == 0 && !premul && 0)\n    divide_by_n("),
    "avg_float_by_postdivision": ("const int premul = kind == 0 || is_float_type(dtype);",
                                  "const int premul = kind == 0;"),
    "premul_scalar_not_rounded_16bit": ("oracle_f16_from_double(scalar));",
                                        "oracle_f16_from_double(scalar * 1.0001));"),
    "fp8_no_saturation": ("  if (fabs(y) > f.maxf) y = copysign(f.maxf, x);\n", ""),
    "fp8_e4m3_nan_code_finite": ("} else if (!f.has_inf && ef == eall && mf == mall) {",
                                 "} else if (!f.has_inf && ef == eall && mf == mall && 0) {"),
    "fp8_e5m2_bias_off": ("static const fmt8 FMT_E5M2 = {3, -14, 15, 5, 1, 57344.0};",
                          "static const fmt8 FMT_E5M2 = {3, -14, 16, 5, 1, 57344.0};"),
    "tree_avg_int_not_divided": ("  if (rc == 0 && !premul) {\n    void* outs[1] = {out};",
                                 "  if (rc == 0 && !premul && 0) {\n    void* outs[1] = {out};"),
    "chunk_index_off_by_one": ("visit(ctx, ch, loop, c, cb + off + lo, cb + off + hi);",
                               "visit(ctx, ch, loop, (c + 1) % N, cb + off + lo, cb + off + hi);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib_path = str(tmp_path / f"libmutant_{name}.so")
    obuild.compile_oracle(str(src), lib_path, extra=("-Wno-unused-parameter", "-w"))
    lib = oracle.load(lib_path)
    failed = []
    for pin in P.ALL_PINS:
        try:
            if pin is P.pin_m2_first_element:
                pin(lib, max_count=4096)
            elif pin is P.pin_fold_equals_simulation:
                pin(lib, quick=True)
            else:
                pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(source, tmp_path):
    src = tmp_path / "same.c"
    src.write_text(source)
    lib_path = str(tmp_path / "libsame.so")
    obuild.compile_oracle(str(src), lib_path)
    lib = oracle.load(lib_path)
    P.pin_sentinel_start_rank(lib)
    P.pin_chunk_map(lib)
