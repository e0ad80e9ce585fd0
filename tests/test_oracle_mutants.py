"""The pins catch plausible mistakes in the oracle.

Each case below compiles a copy of the oracle's C source with one deliberate
mistake (a dropped term, a wrong sign, a wrong gather index, a swapped
operand, a wrong pair partner in the half-split mode, a wrong broadcast
index, a missing slice offset, swapped storage roundings, broken tie
rounding, or a fused multiply-add in place of the separate multiply and add) and runs every pin
check of ``oracle_pins`` against it.  At least one must fail.  The mistakes
are planted only in these temporary copies, on the CPU; every mutant stays
inside its buffers.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    # name: (text to replace, replacement, which occurrence (0-based))
    "fwd_dropped_cos_product": ("t1[j] = v[j] * c[j];", "t1[j] = v[j];", 0),
    "negates_the_wrong_lanes": ("mode == ORC_INTERLEAVE ? (j % 2 == 0)", "mode == ORC_INTERLEAVE ? (j % 2 == 1)", 0),
    "fwd_gather_without_swap": ("t2[j] = v[partner(mode, j, L)] * s[j];", "t2[j] = v[j] * s[j];", 0),
    "bwd_swapped_cos_sin": ("t2[j] = v[partner(mode, j, L)] * s[partner(mode, j, L)];",
                            "t2[j] = v[partner(mode, j, L)] * c[partner(mode, j, L)];", 0),
    "bwd_negates_the_forward_lanes": ("return dir == ORC_FWD ? first : !first;", "return first;", 0),
    "bwd_sin_of_wrong_lane": ("q = b * s[n];  v[i] = p + q;", "q = b * s[i];  v[i] = p + q;", 0),
    "pair_fwd_plus_sign": ("v[i] = p - q;", "v[i] = p + q;", 0),
    "half_partner_off_by_one": ("return j < L / 2 ? j + L / 2 : j - L / 2;",
                                "return j < L / 2 ? j + L / 2 - 1 : j - L / 2;", 0),
    "half_pairs_adjacent": ("mode == ORC_INTERLEAVE ? 2 * k + 1 : k + L / 2;",
                            "mode == ORC_INTERLEAVE ? 2 * k + 1 : k + 1;", 0),
    "half_negates_second_half": ("(j < L / 2);", "(j >= L / 2);", 0),
    "head_index_ignored": ("(r1_shape[2] == 1 ? 0 : n) * r1_stride[2]", "0 * r1_stride[2]", 0),
    "slice_offset_ignored": ("* D + start;", "* D;", 0),
    "storage_rounding_swapped": ("dtype == ORC_BF16 ? oracle_f32_to_bf16(v) : oracle_f32_to_f16(v)",
                                 "dtype == ORC_BF16 ? oracle_f32_to_f16(v) : oracle_f32_to_bf16(v)", 0),
    "ties_round_down": ("if (rem > half || (rem == half && (n & 1ull)))", "if (rem > half)", 0),
    "pair_fused_multiply_add": ("v[i] = p - q;", "v[i] = fmaf(a, c[i], -q);", 0),
    "chain_fused_multiply_add": ("for (j = 0; j < L; j++) v[j] = t1[j] + t2[j];",
                                 "for (j = 0; j < L; j++) v[j] = fmaf(v[j], c[j], t2[j]);", 0),
}


def _build_mutant(tmp_path, name):
    src = open(oracle.SRC).read()
    old, new, occ = MUTANTS[name]
    parts = src.split(old)
    assert len(parts) > occ + 1, f"mutation site for {name} not found"
    src = old.join(parts[: occ + 1]) + new + old.join(parts[occ + 1:])
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src)
    lib = os.path.join(tmp_path, f"lib_{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", lib, path, "-lm"],
                   check=True)
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    lib = _build_mutant(str(tmp_path), name)
    caught = []
    with oracle.using_library(lib):
        for check in P.ALL_CHECKS:
            try:
                check()
            except AssertionError:
                caught.append(check.__name__)
            except ValueError:
                caught.append(check.__name__ + " (rejected)")
    assert caught, f"no pin caught the mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = os.path.join(str(tmp_path), "lib_clean.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", lib,
                    oracle.SRC, "-lm"], check=True)
    with oracle.using_library(lib):
        for check in P.ALL_CHECKS:
            check()
