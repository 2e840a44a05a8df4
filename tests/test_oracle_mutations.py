"""Planted mistakes: each mutant copy of the oracle must fail at least one pin.

A mutant is the oracle's C source with one line changed (a dropped term, a wrong
sign, index or tie-break, a transposed operand).  It is compiled into a temporary
library on the CPU; the real oracle is untouched.  Every mutant here keeps all
memory accesses in bounds.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins as P

SRC_DIR = os.path.dirname(os.path.abspath(oracle.__file__))

MUTANTS = {
    "sigmoid_sign": ("double e = exp(-(double)x);", "double e = exp((double)x);"),
    "sigmoid_in_float": ("double s = 1.0 / (1.0 + e);\n    return (float)s;",
                         "float s = 1.0f / (1.0f + (float)e);\n    return s;"),
    "bf16_truncate": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    "bf16_ties_away": ("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;"),
    "no_bias": ("b[e] = s[e] + bias[e];", "b[e] = s[e];"),
    "group_top1_only": ("gs[g] = m1 + m2;", "gs[g] = m1;"),
    "group_top1_twice": ("gs[g] = m1 + m2;", "gs[g] = m1 + m1;"),
    "top2_no_multiplicity": ("} else if (b[e] > m2) {", "} else if (b[e] > m2 && b[e] < m1) {"),
    "group_tie_to_higher": ("if (best < 0 || gs[g] > gs[best]) best = g;",
                            "if (best < 0 || gs[g] >= gs[best]) best = g;"),
    "group_of_expert_interleaved": ("if (!kept[e / gsize] || taken[e]) continue;",
                                    "if (!kept[e % n_group] || taken[e]) continue;"),
    "expert_tie_to_higher": ("if (best < 0 || b[e] > b[best]) best = e;",
                             "if (best < 0 || b[e] >= b[best]) best = e;"),
    "weights_from_biased": ("float q = s[slot_id[j]] / den;", "float q = b[slot_id[j]] / den;"),
    "den_from_biased": ("den = den + s[slot_id[j]];", "den = den + b[slot_id[j]];"),
    "den_first_slot_dropped": ("for (int j = 0; j < k; ++j) den = den + s[slot_id[j]];",
                               "for (int j = 1; j < k; ++j) den = den + s[slot_id[j]];"),
    "relabel_slot_reversed": ("l = local_count + j;", "l = local_count + (k - 1 - j);"),
    "relabel_local_reversed": ("l = id - local_offset;",
                               "l = local_count - 1 - (id - local_offset);"),
    "perm_slot_major": ("for (int t = 0; t < T; ++t)\n        for (int j = 0; j < k; ++j) {\n"
                        "            int32_t l = lid[(size_t)t * k + j];",
                        "for (int j = 0; j < k; ++j)\n        for (int t = 0; t < T; ++t) {\n"
                        "            int32_t l = lid[(size_t)t * k + j];"),
    "gemm_weight_transposed": ("(double)f32_from_bf16(w[(size_t)e * H + h]);",
                               "(double)f32_from_bf16(w[(size_t)h * E + e]);"),
    "num_experts_no_roundup": ("return ((local_count + k + 3) / 4) * 4;",
                               "return local_count + k;"),
    "layout_inverse_transposed": ("for (int p = 0; p < n; ++p) inv_perm[perm[p]] = p;",
                                  "for (int p = 0; p < n; ++p) inv_perm[p] = perm[p];"),
    "layout_round_down": ("long long blocks = ((long long)counts[e] + tile - 1) / tile;",
                          "long long blocks = ((long long)counts[e]) / tile;"),
    "layout_pad_zero": ("        if (padded_rows) padded_rows[r] = -1;",
                        "        if (padded_rows) padded_rows[r] = 0;"),
    "layout_bin_index_shifted": ("            if (m_indices) m_indices[poff[e] + i] = e;",
                                 "            if (m_indices) m_indices[poff[e] + i] = e + 1;"),
    "index_weight_bits_as_id": ("        int l = (int)((uint32_t)packed[i] >> 16);\n        perm[cursor[l]] = (int32_t)i;",
                                "        int l = (int)((uint32_t)packed[i] >> 16);\n        perm[cursor[l]] = (int32_t)(n - 1 - i);"),
    "dispatch_interleaved_ranks": ("        send_counts[ids[i] / per] += 1;", "        send_counts[ids[i] % R] += 1;"),
    "alltoall_row_for_column": ("        recv_counts[s] = matrix[(size_t)s * R + me];",
                                "        recv_counts[s] = matrix[(size_t)me * R + s];"),
    "e2m1_ties_to_larger": ("if (dc < db || (dc == db && (c & 1) == 0)) best = c;",
                            "if (dc <= db) best = c;"),
    "e2m1_sign_dropped": ("int neg = signbit(v) ? 1 : 0;", "int neg = 0;"),
    "mx_emax_three": ("e = (ex - 1) - 2;", "e = (ex - 1) - 3;"),
    "mx_ceil_log2": ("e = (ex - 1) - 2;", "e = ex - 2;"),
    "mx_zero_block_unit_scale": ("                e = -127;\n            } else {",
                                 "                e = 0;\n            } else {"),
    "mx_no_low_clamp": ("if (e < -127) e = -127;", "if (e < -200) e = -200;"),
    "mx_nibbles_swapped": ("(uint8_t)(lo | (hi << 4));", "(uint8_t)(hi | (lo << 4));"),
}

# cheap pins first; the exhaustive sigmoid sweep last
ORDER = [p for p in P.ALL_PINS if p is not P.pin_sigmoid_exact] + [P.pin_sigmoid_exact]


def _build_mutant(tmp_path, old, new):
    d = tmp_path / "mut"
    d.mkdir()
    for f in ("oracle.c", "oracle.h"):
        shutil.copy(os.path.join(SRC_DIR, f), d / f)
    src = (d / "oracle.c").read_text()
    assert src.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
    (d / "oracle.c").write_text(src.replace(old, new))
    so = d / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(d / "oracle.c"), "-lm"])
    return oracle.load(str(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, old, new)
    for pin in ORDER:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError):
            return  # caught
    pytest.fail(f"no pin caught mutant {name}")
