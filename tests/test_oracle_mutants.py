"""Plant plausible mistakes in copies of the oracle source and check that the
pins catch every one of them.

Each mutant is a one-line textual edit (a dropped term, a flipped sign, a wrong
index or a transposed operand).  The edit must match the oracle source exactly
once, so that a later change to the oracle that removes the line fails here
loudly instead of silently weakening the check.  The mutant library is built
in a temporary directory; the real oracle is not touched.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))

MUTANTS = {
    "lse_drops_max": ("attn_oracle.c", "const double lse = M + log(sum);",
                      "const double lse = log(sum);"),
    "causal_strict": ("attn_oracle.c", "return (i + 1 < Sk) ? i + 1 : Sk;",
                      "return (i < Sk) ? i : Sk;"),
    "gqa_head_modulo": ("attn_oracle.c", "return (int)(((long long)h * Hkv) / Hq);",
                        "return h % Hkv;"),
    "scale_missing": ("attn_oracle.c", "s[j] = scale * dot(q_row, k_head + j * D, D);",
                      "s[j] = dot(q_row, k_head + j * D, D);"),
    "p_unnormalised": ("attn_oracle.c", "const double p = exp(s[j] - lse);",
                       "const double p = exp(s[j] - M);"),
    "dq_ds_sign": ("attn_oracle.c", "const double ds = p * (dp - Di);",
                   "const double ds = p * (Di - dp);"),
    "dk_delta_sign": ("attn_oracle.c",
                      "const double ds = p * (dp - delta[gi * (long)Sq + i]);",
                      "const double ds = p * (dp + delta[gi * (long)Sq + i]);"),
    "dk_scale_missing": ("attn_oracle.c", "dkj[d] += scale * ds * qi[d];",
                         "dkj[d] += ds * qi[d];"),
    "dv_wrong_operand": ("attn_oracle.c", "dvj[d] += p * doi[d];", "dvj[d] += ds * doi[d];"),
    "dp_uses_k": ("attn_oracle.c", "const double dp = dot(doi, v_head + j * D, D);",
                  "const double dp = dot(doi, k_head + j * D, D);"),
    "dkdv_ignores_causal": ("attn_oracle.c", "for (long i = causal ? j : 0; i < Sq; ++i) {",
                            "for (long i = 0; i < Sq; ++i) {"),
    "mod_window_left_off_by_one": ("attn_oracle.c", "if (wl >= 0 && i - wl > a) a = i - wl;",
                                   "if (wl >= 0 && i - wl > a) a = i - wl + 1;"),
    "mod_window_right_off_by_one": ("attn_oracle.c",
                                    "if (wr >= 0 && i + wr + 1 < b) b = i + wr + 1;",
                                    "if (wr >= 0 && i + wr + 1 < b) b = i + wr;"),
    "mod_bias_sign": ("attn_oracle.c",
                      "return scale * dot(qi, kj, D) + slope * (double)(j - i);",
                      "return scale * dot(qi, kj, D) + slope * (double)(i - j);"),
    "mod_slope_head_index": ("attn_oracle.c", "return slopes ? slopes[h] : 0.0;",
                             "return slopes ? slopes[0] : 0.0;"),
    "mod_dkdv_ignores_window": ("attn_oracle.c", "if (j < lo || j >= hi) continue;",
                                "if (j >= hi) continue;"),
    "mod_dq_row_term_sign": ("attn_oracle.c",
                             "const double g_w = w * (dot(gi_row, vh + j * D, D) - rterm);",
                             "const double g_w = w * (dot(gi_row, vh + j * D, D) + rterm);"),
    "padding_length_ignored": ("attn_oracle.c", "return L < 0 ? 0 : (L > Sk ? Sk : L);",
                               "return Sk + 0 * L;"),
    "padding_length_inclusive": ("attn_oracle.c", "const long L = seqlens_k[b];",
                                 "const long L = seqlens_k[b] + 1;"),
    "merge_lse_drops_max": ("attn_oracle.c", "const double row_lse = M + log(z);",
                            "const double row_lse = log(z);"),
    "merge_weights_unnormalised": ("attn_oracle.c",
                                   "const double w = exp(lse_parts[(long)c * rows + r] - row_lse);",
                                   "const double w = exp(lse_parts[(long)c * rows + r] - M);"),
    "range_ignores_k0": ("attn_oracle.c", "if (lo < k0) lo = k0;", "if (lo < 0) lo = k0;"),
    "range_upper_inclusive": ("attn_oracle.c", "if (hi > k1) hi = k1;",
                              "if (hi > k1 + 1) hi = k1 + 1;"),
    "tiled_threshold_reversed": ("tiled_body.h",
                                 "} else if (tile_max - m[r] > (REAL)threshold) {",
                                 "} else if (m[r] - tile_max > (REAL)threshold) {"),
    "tiled_acc_not_rescaled": ("tiled_body.h",
                               "acc[r * D + d] = acc[r * D + d] * alpha + pv;",
                               "acc[r * D + d] = acc[r * D + d] + pv;"),
    "tiled_lse_base2": ("tiled_body.h", "lse[flat] = (double)(ln2 * (m[r] + LOG2(l[r])));",
                        "lse[flat] = (double)(m[r] + LOG2(l[r]));"),
    "tiled_sum_not_rescaled": ("tiled_body.h", "l[r] = l[r] * alpha + tile_l;",
                               "l[r] = l[r] + tile_l;"),
}


def _build_mutant(tmp_path, name):
    fname, old, new = MUTANTS[name]
    d = tmp_path / name
    d.mkdir()
    for f in ("attn_oracle.c", "tiled_body.h"):
        shutil.copy(os.path.join(ORACLE_DIR, f), d / f)
    src = (d / fname).read_text()
    assert src.count(old) == 1, f"mutant {name}: target line not found exactly once"
    (d / fname).write_text(src.replace(old, new))
    out = d / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(d / "attn_oracle.c"), "-o", str(out), "-lm"], check=True)
    return oracle.load(str(out))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
