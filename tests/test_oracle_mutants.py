"""Plant plausible mistakes in copies of the oracle (on the CPU) and require
the pins to catch every one: a pin set that a dropped scale, an off-by-one
mask, a transposed value index or a mis-ordered concat slips through is not
pinning the oracle."""
import os
import re

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement).  Each text must occur once.
MUTANTS = [
    ("scale_dropped", "w[j] = scale * dot +", "w[j] = dot +"),
    ("default_scale_1_over_d", "1.0 / sqrt((double)d) : scale", "1.0 / (double)d : scale"),
    ("causal_off_by_one", "(mask_kind & ORACLE_MASK_CAUSAL) && j > i",
     "(mask_kind & ORACLE_MASK_CAUSAL) && j >= i"),
    ("padding_off_by_one", "(mask_kind & ORACLE_MASK_KEY_PADDING) && j >= len_b",
     "(mask_kind & ORACLE_MASK_KEY_PADDING) && j > len_b"),
    ("no_normalisation", "w[j] = w[j] / Z;", "w[j] = w[j];"),
    ("value_dims_reversed", "o[c] += w[j] * V[(ptrdiff_t)j * ldv + c];",
     "o[c] += w[j] * V[(ptrdiff_t)j * ldv + (d - 1 - c)];"),
    ("max_not_subtracted_sign", "w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);"),
    ("heads_concat_reversed", "double *o = ctx + ((size_t)b * Lq + i) * D + (size_t)hh * d;",
     "double *o = ctx + ((size_t)b * Lq + i) * D + (size_t)(h - 1 - hh) * d;"),
    ("mha_scale_uses_dmodel", "const double sc = 1.0 / sqrt((double)d);\n#ifdef",
     "const double sc = 1.0 / sqrt((double)D);\n#ifdef"),
    ("key_proj_uses_wq", "matmul(x_kv, Wk, Kp,", "matmul(x_kv, Wq, Kp,"),
    ("float_mask_before_scale", "w[j] = scale * dot + mask_entry(i, j, mask_kind, len_b, Lq);\n        if (add_row)\n            w[j] += add_row[j];",
     "w[j] = scale * (dot + (add_row ? add_row[j] : 0.0)) + mask_entry(i, j, mask_kind, len_b, Lq);"),
    ("float_mask_transposed", "(int64_t)hh * add_stride_h + (int64_t)i * Lk\n                                          : NULL;",
     "(int64_t)hh * add_stride_h + (int64_t)i\n                                          : NULL;"),
    ("layernorm_unbiased_var", "        var /= D;\n", "        var /= (D - 1);\n"),
    ("ffn_no_relu", "hid[i] = hid[i] > 0.0 ? hid[i] : 0.0;", "hid[i] = hid[i];"),
    ("encoder_prenorm_residual", "add_layernorm(x1, f, g2, be2, eps, out, M, D);",
     "add_layernorm(x, f, g2, be2, eps, out, M, D);"),
    ("decode_top_left_alignment", "j > len_b - Lq + i)", "j > i)"),
    ("decode_off_by_one", "j > len_b - Lq + i)", "j >= len_b - Lq + i)"),
    ("pe_sin_cos_swapped", "(c % 2 == 0) ? sin(angle) : cos(angle)",
     "(c % 2 == 0) ? cos(angle) : sin(angle)"),
    ("pe_exponent_i_over_d", "(2.0 * i) / (double)D", "(double)i / (double)D"),
    ("pe_pair_index_is_column", "const int i = c / 2;", "const int i = c;"),
    ("pe_offset_ignored", "const double pos = (double)(first_pos + r);",
     "const double pos = (double)(r);"),
    ("embed_not_scaled", "scale == 0.0 ? sqrt((double)D) : scale", "scale == 0.0 ? 1.0 : scale"),
    ("bwd_ds_sign_flipped", "const double ds = w[j] * (dP[j] - mean);",
     "const double ds = w[j] * (mean - dP[j]);"),
    ("bwd_ds_no_mean", "const double ds = w[j] * (dP[j] - mean);", "const double ds = w[j] * dP[j];"),
    ("bwd_dq_unscaled", "dq[c] += sc * ds * Kh[(size_t)j * d + c];", "dq[c] += ds * Kh[(size_t)j * d + c];"),
    ("bwd_dv_uses_ds", "dVh[(size_t)j * d + c] += w[j] * g[c];", "dVh[(size_t)j * d + c] += w[j] * g[c] * sc;"),
    ("bwd_dk_uses_key", "dKh[(size_t)j * d + c] += sc * ds * q[c];",
     "dKh[(size_t)j * d + c] += sc * ds * Kh[(size_t)j * d + c];"),
    ("query_row_stride_wrong", "bad += attend_row(Qh + (size_t)i * d,",
     "bad += attend_row(Qh + (size_t)(Lq - 1 - i) * d,"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut_src = tmp_path / f"oracle_{name}.c"
    mut_src.write_text(src.replace(old, new))
    lib_path = oracle.build(str(mut_src), str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(oracle.load_library(lib_path))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
