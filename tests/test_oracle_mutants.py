"""Planted mistakes: every plausible slip in the oracle must fail some pin.

Each mutant is a copy of the oracle's C source with one edit (a dropped term,
a wrong sign or index, a transposed operand, a wrong rounding rule), compiled
on the CPU into a temporary library. The pins of the other oracle test files
run against it, and at least one of them must fail. Nothing here touches the
CUDA path.
"""

import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_codec as codec
import test_oracle_gemm_master as gm
import test_oracle_scale_cast as sc

MUTANTS = [
    ("ties away from zero", "if (rem > half || (rem == half && (n & 1ull)))", "if (rem >= half)"),
    ("truncation", "if (rem > half || (rem == half && (n & 1ull)))", "if (0)"),
    ("wrong E4M3 bias in decode", "v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("E4M3 subnormal scale", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    ("Inf not saturated", "return sign | fmt_maxcode(fmt);      /* +-Inf saturates */",
     "return sign | 0x7C;"),
    ("no saturation above range", "return sign | fmt_maxcode(fmt);      /* at least 2^(emax+1): saturate */",
     "return sign | 0x7F;"),
    ("NaN sign kept", "return 0x7F;                         /* NaN */", "return sign | 0x7F;"),
    ("scale ignored in cast", "const float p = x[i] * scale;", "const float p = x[i];"),
    ("amax keeps sign", "const float a = fabsf(x[i]);", "const float a = x[i];"),
    ("history not rolled", "hist[j] = hist[j - 1];", "hist[j] = hist[j];"),
    ("most_recent picks the oldest", "a = (L >= 1) ? hist[0] : *cur_amax;", "a = hist[L - 1];"),
    ("margin sign", "ldexp(1.0, -margin)", "ldexp(1.0, margin)"),
    ("scale_inv not inverted", "*scale_inv = 1.0f / *scale;", "*scale_inv = *scale;"),
    ("infinite scale accepted", "if (isfinite(s2) && s2 > 0.0f)", "if (s2 > 0.0f)"),
    ("transposed B in GEMM", "const double p = ad[k] * bj[k];",
     "const double p = ad[k] * bd[(k % rows_b) * kc + (j % kc)];"),
    ("dropped scale in GEMM", "s * sinv_a * sinv_b + (bias ? bias[j] : 0.0)", "s * sinv_a + (bias ? bias[j] : 0.0)"),
    ("dropped bias", "s * sinv_a * sinv_b + (bias ? bias[j] : 0.0)", "s * sinv_a * sinv_b"),
    ("update sign", "fmaf(neg_lr, vn, w[i])", "fmaf(lr, vn, w[i])"),
    ("dropped gradient", "fmaf(mu, v[i], u)", "fmaf(mu, v[i], 0.0f)"),
    ("momentum ignored", "fmaf(mu, v[i], u)", "u + 0.0f * mu"),
    ("no unscale", "bf16_to_f32(g[i]) * inv_s", "bf16_to_f32(g[i])"),
    ("no backoff", "*S = *S * backoff;", "*S = *S;"),
    ("growth never resets", "        *growth = 0;\n    }\n}", "    }\n}"),
    ("recast ignores scale_w", "orc_encode(ORC_E4M3, wn * scale_w)", "orc_encode(ORC_E4M3, wn)"),
    ("recast as E5M2", "orc_encode(ORC_E4M3, wn * scale_w)", "orc_encode(ORC_E5M2, wn * scale_w)"),
    ("NaN gradient missed", "if ((g[i] & 0x7F80u) == 0x7F80u)", "if (g[i] == 0x7F80u)"),
    ("Adam second moment uses u", "const float uu = u * u;", "const float uu = u;"),
    ("Adam without bias correction", "const float mh = mn / bc1;", "const float mh = mn;"),
    ("Adam eps inside the sqrt", "const float den = sqrtf(vh) + eps;", "const float den = sqrtf(vh + eps);"),
    ("Adam step count advances on skips", "        *S = *S * backoff;\n        *growth = 0;\n        return;\n    }\n    const float inv_s = 1.0f / *S;\n    const float b1t",
     "        *S = *S * backoff;\n        *growth = 0;\n        *b1p = *b1p * beta1;\n        return;\n    }\n    const float inv_s = 1.0f / *S;\n    const float b1t"),
    ("dbias sums a transposed view", "((const uint16_t *)dy)[r * cols + c]", "((const uint16_t *)dy)[c * rows + r]"),
    ("dbias drops its last row", "for (int64_t r = 0; r < rows; ++r) {\n            const double v = is_bf16",
     "for (int64_t r = 0; r + 1 < rows; ++r) {\n            const double v = is_bf16"),
]


def _pins():
    """(name, callable) for every pin, with parameters bound."""
    p = []
    for f in (0, 1):
        p += [
            (f"decoder_torch[{f}]", lambda f=f: codec.test_decoder_matches_torch_dtype_on_all_codes(oracle, f)),
            (f"roundtrip[{f}]", lambda f=f: codec.test_roundtrip_every_finite_code(oracle, f)),
            (f"brute_boundaries[{f}]", lambda f=f: codec.test_encoder_brute_force_boundaries(oracle, f)),
            (f"scaled_cast_torch[{f}]", lambda f=f: sc.test_scaled_cast_vs_torch(oracle, f)),
        ]
    p += [
        ("finfo", lambda: codec.test_finfo_table_from_page(oracle)),
        ("worked_cast", lambda: codec.test_worked_cast_example_from_page(oracle)),
        ("special", lambda: codec.test_special_values(oracle)),
        ("saturate_scaled", lambda: sc.test_cast_saturates_under_scale(oracle)),
        ("amax", lambda: sc.test_amax_definition(oracle)),
        ("scale_golden", lambda: sc.test_scale_sequences_from_hand_derivation(oracle)),
        ("margin_degenerate", lambda: sc.test_margin_and_degenerate_amax(oracle)),
        ("gemm_fraction", lambda: gm.test_gemm_exact_rational_tiny(oracle, 0, 0)),
        ("gemm_matmul", lambda: gm.test_gemm_vs_library_matmul(oracle, 1, 0)),
        ("gemm_bias", lambda: gm.test_gemm_row_selection_and_bias(oracle)),
        ("master_hand", lambda: gm.test_master_step_hand_example(oracle)),
        ("master_skip", lambda: gm.test_master_step_overflow_skips_and_backs_off(oracle)),
        ("master_growth", lambda: gm.test_master_step_growth_after_interval(oracle)),
        ("master_nan_alone", lambda: gm.test_master_step_each_nonfinite_kind_alone_skips(oracle, 0xFFC1)),
        ("master_neginf_alone", lambda: gm.test_master_step_each_nonfinite_kind_alone_skips(oracle, 0xFF80)),
        ("master_torch_sgd", lambda: gm.test_master_step_vs_torch_sgd_momentum(oracle)),
        ("dbias", lambda: sc.test_dbias_definition(oracle)),
        ("adam_first", lambda: gm.test_adam_first_step_is_sign_descent(oracle)),
        ("adam_torch", lambda: gm.test_adam_vs_torch_optim_adam(oracle)),
        ("adam_skip", lambda: gm.test_adam_skip_step_keeps_everything(oracle)),
        ("current_scaling", lambda: sc.test_current_scaling_maps_amax_to_fmt_max(oracle)),
    ]
    return p


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="orc_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_unmutated_passes_every_pin(orc):
    for name, fn in _pins():
        fn()


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(orc, mutant_dir, label, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fp8_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    tag = "".join(ch if ch.isalnum() else "_" for ch in label)
    c_path = os.path.join(mutant_dir, tag + ".c")
    so_path = os.path.join(mutant_dir, tag + ".so")
    with open(c_path, "w") as f:
        f.write(mutated)
    r = subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", c_path,
                        "-o", so_path, "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    failed = []
    with oracle.swapped_library(so_path):
        for name, fn in _pins():
            try:
                with np.errstate(all="ignore"):
                    fn()
            except (AssertionError, ValueError, IndexError):
                failed.append(name)
    assert failed, f"no pin caught the planted mistake: {label}"
