"""The pins are strong enough: each plausible slip planted in a copy of the
oracle's C source (on the CPU, in a temporary directory) makes at least one
pin of ``test_oracle_pins.py`` fail."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("eps_outside_root", "1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    ("sum_not_mean", "double ms = sum_sq / (double)hidden;", "double ms = sum_sq;"),
    ("scale_not_one_plus_scale", "y[t * hidden + j] = n * (1.0 + s) + b;", "y[t * hidden + j] = n * s + b;"),
    ("shift_subtracted", "y[t * hidden + j] = n * (1.0 + s) + b;", "y[t * hidden + j] = n * (1.0 + s) - b;"),
    ("shift_before_scale", "y[t * hidden + j] = n * (1.0 + s) + b;", "y[t * hidden + j] = (n + b) * (1.0 + s);"),
    ("norm_weight_dropped", "double n = oracle_bf16_to_f64(xr[j]) * inv_rms * (double)weight[j];",
     "double n = oracle_bf16_to_f64(xr[j]) * inv_rms;"),
    ("mod_row_ignored", "double s = (double)scale[(int64_t)m * hidden + j];", "double s = (double)scale[j];"),
    ("head_norm_over_whole_row", "double inv_rms = 1.0 / sqrt(sum_sq / (double)head_dim + eps);",
     "double inv_rms = 1.0 / sqrt(sum_sq / (double)(head_dim * n_heads) + eps);"),
    ("head_weight_dropped", "oh[d] = oracle_bf16_to_f64(vh[d]) * inv_rms * (double)weight[d];",
     "oh[d] = oracle_bf16_to_f64(vh[d]) * inv_rms;"),
    ("rope_first_sign", "vh[i] = a * c - b * s;", "vh[i] = a * c + b * s;"),
    ("rope_second_sign", "vh[i + half] = b * c + a * s;", "vh[i + half] = b * c - a * s;"),
    ("rope_freq_exponent", "-(2.0 * (double)i) / (double)head_dim", "-((double)i) / (double)head_dim"),
    ("rope_cos_sin_swapped", "double c = cos(angle), s = sin(angle);", "double c = sin(angle), s = cos(angle);"),
    ("rope_interleaved_pairs", "double a = vh[i], b = vh[i + half];", "double a = vh[2 * (i % (half / 2 > 0 ? half / 2 : 1))], b = vh[i + half];"),
    ("qk_weights_swapped", "oracle_head_rmsnorm(k, in_row_stride, rows, n_heads, head_dim, k_weight, eps, k_out);",
     "oracle_head_rmsnorm(k, in_row_stride, rows, n_heads, head_dim, q_weight, eps, k_out);"),
    ("swiglu_halves_swapped", "double g = oracle_bf16_to_f64(r[j]);\n            double u = oracle_bf16_to_f64(r[ffn + j]);",
     "double g = oracle_bf16_to_f64(r[ffn + j]);\n            double u = oracle_bf16_to_f64(r[j]);"),
    ("silu_sign", "double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    ("merge_negative_zero_tail", ": (uint16_t)0x0000;", ": (uint16_t)0x8000;"),
    ("gather_off_by_one", "for (int64_t i = 0; i < valid_rows; ++i)\n        for (int32_t j = 0; j < hidden; ++j)\n            compact",
     "for (int64_t i = 0; i + 1 < valid_rows; ++i)\n        for (int32_t j = 0; j < hidden; ++j)\n            compact"),
    ("rope_one_middle_frequency", "double angle = (double)pos[t] * inv_freq;",
     "double angle = (double)pos[t] * (i == 37 ? inv_freq * 1.001 : inv_freq);"),
    ("rope_last_pair_unrotated", "double c = cos(angle), s = sin(angle);",
     "double c = i == half - 1 ? 1.0 : cos(angle), s = i == half - 1 ? 0.0 : sin(angle);"),
    ("adaln_last_column_unmodulated", "y[t * hidden + j] = n * (1.0 + s) + b;",
     "y[t * hidden + j] = j == hidden - 1 ? n : n * (1.0 + s) + b;"),
    ("round_half_up", "double n = rint(a / quantum);", "double n = floor(a / quantum + 0.5);"),
    ("round_truncates", "double n = rint(a / quantum);", "double n = floor(a / quantum);"),
]

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and n != "test_workload_recipes"]


def _run_pins() -> list:
    failed = []
    for t in PIN_TESTS:
        try:
            params = getattr(t, "pytestmark", [])
            args_list = [()]
            for m in params:
                if m.name == "parametrize":
                    args_list = [(v,) for v in m.args[1]]
            for args in args_list:
                t(*args)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(t.__name__)
        except pytest.skip.Exception:
            pass
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mutant.c")
        so = os.path.join(d, "libmutant.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
        saved = oracle._load()
        oracle._lib = oracle.bind(so)
        try:
            failed = _run_pins()
        finally:
            oracle._lib = saved
    assert failed, f"no pin caught the planted mistake {name}"
