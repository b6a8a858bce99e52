"""Planted mistakes in the oracle must each fail at least one pin.

Each case copies oracle/softmax_oracle.c, applies one textual mutation (a
dropped term, a wrong sign, index or stride, a wrong rounding rule), builds the
mutant with gcc into a temporary directory and runs the pins of
test_oracle_pins.py against it.  Mistakes are planted only in copies of the
oracle, on the CPU; the committed oracle is never modified.
"""
import inspect
import os

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "softmax_oracle.c")

MUTANTS = {
    "no_max_subtract": ("y[j] = exp(x[j] - m);", "y[j] = exp(x[j]);"),
    "sum_skips_last": ("l += y[j];", "if (j + 1 < n) l += y[j];"),
    "max_wrong_sign": ("if (x[j] > m)\n            m = x[j];", "if (x[j] < m)\n            m = x[j];"),
    "multiply_not_divide": ("y[j] = y[j] / l;", "y[j] = y[j] * l;"),
    "input_stride_ignored": ("(const float*)in + r * in_row_stride", "(const float*)in + r * n_cols"),
    "output_row_index": ("double* y = out + r * out_row_stride;", "double* y = out + r;"),
    "online_no_rescale": ("l = l * exp(m - m_new) + s;", "l = l + s;"),
    "online_no_inf_guard": ("if (m_new == -INFINITY) {", "if (0) {"),
    "online_rescale_sign": ("l = l * exp(m - m_new) + s;", "l = l * exp(m_new - m) + s;"),
    "bf16_round_ties_away": ("const double n = rint(", "const double n = round("),
    "bf16_round_truncate": ("const double n = rint(", "const double n = trunc("),
    "bf16_decode_shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "bf16_overflow_early": ("if (a >= overflow_at)", "if (a > ldexp(1.0, 127))"),
    "causal_off_by_one": ("return last + 1 < n_cols ? last + 1 : n_cols;",
                          "return last < n_cols ? last : n_cols;"),
    "causal_period_ignored": ("const int64_t last = r % period + offset;",
                              "const int64_t last = r + offset;"),
    "causal_offset_sign": ("const int64_t last = r % period + offset;",
                           "const int64_t last = r % period - offset;"),
    "causal_default_period": ("if (period <= 0)\n        period = n_rows;",
                              "if (period <= 0)\n        period = 1;"),
    "causal_masked_as_zero": ("for (int64_t j = vis; j < n_cols; ++j)\n            x[j] = -INFINITY;",
                              "for (int64_t j = vis; j < n_cols; ++j)\n            x[j] = 0.0;"),
    "scale_dropped_f32": ("x[j] = scale * (double)src[j];", "x[j] = (double)src[j];"),
    "scale_dropped_bf16": ("x[j] = scale * oracle_bf16_to_double(src[j]);",
                           "x[j] = oracle_bf16_to_double(src[j]);"),
    "scale_divides": ("x[j] = scale * (double)src[j];", "x[j] = (double)src[j] / scale;"),
    "f16_decode_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "f16_round_ties_away": ("const double r = ldexp(rint(ldexp(a, -q_exp)), q_exp);",
                            "const double r = ldexp(round(ldexp(a, -q_exp)), q_exp);"),
    "f16_overflow_early": ("if (a >= 65520.0)", "if (a > 65504.0)"),
    "f16_subnormal_spacing": ("if (q_exp < -24)\n        q_exp = -24;", "if (q_exp < -25)\n        q_exp = -25;"),
    "f16_input_decoded_as_bf16": ("x[j] = scale * oracle_f16_to_double(src[j]);",
                                  "x[j] = scale * oracle_bf16_to_double(src[j]);"),
    "backward_no_y_factor": ("dx[r * dx_row_stride + j] = yj * (gj - dot);",
                             "dx[r * dx_row_stride + j] = (gj - dot);"),
    "backward_sign": ("dx[r * dx_row_stride + j] = yj * (gj - dot);",
                      "dx[r * dx_row_stride + j] = yj * (gj + dot);"),
    "backward_dot_without_y": ("dot += load_elem(y, r * y_row_stride + j, dtype) *\n                   load_elem(dy, r * dy_row_stride + j, dtype);",
                               "dot += load_elem(dy, r * dy_row_stride + j, dtype);"),
    "backward_dy_stride": ("const double gj = load_elem(dy, r * dy_row_stride + j, dtype);",
                           "const double gj = load_elem(dy, r * y_row_stride + j, dtype);"),
    "strided_ignores_col_stride": ("const int64_t idx = r * in_row_stride + c * in_col_stride;",
                                   "const int64_t idx = r * in_row_stride + c;"),
    "strided_swaps_strides": ("const int64_t idx = r * in_row_stride + c * in_col_stride;",
                              "const int64_t idx = r * in_col_stride + c * in_row_stride;"),
    "tiled_sum_ragged_lane": ("if (t0 + i < n)         /* masked lanes load 0 */",
                              "if (t0 + i <= n)"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = list(inspect.signature(fn).parameters)
        if params == ["oracle_lib"]:
            out.append((name, fn, {}))
        elif params == ["oracle_lib", "tile"]:
            for t in (1, 3, 64):
                out.append(("%s[%d]" % (name, t), fn, {"tile": t}))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path):
    before, after = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(before) >= 1, "mutation anchor vanished from the oracle: " + mutant
    mutated = src.replace(before, after)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.Oracle(oracle.build(force=True, src=str(path), out=str(tmp_path / "mutant.so")))
    caught = []
    for name, fn, kw in _pin_functions():
        try:
            fn(lib, **kw)
        except pytest.skip.Exception:
            continue
        except Exception:               # AssertionError, or a crash-free ValueError
            caught.append(name)
    assert caught, "no pin fails on planted mistake " + mutant


def test_unmutated_oracle_passes_every_pin(oracle_lib):
    for name, fn, kw in _pin_functions():
        fn(oracle_lib, **kw)
