"""Plants one plausible mistake at a time in a copy of the oracle (on the CPU)
and checks that the pins catch every one of them.

The copies are compiled into a temporary directory; the real oracle source is
only read.
"""
import os

import pytest

import oracle
from tests import oracle_pins

# (name, text in fnorm_oracle.cpp, replacement)
MUTANTS = [
    ("unbiased_variance", "*var = q / static_cast<double>(n);",
     "*var = q / static_cast<double>(n - 1);"),
    ("dropped_eps", "return (v - mean) / std::sqrt(var + eps);",
     "return (v - mean) / std::sqrt(var);"),
    ("sign_flip", "return (v - mean) / std::sqrt(var + eps);",
     "return (mean - v) / std::sqrt(var + eps);"),
    ("eps_outside_sqrt", "return (v - mean) / std::sqrt(var + eps);",
     "return (v - mean) / (std::sqrt(var) + eps);"),
    ("clamp_order", "return std::fmin(std::fmax(t, lo), hi);",
     "return std::fmax(std::fmin(t, hi), lo) * 0.999;"),
    ("dropped_premultiply", "v[s] = static_cast<double>(xs[s]) * mc;",
     "v[s] = static_cast<double>(xs[s]);"),
    ("dropped_postmultiply", "z[c * S + s] = static_cast<float>(mc * clamp(",
     "z[c * S + s] = static_cast<float>(1.0 * clamp("),
    ("argmax_last_tie", "if (zc > best) {", "if (zc >= best) {"),
    ("bn_transposed_index", "v[n * S + s] = static_cast<double>(x[(n * C + c) * S + s]);",
     "v[n * S + s] = static_cast<double>(x[(c * N + n) * S + s]);"),
    ("bn_momentum_swapped",
     "running_mean[c] = (1.0 - momentum) * running_mean[c] + momentum * mean;",
     "running_mean[c] = momentum * running_mean[c] + (1.0 - momentum) * mean;"),
    ("bn_running_var_biased",
     "const double unbiased = var * static_cast<double>(cnt) / static_cast<double>(cnt - 1);",
     "const double unbiased = var;"),
    ("bn_scale_before_beta",
     "static_cast<float>(scale * (g * normalize(v[n * S + s], mean, var, eps) + b));",
     "static_cast<float>(scale * g * normalize(v[n * S + s], mean, var, eps) + b);"),
    ("in_affine_beta_inside", "y[q * S + i] = g * normalize(v[i], mean, var, eps) + b;",
     "y[q * S + i] = g * (normalize(v[i], mean, var, eps) + b);"),
    ("in_affine_swapped", "y[q * S + i] = g * normalize(v[i], mean, var, eps) + b;",
     "y[q * S + i] = b * normalize(v[i], mean, var, eps) + g;"),
    ("bn_eval_scale_before_beta",
     "scale * (g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);",
     "scale * g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b;"),
    ("bn_eval_stats_swapped",
     "scale * (g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);",
     "scale * (g * normalize(x[base + s], running_var[c], running_mean[c], eps) + b);"),
    ("bn_eval_dropped_scale",
     "scale * (g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);",
     "(g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);"),
    ("in_affine_wrong_channel",
     "if (S > 0) moments(v.data(), S, &mean, &var);\n      const double g = gamma ? gamma[c] : 1.0;",
     "if (S > 0) moments(v.data(), S, &mean, &var);\n      const double g = gamma ? gamma[(c + 1) % C] : 1.0;"),
    ("bn_eval_affine_swapped",
     "scale * (g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);",
     "scale * (b * normalize(x[base + s], running_mean[c], running_var[c], eps) + g);"),
    ("bf16_truncate", "const double r = std::nearbyint(q);", "const double r = std::trunc(q);"),
    ("bf16_ties_away", "const double r = std::nearbyint(q);", "const double r = std::round(q);"),
]


def _fails_some_pin(orc) -> list:
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except Exception:  # AssertionError, or a crash the mistake causes
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant_src = tmp_path / "mutant.cpp"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutant_src), str(tmp_path / "libmutant.so"))
    caught = _fails_some_pin(oracle.Oracle(lib))
    assert caught, f"no pin catches the planted mistake {name}"


def test_real_oracle_passes_every_pin(orc):
    assert _fails_some_pin(orc) == []
    assert os.path.exists(oracle.LIBRARY)
