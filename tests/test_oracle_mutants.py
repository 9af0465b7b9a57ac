"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of oracle/adaln_oracle.cpp with one plausible mistake
(a dropped term, a wrong sign, a wrong index or normaliser, swapped operands),
compiled on the CPU into a temporary library; the pins of tests/pins.py are
then run against it and at least one must fail.  This shows the pins constrain
every part of the oracle, rather than the oracle checking itself.
"""
import os

import pytest

import oracle
from oracle import build as obuild
import pins

# (name, exact text in the oracle source, replacement)
MUTANTS = [
    ("dx_drops_mean_g", "(g[d] - mean_g - xhat[d] * mean_gx)", "(g[d] - xhat[d] * mean_gx)"),
    ("dx_sign_of_proj", "(g[d] - mean_g - xhat[d] * mean_gx)", "(g[d] - mean_g + xhat[d] * mean_gx)"),
    ("dx_drops_rstd", "dx[i * D + d] = rs[t] * (", "dx[i * D + d] = ("),
    ("dx_mean_gx_not_normalised", "mean_gx /= D;", ""),
    ("dx_xhat_not_scaled", "xhat[d] = (elem(x, dtype, t * D + d) - mu[t]) * rs[t];",
     "xhat[d] = (elem(x, dtype, t * D + d) - mu[t]);"),
    ("dx_g_without_one_plus", "g[d] = elem(dy, dtype, t * D + d) * (1.0 + elem(scale, dtype, b * D + d));",
     "g[d] = elem(dy, dtype, t * D + d) * elem(scale, dtype, b * D + d);"),
    ("var_unbiased", "s += c * c;\n  }\n  return s / D;", "s += c * c;\n  }\n  return s / (D - 1);"),
    ("mean_wrong_normaliser", "s += elem(x, dtype, t * D + d);\n  return s / D;",
     "s += elem(x, dtype, t * D + d);\n  return s / (D + 1);"),
    ("eps_outside_sqrt", "1.0 / std::sqrt(var + eps)", "1.0 / (std::sqrt(var) + eps)"),
    ("y_without_one_plus", "xhat * (1.0 + sc) + sh", "xhat * sc + sh"),
    ("y_scale_shift_swapped", "const double sc = elem(scale, dtype, b * D + d);",
     "const double sc = elem(shift, dtype, b * D + d);"),
    ("y_shift_segment_zero", "const double sh = elem(shift, dtype, b * D + d);",
     "const double sh = elem(shift, dtype, 0 * D + d);"),
    ("dscale_uses_x", "dscale[b * D + d] += dyv * xhat;",
     "dscale[b * D + d] += dyv * elem(x, dtype, t * D + d);"),
    ("dshift_dscale_swapped", "if (dshift) dshift[b * D + d] += dyv;",
     "if (dshift) dshift[b * D + d] += dyv * (elem(x, dtype, t * D + d) - mu[t]) * rs[t];"),
    ("bf16_widening_shift", "<< 16;", "<< 15;"),
]


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not unique/present"
    src = tmp_path / f"{name}.cpp"
    src.write_text(source.replace(old, new))
    # the oracle header sits beside the original source
    lib_path = obuild.compile_oracle(str(src), str(tmp_path / f"lib{name}.so"),
                                     extra=("-I" + os.path.dirname(obuild.SRC),))
    lib = oracle.load(lib_path)
    caught = []
    for pin in pins.ALL:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught mutant {name}"
