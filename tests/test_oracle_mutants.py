"""Plant plausible mistakes in a copy of the C oracle and check that the pins
catch each one: a wrong sign, a swapped index or axis, a dropped factor or
term, an off-by-one bound, trunc for floor, the fp64 coordinate in place of the
binary32 one, and in the fused locations a sum taken before the division,
(H, W) for (W, H), one rounding in place of two, or a flipped offset.  CPU
only."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "msda_oracle.c")

# (name, text to find, replacement); each text must occur exactly once
MUTANTS = [
    ("offset_sign_fp64", "x_im = x * (double)s->W - 0.5;", "x_im = x * (double)s->W + 0.5;"),
    ("offset_sign_fp32", "x_im = (double)fmaf((float)x, (float)s->W, -0.5f);",
     "x_im = (double)fmaf((float)x, (float)s->W, 0.5f);"),
    ("weight_swap_y", "double wy = i ? s->ly : 1.0 - s->ly;", "double wy = i ? 1.0 - s->ly : s->ly;"),
    ("weight_swap_x", "double wx = j ? s->lx : 1.0 - s->lx;", "double wx = j ? 1.0 - s->lx : s->lx;"),
    ("hw_swap", "s->H = P->shapes[2 * l];\n    s->W = P->shapes[2 * l + 1];",
     "s->W = P->shapes[2 * l];\n    s->H = P->shapes[2 * l + 1];"),
    ("loc_xy_swap", "double x = load_el(P->loc, 2 * p, P->pdt);\n    double y = load_el(P->loc, 2 * p + 1, P->pdt);",
     "double y = load_el(P->loc, 2 * p, P->pdt);\n    double x = load_el(P->loc, 2 * p + 1, P->pdt);"),
    ("gloc_drop_attn", "gloc[2 * sl] = s.a * (double)s.W * gx;", "gloc[2 * sl] = (double)s.W * gx;"),
    ("gloc_y_scale", "gloc[2 * sl + 1] = s.a * (double)s.H * gy;", "gloc[2 * sl + 1] = s.a * (double)s.W * gy;"),
    ("dwdx_sign", "s->dwdx[i][j] = wy * (j ? 1.0 : -1.0);", "s->dwdx[i][j] = wy * (j ? -1.0 : 1.0);"),
    ("dwdy_drop_weight", "s->dwdy[i][j] = wx * (i ? 1.0 : -1.0);", "s->dwdy[i][j] = (i ? 1.0 : -1.0);"),
    ("bound_off_by_one", "(xx < (double)s->W)", "(xx <= (double)s->W)"),
    ("trunc_for_floor", "double x0 = floor(x_im), y0 = floor(y_im);", "double x0 = trunc(x_im), y0 = trunc(y_im);"),
    ("ignore_level_start", "start + (int64_t)yy * s->W + (int64_t)xx", "(int64_t)yy * s->W + (int64_t)xx"),
    ("value_transposed", "return ((b * P->S + row) * P->M + m) * P->D;", "return ((b * P->M + m) * P->S + row) * P->D;"),
    ("gattn_drop_weight", "ga += s.w[i][j] * dot;", "ga += dot;"),
    ("scatter_drop_weight", "double c = s.a * s.w[i][j];\n                        for (int64_t d = 0; d < D; ++d) gv[",
     "double c = s.a;\n                        for (int64_t d = 0; d < D; ++d) gv["),
    ("fwd_drop_attn", "double c = s.a * s.w[i][j];\n                    int64_t vi",
     "double c = s.w[i][j];\n                    int64_t vi"),
    ("fp32_mode_ignored", "if (P->coord_mode == 1) {", "if (0) {"),
    ("unit_q_index", "int64_t p = (((b * P->Q + q) * P->M + m) * P->L + l) * P->K + k;",
     "int64_t p = (((b * P->Q + q) * P->M + m) * P->L + k) * P->K + l;"),
    # fused locations in binary32 (coord_mode 1)
    ("fused_sum_before_divide", "float quot = (float)o / (float)size[c];\n                                float sum = (float)r[c] + quot;",
     "float sum = ((float)r[c] + (float)o) / (float)size[c];"),
    ("fused_divide_by_hw", "float quot = (float)o / (float)size[c];", "float quot = (float)o / (float)size[1 - c];"),
    ("fused_one_rounding", "float quot = (float)o / (float)size[c];\n                                float sum = (float)r[c] + quot;",
     "float sum = (float)(r[c] + o / size[c]);"),
    ("fused_offset_sign", "float sum = (float)r[c] + quot;", "float sum = (float)r[c] - quot;"),
]


def _build_mutant(tmp, name, find, repl):
    src = open(SRC).read()
    assert src.count(find) == 1, f"mutant {name}: pattern occurs {src.count(find)} times"
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"lib_{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(find, repl))
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", path_c,
                    "-o", path_so, "-lm"], check=True)
    return path_so


_CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[2])
import oracle, pins
caught = []
with oracle.using_library(sys.argv[3]):
    for pin in pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
print("caught:", caught)
sys.exit(3 if caught else 0)
"""


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, find, repl):
    """A mutant is caught when some pin fails or the planted mistake crashes
    the child process (e.g. an out-of-bounds read)."""
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(tests_dir)
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, name, find, repl)
        r = subprocess.run([sys.executable, "-c", _CHILD, root, tests_dir, so], capture_output=True, text=True,
                           timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake {name!r}: {r.stdout[-500:]}"
