"""The oracle's pins bite: plant one plausible mistake at a time in a copy of
the oracle source (on the CPU, in a temporary directory), rebuild it, and
check that at least one pin fails for every planted mistake.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import build as obuild

import test_oracle_pins as pins
import test_oracle_scale_rot as sr_pins
import test_oracle_absgrad as abs_pins
import test_oracle_render_scale as scale_pins
import test_oracle_merge as merge_pins

# (name, text in the oracle source, replacement)
MUTATIONS = [
    ("fp32 off-diagonal sign", "const float B = -(t * C);", "const float B = (t * C);"),
    ("double off-diagonal sign", "*B = -sxy / det;", "*B = sxy / det;"),
    ("dropped one half in the weight", "return exp(-0.5 * q);", "return exp(-q);"),
    ("transposed Cholesky (b<->c in Syy)", "syy = b * b + c * c;", "syy = a * a + c * c;"),
    ("box radius from the wrong factor", "const float rx = k * fabsf(a);",
     "const float rx = k * fabsf(c);"),
    ("tile rectangle end from the start", "rc[2] = b4[2] / cfg->tile;", "rc[2] = b4[0] / cfg->tile;"),
    ("mean gradient uses C for B", "const double gx = dq * (-2.0) * (A * dx + B * dy);",
     "const double gx = dq * (-2.0) * (A * dx + C * dy);"),
    ("chain rule dA/da halved", "dchol[0] = dA * (-2.0 * A / a)", "dchol[0] = dA * (-1.0 * A / a)"),
    ("chain rule dC/dc sign", "dC * (-2.0 / (c * c * c));", "dC * (2.0 / (c * c * c));"),
    ("composite: no division by 1-alpha", "S[d] / (1.0 - e->alpha)", "S[d]"),
    ("composite: background dropped", "C[d] += T * s->bg[d];", "C[d] += 0.0 * s->bg[d];"),
    ("composite: transmittance from opacity", "T *= (1.0 - alpha);", "T *= (1.0 - s->opacity[g]);"),
    ("composite: no early termination", "if (T < (double)cfg->t_min) break;", "if (T < 0.0) break;"),
    ("loss gradient without the 2", "d_image[k] = 2.0 * e / (double)m;", "d_image[k] = e / (double)m;"),
    ("scale-rot: fp32 off-diagonal sign", "const float B = cs * (u - v);",
     "const float B = cs * (v - u);"),
    ("scale-rot: double A with the axes swapped", "*A = c * c * u + s * s * v;",
     "*A = s * s * u + c * c * v;"),
    ("scale-rot: box radius from the other axis", "const float rx = k * sqrtf(fmaf(cc, sx2, ss * sy2));",
     "const float rx = k * sqrtf(fmaf(ss, sx2, cc * sy2));"),
    ("scale-rot: rotation gradient sign", "dchol[2] = dA * (-2.0 * B)", "dchol[2] = dA * (2.0 * B)"),
    ("scale-rot: s_y gradient from s_x", "(-2.0 / (sy * sy * sy));", "(-2.0 / (sx * sy * sy));"),
    ("fp32 sin: wrong Taylor coefficient", "p = fmaf(p, r2, -1.66666672e-01f);",
     "p = fmaf(p, r2, -1.66666672e-02f);"),
    ("fp32 sincos: quadrant sign", "case 1: *sn = c; *cs = -s; break;", "case 1: *sn = c; *cs = s; break;"),
    ("absgrad: signed instead of absolute", "g->dmu_abs[0] += fabs(gx);", "g->dmu_abs[0] += gx;"),
    ("absgrad: y from x", "g->dmu_abs[1] += fabs(gy);", "g->dmu_abs[1] += fabs(gx);"),
    ("render scale: mean not scaled in the mask", "const float dx = ((float)j + 0.5f) - sc * xy[0];",
     "const float dx = ((float)j + 0.5f) - xy[0];"),
    ("render scale: gradient not scaled back", "dxy[0] = sc * g->dmu[0];", "dxy[0] = g->dmu[0];"),
    ("merge: weight from the partner's area", "double wi = ri * (fabs", "double wi = rj * (fabs"),
    ("merge: spread term transposed", "(wi * (Si[0] + di0 * di0)", "(wi * (Si[0] + di0 * di1)"),
    ("merge: colour mass over the wrong area", "(double)cj[d] * rj) / r);", "(double)cj[d] * rj) / ri);"),
    ("merge: cost cross-term sign", "((m2 * dx) * dx - ((2.0f * m1) * dx) * dy)",
     "((m2 * dx) * dx + ((2.0f * m1) * dx) * dy)"),
    ("merge: pairs not mutual", "if (j > i && nn[j] == i) {", "if (j > i) {"),
    ("merge: cost with the sum of the covariances, not their mean",
     "const float m0 = 0.5f * (Si[0] + Sj[0]), m1 = 0.5f * (Si[1] + Sj[1]), m2 = 0.5f * (Si[2] + Sj[2]);",
     "const float m0 = (Si[0] + Sj[0]), m1 = (Si[1] + Sj[1]), m2 = (Si[2] + Sj[2]);"),
    ("merge: cost with one Gaussian's covariance only",
     "const float m0 = 0.5f * (Si[0] + Sj[0]), m1 = 0.5f * (Si[1] + Sj[1]), m2 = 0.5f * (Si[2] + Sj[2]);",
     "const float m0 = Si[0], m1 = Si[1], m2 = Si[2];"),
    ("composite lists not depth sorted", "if (cfg->mode == REF_MODE_COMPOSITE) {\n      g_sort_depth = depth;\n      for",
     "if (0) {\n      g_sort_depth = depth;\n      for"),
]

PINS = [
    pins.test_golden_single_gaussian_values,
    pins.test_golden_composite_values,
    pins.test_single_gaussian_matches_library_density,
    pins.test_pixel_box_formula,
    lambda: pins.test_tile_lists_by_brute_force(oracle.SUM),
    lambda: pins.test_tile_lists_by_brute_force(oracle.COMPOSITE),
    lambda: pins.test_tiled_equals_brute_force(40, 33, 64, oracle.SUM),
    lambda: pins.test_tiled_equals_brute_force(40, 33, 64, oracle.COMPOSITE),
    pins.test_composite_early_termination,
    pins.test_composite_depends_on_depth_order,
    pins.test_sum_gradients_by_central_differences,
    pins.test_composite_gradients_by_central_differences,
    pins.test_loss_gradient_by_central_differences,
    sr_pins.test_fp32_sincos_accuracy,
    sr_pins.test_single_gaussian_matches_library_density,
    sr_pins.test_pixel_box_is_the_ellipse_box,
    sr_pins.test_sum_gradients_by_central_differences,
    lambda: abs_pins.test_absgrad_by_per_pixel_central_differences(oracle.SUM, oracle.CHOLESKY),
    abs_pins.test_triangle_inequality_and_culled_zero,
    lambda: scale_pins.test_peak_keeps_the_colour(2.0),
    lambda: scale_pins.test_same_as_prescaled_parameters(oracle.CHOLESKY),
    lambda: scale_pins.test_gradients_by_central_differences(oracle.CHOLESKY, oracle.SUM),
    merge_pins.test_identical_twins,
    lambda: merge_pins.test_moments_of_the_image_are_kept(oracle.CHOLESKY),
    merge_pins.test_channel_masses_are_kept,
    lambda: merge_pins.test_pairs_are_mutual_nearest_neighbours(oracle.CHOLESKY),
    merge_pins.test_merge_cost_closed_forms,
    merge_pins.test_merge_cost_against_linear_algebra,
]


@pytest.fixture(scope="module")
def source():
    return open(obuild.SRC).read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(source, name, old, new, tmp_path):
    assert source.count(old) == 1, f"mutation anchor not found once: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(lib), str(src), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(lib)):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(getattr(pin, "__name__", "lambda"))
    assert caught, f"no pin caught the planted mistake: {name}"
