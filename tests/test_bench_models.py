"""The algorithmic byte models bench.py reports rooflines with, checked on
small workloads against a plain loop over samples and corners: the number of
in-level (sample, corner) pairs (per-corner model) and of distinct value rows
(unique model), on the binary32 pixel coordinate the kernels use."""
import importlib.util
import math
import os
import sys

import numpy as np
import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def loop_counts(wl, inp):
    loc = W.to_f64(inp["sampling_locations"], wl.dtype)
    starts = W.level_start_index(wl.shapes)
    B, Q, M = loc.shape[:3]
    n, rows = 0, set()
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                for l, (h, w) in enumerate(wl.shapes):
                    for k in range(wl.K):
                        x = math.floor(float(np.float32(loc[b, q, m, l, k, 0] * w - 0.5)))
                        y = math.floor(float(np.float32(loc[b, q, m, l, k, 1] * h - 0.5)))
                        for dy in (0, 1):
                            for dx in (0, 1):
                                if 0 <= x + dx < w and 0 <= y + dy < h:
                                    n += 1
                                    rows.add(((b * wl.S + starts[l] + (y + dy) * w + x + dx) * M + m))
    return n, len(rows)


@pytest.mark.parametrize("name,over", [("tiny_fp32", {}), ("tiny_fp32", {"dtype": "bf16", "B": 2, "Q": 33, "M": 3}),
                                       ("decoder_bf16", {"B": 1, "Q": 7})])
def test_corner_counts_match_a_loop(bench, name, over):
    wl = W.WORKLOADS[name].with_(**over) if over else W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    assert bench.corner_counts(wl, inp) == loop_counts(wl, inp)


def test_byte_model_formula(bench):
    wl = W.WORKLOADS["decoder_bf16"]
    es = 2
    corners, rows = 596431, 265129
    m = bench.byte_model(wl, corners, rows)
    samples = wl.B * wl.Qn * wl.M * wl.L * wl.K
    out = wl.B * wl.Qn * wl.M * wl.D * es
    n_value = wl.B * wl.S * wl.M * wl.D
    assert m["forward"] == corners * wl.D * es + samples * 3 * es + out
    assert m["backward"] == 2 * corners * wl.D * es + out + 2 * samples * 3 * es
    assert m["bwd_total"] == m["backward"] + n_value * es
    assert m["forward_unique"] == rows * wl.D * es + samples * 3 * es + out
    assert m["bwd_total_unique"] == rows * wl.D * es + out + 2 * samples * 3 * es + n_value * es


def test_bound_labels(bench):
    """The roofline's bound names the ceiling that binds: HBM when value (or the
    fp32 accumulator) exceeds the L2, else the L2 (its reduction rate for the
    backward)."""
    l2 = 126 << 20
    stress = W.WORKLOADS["stress_bf16"]
    decoder = W.WORKLOADS["decoder_bf16"]
    assert bench.bound_of("backward", stress, "fp32", l2) == "hbm"
    assert bench.bound_of("forward", stress, "fp32", l2) == "hbm"
    assert bench.bound_of("backward", decoder, "native", l2) == "l2_reductions"
    assert bench.bound_of("forward", decoder, "native", l2) == "l2"
    assert bench.bound_of("zero", decoder, "fp32", l2) == "l2"
    assert bench.bound_of("convert", stress, "fp32", l2) == "hbm"


def test_oracle_sample_is_batch0_prefix(bench):
    wl = W.WORKLOADS["decoder_bf16"].with_(B=2, Q=10)
    inp = W.make_inputs(wl)
    sub, q, units = bench.oracle_sample(wl, inp, 4.7)
    assert q == 4 and units == 4 * wl.M
    assert sub["value"].shape[0] == 1 and sub["sampling_locations"].shape[:2] == (1, 4)
    assert np.array_equal(sub["grad_out"], inp["grad_out"][:1, :4])
    assert bench.oracle_sample(wl, inp, 1e9)[1] == wl.Qn


def test_fp32_backward_roofline_group(bench):
    """With the FP32 accumulator the roofline takes the backward whole: the
    backward kernel's, the rounding's and the touch count's bytes over the wall
    time of the backward call (its kernels overlap on two streams), not the sum
    of the traced kernel times; the compulsory fraction uses that wall time too."""
    wl = W.WORKLOADS["stress_bf16"]
    model = bench.byte_model(wl, corners=80_000_000, unique_rows=28_000_000)
    kernels = {"forward": {"launches": 4, "avg_ms": 0.8, "ms_per_step": 0.8, "steps": 4},
               "touch_count": {"launches": 4, "avg_ms": 0.2, "ms_per_step": 0.2, "steps": 4},
               "backward": {"launches": 16, "avg_ms": 1.0, "ms_per_step": 4.0, "steps": 4},
               "convert": {"launches": 8, "avg_ms": 1.0, "ms_per_step": 2.0, "steps": 4}}
    per = {k: [v["avg_ms"]] * v["launches"] for k, v in kernels.items()}
    r = bench.roofline_of("backward", per, wl, model, "fp32", 126 << 20, kernels, bwd_wall_ms=4.1)
    alg = model["backward"] + model["convert"] + model["touch_count"]
    assert r["kernel"] == "backward+convert" and r["algorithmic_bytes"] == alg
    assert r["ms_per_step"] == 4.1 and r["launches_per_step"] == 7.0
    assert math.isclose(r["achieved"], alg / 4.1e-3 / 1e9, rel_tol=1e-4)
    assert "wall time" in r["time_source"]
    # without the wall time: the traced kernels' sum
    r2 = bench.roofline_of("backward", per, wl, model, "fp32", 126 << 20, kernels)
    assert r2["ms_per_step"] == 6.2 and "time_source" not in r2
    uf = bench.unique_fractions(model, kernels, 6781.1, 4.1)
    assert math.isclose(uf["backward_frac"], model["bwd_total_unique"] / 4.1e-3 / 1e9 / 6781.1, rel_tol=1e-3)
