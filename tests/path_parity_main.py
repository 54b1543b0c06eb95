"""Compact forward + backward parity check against the oracle, run by
test_gpu_kernel_paths.py in a child process whose MSDA_TUNE forces one kernel
family (the library reads MSDA_TUNE once per process)."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from msda_testutil import assert_forward, assert_grad, f64, to_torch  # noqa: E402


def main():
    import torch

    import scale_deformable_attention_gb300 as msda

    cases = [
        ("bf16", 32, 4, "native"), ("bf16", 32, 2, "fp32"), ("f16", 64, 8, "native"), ("f32", 48, 4, "auto"),
        ("bf16", 96, 1, "native"), ("f32", 32, 8, "auto"), ("bf16", 32, 4, "deterministic"),
        ("f32", 48, 2, "deterministic"), ("f16", 64, 4, "fp32"), ("bf16", 96, 2, "fp32"),
        ("bf16", 32, 4, "fp32"), ("f16", 32, 4, "native"), ("f32", 16, 4, "auto"),
        ("bf16", 128, 4, "native"), ("f16", 128, 2, "fp32"), ("f32", 64, 4, "auto"),
    ]
    small = ((11, 13), (6, 7), (3, 5), (2, 2))
    # a pyramid whose large levels take few samples a row: 4*Q*K = 656 corners
    # over 3072, 768, 192 and 48 rows a head (the touch classes of the FP32
    # workspace's rows find untouched, once- and several-times-touched rows)
    sparse = ((48, 64), (24, 32), (12, 16), (6, 8))
    cases = [c + (small,) for c in cases] + [
        ("bf16", 32, 4, "fp32", sparse), ("f16", 64, 4, "fp32", sparse), ("bf16", 96, 4, "fp32", sparse),
        ("f16", 128, 4, "fp32", sparse), ("bf16", 32, 4, "native", sparse),
    ]
    for dtype, D, K, accum, shapes in cases:
        wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, D=D, K=K, B=2, Q=41, M=3, shapes=shapes)
        inp = W.make_inputs(wl)
        t = to_torch(inp, dtype, "cuda:0")
        out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                           t["attention_weights"])
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], t["grad_out"], accum=accum)
        torch.cuda.synchronize()
        what = f"{os.environ.get('MSDA_TUNE')} {dtype} D={D} K={K} {accum} S={wl.S}"
        assert_forward(dtype, f64(out), oracle.forward(inp, dtype), what)
        rgv, rgl, rga = oracle.backward(inp, dtype)
        assert_grad(dtype, f64(gv), rgv, what + " grad_value")
        assert_grad(dtype, f64(gl), rgl, what + " grad_loc")
        assert_grad(dtype, f64(ga), rga, what + " grad_attn")
    # Exact cases: integer values, weights and output gradients, and samples at
    # pixel centres of power-of-two levels (one corner of weight exactly 1), so
    # every product and every partial sum is an integer the dtype holds and the
    # results must equal the oracle's rounded once: a lost, repeated or
    # misrouted contribution (a reduction, a directly written row, a rounding)
    # shows as an exact mismatch.
    pow2 = ((32, 64), (16, 32), (8, 16), (4, 8))
    exact = [("bf16", 32, "fp32"), ("bf16", 32, "native"), ("f16", 64, "fp32"), ("f32", 48, "auto"),
             ("bf16", 96, "fp32"), ("bf16", 32, "deterministic"), ("bf16", 128, "fp32")]
    for dtype, D, accum in exact:
        wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, D=D, K=4, B=2, Q=41, M=3, shapes=pow2)
        inp = _exact_inputs(wl)
        t = to_torch(inp, dtype, "cuda:0")
        out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                           t["attention_weights"])
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], t["grad_out"], accum=accum)
        torch.cuda.synchronize()
        what = f"{os.environ.get('MSDA_TUNE')} exact {dtype} D={D} {accum}"
        rgv, rgl, rga = oracle.backward(inp, dtype)
        for got, ref, name in ((out, oracle.forward(inp, dtype), "out"), (gv, rgv, "grad_value"),
                               (gl, rgl, "grad_loc"), (ga, rga, "grad_attn")):
            want = W.to_f64(W.cast(ref, dtype), dtype)
            bad = np.flatnonzero(f64(got).ravel() != want.ravel())
            assert bad.size == 0, f"{what} {name}: {bad.size} differ, first at {bad[0]}: " \
                                  f"{f64(got).ravel()[bad[0]]} vs {want.ravel()[bad[0]]}"
    assert msda.device_errors() == 0
    print("ok", os.environ.get("MSDA_TUNE"))


def _exact_inputs(wl):
    """Inputs whose products and sums are small integers (see the exact cases)."""
    rng = np.random.Generator(np.random.PCG64(77))
    B, M, D, L, K, S, Q = wl.B, wl.M, wl.D, wl.L, wl.K, wl.S, wl.Qn
    inp = dict(W.make_inputs(wl))
    inp["value"] = W.cast(rng.integers(-4, 5, (B, S, M, D)).astype(np.float64), wl.dtype)
    loc = np.empty((B, Q, M, L, K, 2))
    for l, (h, w) in enumerate(wl.shapes):
        loc[:, :, :, l, :, 0] = (rng.integers(0, w, (B, Q, M, K)) + 0.5) / w
        loc[:, :, :, l, :, 1] = (rng.integers(0, h, (B, Q, M, K)) + 0.5) / h
    inp["sampling_locations"] = W.cast(loc, wl.dtype)
    inp["attention_weights"] = W.cast(rng.integers(1, 3, (B, Q, M, L, K)).astype(np.float64), wl.dtype)
    inp["grad_out"] = W.cast(rng.integers(-3, 4, (B, Q, M * D)).astype(np.float64), wl.dtype)
    return inp


if __name__ == "__main__":
    main()
