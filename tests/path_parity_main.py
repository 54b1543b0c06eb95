"""Compact forward + backward parity check against the oracle, run by
test_gpu_kernel_paths.py in a child process whose MSDA_TUNE forces one kernel
family (the library reads MSDA_TUNE once per process)."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

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
    assert msda.device_errors() == 0
    print("ok", os.environ.get("MSDA_TUNE"))


if __name__ == "__main__":
    main()
