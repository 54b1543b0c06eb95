"""The deterministic grad_value accumulator: parity with the oracle, and
bit-identical grad_value from run to run (where the atomics of the other
accumulators commit in arbitrary order; course ch. 5, "Atomics make gradients
nondeterministic")."""
import pytest

import oracle
import workloads as W
from msda_testutil import assert_forward, assert_grad, f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    ("tiny_fp32", {}),
    ("tiny_fp32", {"dtype": "bf16", "B": 2, "Q": 33}),
    ("decoder_bf16", {}),
    ("decoder_bf16", {"dtype": "f16", "B": 2}),
    ("oddD_fp32", {"B": 2}),
    ("encoder_fp16", {"B": 1}),
]


@pytest.mark.parametrize("name,over", CASES, ids=[f"{n}-{o}" for n, o in CASES])
def test_deterministic_parity_and_repeatability(name, over):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS[name].with_(**over) if over else W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    t = to_torch(inp, wl.dtype, DEV)
    args = (t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"], t["attention_weights"],
            t["grad_out"])
    runs = [msda.backward(*args, accum="deterministic") for _ in range(3)]
    torch.cuda.synchronize()
    for gv, gl, ga in runs[1:]:
        assert torch.equal(gv, runs[0][0]), "grad_value differs between runs"
        assert torch.equal(gl, runs[0][1]) and torch.equal(ga, runs[0][2])
    rgv, rgl, rga = oracle.backward(inp, wl.dtype)
    gv, gl, ga = runs[0]
    assert_grad(wl.dtype, f64(gv), rgv, "deterministic grad_value")
    assert_grad(wl.dtype, f64(gl), rgl, "grad_loc")
    assert_grad(wl.dtype, f64(ga), rga, "grad_attn")
    # accumulating into the first result gives 2x, also bit for bit repeatable
    acc1 = msda.backward(*args, accum="deterministic", grad_value=runs[0][0].clone(), accumulate=True)[0]
    acc2 = msda.backward(*args, accum="deterministic", grad_value=runs[0][0].clone(), accumulate=True)[0]
    torch.cuda.synchronize()
    assert torch.equal(acc1, acc2)
    assert_grad(wl.dtype, f64(acc1), 2 * rgv, "deterministic accumulate")
    assert msda.device_errors() == 0


def test_deterministic_fp32_is_tight():
    """fp32 I/O: the fixed-point sum is exact to far below fp32 rounding, so the
    result matches the oracle about as well as a single fp32 rounding."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS["oddD_fp32"].with_(B=1)
    inp = W.make_inputs(wl)
    t = to_torch(inp, "f32", DEV)
    gv, _, _ = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                             t["attention_weights"], t["grad_out"], accum="deterministic")
    rgv, _, _ = oracle.backward(inp, "f32")
    err = assert_grad("f32", f64(gv), rgv, "deterministic fp32")
    assert err < 1e-6
