"""Stream-order safety of the programmatic (early) launches.

The forward and the backward's zero kernel are launched as programmatic
dependents: they may start before the kernel ahead of them finishes, and must
wait for it before touching memory it uses.  These tests make that matter:
every input is written by a kernel right before the call, and freed buffers
are handed back by the caching allocator (a freed tensor's block becomes the
next call's output while the kernel that read it may still be in flight).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from msda_testutil import assert_forward, assert_grad, f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    msda._lib.lib()
    msda.device_errors(clear=True)
    yield
    assert msda.device_errors(clear=True) == 0


@pytest.mark.parametrize("name,over", [("decoder_bf16", {}), ("tiny_fp32", {"D": 32, "B": 2, "Q": 50}),
                                       ("oddD_fp32", {"B": 2})])
def test_inputs_written_just_before_the_call(name, over):
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS[name].with_(**over) if over else W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    t = to_torch(inp, wl.dtype, DEV)
    want_out = oracle.forward(inp, wl.dtype)
    want = oracle.backward(inp, wl.dtype)
    for _ in range(4):
        # each input is the output of a kernel enqueued just before the call
        value = t["value"] * 1
        loc = t["sampling_locations"] + 0
        attn = t["attention_weights"] * 1
        g = t["grad_out"] + 0
        out = msda.forward(value, t["spatial_shapes"], t["level_start_index"], loc, attn)
        # value / loc / attn are dropped: their blocks go back to the
        # allocator and come out again as the backward's outputs
        v2, l2, a2 = value * 1, loc + 0, attn * 1
        del value, loc, attn
        gv, gl, ga = msda.backward(v2, t["spatial_shapes"], t["level_start_index"], l2, a2, g)
        torch.cuda.synchronize()
        assert_forward(wl.dtype, f64(out), want_out, "out")
        for got, ref, what in zip((gv, gl, ga), want, ("grad_value", "grad_loc", "grad_attn")):
            assert_grad(wl.dtype, f64(got), ref, what)


def test_grad_value_reuses_the_block_the_forward_reads():
    """grad_value allocated from the block of the forward's value tensor:
    the backward's zero kernel must not start writing it while the forward
    still reads it."""
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS["decoder_bf16"]
    inp = W.make_inputs(wl)
    t = to_torch(inp, wl.dtype, DEV)
    want_out = oracle.forward(inp, wl.dtype)
    keep = t["value"].clone()
    for _ in range(4):
        value = keep * 1
        ptr = value.data_ptr()
        out = msda.forward(value, t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                           t["attention_weights"])
        del value
        grad_value = torch.empty_like(keep)
        reused = grad_value.data_ptr() == ptr
        msda.backward(keep, t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                      t["attention_weights"], t["grad_out"], grad_value=grad_value)
        torch.cuda.synchronize()
        assert_forward(wl.dtype, f64(out), want_out, f"out (grad_value reused the block: {reused})")


def test_backward_inputs_from_the_kernel_ahead():
    """grad_out written by the kernel right before the backward: the
    backward's early gather phase must see it (the zero kernel waits for that
    kernel before letting the backward start)."""
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS["decoder_bf16"]
    inp = W.make_inputs(wl)
    t = to_torch(inp, wl.dtype, DEV)
    want = oracle.backward(inp, wl.dtype)
    big = torch.empty(64 << 20, dtype=torch.float32, device=DEV)
    for _ in range(4):
        g = torch.zeros_like(t["grad_out"])
        big.add_(1)                      # a long kernel ahead, so the next one is still running
        g.copy_(t["grad_out"])           # grad_out written by the kernel right before the call
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"],
                                   t["sampling_locations"], t["attention_weights"], g)
        torch.cuda.synchronize()
        for got, ref, what in zip((gv, gl, ga), want, ("grad_value", "grad_loc", "grad_attn")):
            assert_grad(wl.dtype, f64(got), ref, what)
    assert np.isfinite(f64(big[:4])).all()


def test_two_streams_run_independent_problems():
    """Two problems on two streams at once (programmatic launches on both):
    each matches the oracle, whatever the interleaving."""
    import scale_deformable_attention_gb300 as msda

    cases = []
    for seed, name in ((5, "decoder_bf16"), (6, "oddD_fp32")):
        wl = W.WORKLOADS[name].with_(B=2, seed=seed)
        inp = W.make_inputs(wl)
        cases.append((wl, inp, to_torch(inp, wl.dtype, DEV), torch.cuda.Stream()))
    torch.cuda.synchronize()
    results = []
    for _ in range(3):
        outs = []
        for wl, inp, t, s in cases:
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], validate=False)
                grads = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"],
                                      t["sampling_locations"], t["attention_weights"], t["grad_out"], validate=False)
            outs.append((out, grads))
        torch.cuda.synchronize()
        results.append(outs)
    for (wl, inp, _, _), k in zip(cases, range(2)):
        want_out = oracle.forward(inp, wl.dtype)
        want = oracle.backward(inp, wl.dtype)
        for outs in results:
            out, (gv, gl, ga) = outs[k]
            assert_forward(wl.dtype, f64(out), want_out, f"{wl.name} out")
            for got, ref, what in zip((gv, gl, ga), want, ("grad_value", "grad_loc", "grad_attn")):
                assert_grad(wl.dtype, f64(got), ref, f"{wl.name} {what}")
