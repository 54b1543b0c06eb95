"""The C-ABI calls captured into a CUDA graph (README, "Caveats": the operator
is graph capturable): capture forward + backward once, replay on new inputs
copied into the captured buffers, and compare with eager calls."""
import pytest

import workloads as W
from msda_testutil import f64, rel_l2, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


# large enough for one backward pass per level, with a sparse level 0: the FP32
# accumulator then counts touch classes and rounds on a second stream, which
# the capture forks and joins
_BIG = dict(Q=15000, shapes=((256, 256), (128, 128), (64, 64), (32, 32)))


def _inputs(dtype, seed, big=False):
    kw = dict(dtype=dtype, B=2, Q=120, seed=seed)
    kw.update(_BIG if big else {})
    wl = W.WORKLOADS["decoder_bf16"].with_(**kw)
    return wl, to_torch(W.make_inputs(wl), dtype, DEV)


@pytest.mark.parametrize("dtype,accum,big", [("bf16", "native", False), ("bf16", "fp32", False), ("f32", "auto", False),
                                             ("bf16", "fp32", True)])
def test_graph_replay_matches_eager(dtype, accum, big):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl, t = _inputs(dtype, 31, big)
    bufs = {k: v.clone() for k, v in t.items()}

    def step():
        out = msda.forward(bufs["value"], bufs["spatial_shapes"], bufs["level_start_index"],
                           bufs["sampling_locations"], bufs["attention_weights"], validate=False)
        gv, gl, ga = msda.backward(bufs["value"], bufs["spatial_shapes"], bufs["level_start_index"],
                                   bufs["sampling_locations"], bufs["attention_weights"], bufs["grad_out"],
                                   accum=accum, validate=False)
        return out, gv, gl, ga

    # the first calls on a device look up device state: make them before capturing
    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = step()

    for seed in (32, 33):
        _, fresh = _inputs(dtype, seed, big)
        for k in bufs:
            bufs[k].copy_(fresh[k])
        g.replay()
        torch.cuda.synchronize()
        eager = step()
        torch.cuda.synchronize()
        tol = 1e-6 if dtype == "f32" else 1e-2
        assert torch.equal(captured[0], eager[0]), "forward differs between graph replay and eager"
        assert torch.equal(captured[2], eager[2]) and torch.equal(captured[3], eager[3])
        assert rel_l2(f64(captured[1]), f64(eager[1])) <= tol
    assert msda.device_errors() == 0


@pytest.mark.parametrize("shapes_on", ["cuda", "cpu"])
def test_autograd_op_needs_no_host_sync(shapes_on):
    """The differentiable operator (README, "Quickstart") checks spatial_shapes
    on the host the first time it sees the tensor only: later forward +
    backward calls make no synchronising call (torch's sync debug mode turns
    one into an error)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl, t = _inputs("bf16", 34)
    ss = t["spatial_shapes"].to(shapes_on)
    leaves = [t[k].clone().requires_grad_(True) for k in ("value", "sampling_locations", "attention_weights")]

    def run():
        out = msda.multi_scale_deformable_attention(leaves[0], ss, None, leaves[1], leaves[2])
        out.backward(t["grad_out"])
        return out

    run()                               # first sight of ss: checked (and copied) once
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        for _ in range(3):
            run()
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()
    bad = torch.tensor([[3, 3]] + [[1, 1]] * (wl.L - 1), dtype=torch.int64)
    with pytest.raises(ValueError):
        msda.multi_scale_deformable_attention(leaves[0], bad.to(shapes_on), None, leaves[1], leaves[2])


def test_autograd_op_graph_capture():
    """Forward + backward through the autograd operator captured as one CUDA
    graph (README, "Caveats": graph capturable) and replayed on new inputs
    copied into the captured leaves; compared with eager autograd calls."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl, t = _inputs("bf16", 35)
    ss, lsi = t["spatial_shapes"], t["level_start_index"]
    names = ("value", "sampling_locations", "attention_weights")
    leaves = {k: t[k].clone().requires_grad_(True) for k in names}
    gout = t["grad_out"].clone()

    def run():
        out = msda.multi_scale_deformable_attention(leaves["value"], ss, lsi, leaves["sampling_locations"],
                                                    leaves["attention_weights"])
        out.backward(gout)
        return out

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            for v in leaves.values():
                v.grad = None
            run()
    torch.cuda.current_stream().wait_stream(s)
    for v in leaves.values():
        v.grad = None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = run()

    for seed in (36, 37):
        _, fresh = _inputs("bf16", seed)
        with torch.no_grad():
            for k in names:
                leaves[k].copy_(fresh[k])
        gout.copy_(fresh["grad_out"])
        g.replay()
        torch.cuda.synchronize()
        got = [captured.clone()] + [leaves[k].grad.clone() for k in names]
        eager_leaves = {k: fresh[k].clone().requires_grad_(True) for k in names}
        out = msda.multi_scale_deformable_attention(eager_leaves["value"], ss, lsi,
                                                    eager_leaves["sampling_locations"],
                                                    eager_leaves["attention_weights"])
        out.backward(fresh["grad_out"])
        torch.cuda.synchronize()
        assert torch.equal(got[0], out.detach()), "forward differs between graph replay and eager"
        assert torch.equal(got[2], eager_leaves["sampling_locations"].grad)
        assert torch.equal(got[3], eager_leaves["attention_weights"].grad)
        assert rel_l2(f64(got[1]), f64(eager_leaves["value"].grad)) <= 1e-2
    assert msda.device_errors() == 0
