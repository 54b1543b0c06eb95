"""The C-ABI calls captured into a CUDA graph (README, "Caveats": the operator
is graph capturable): capture forward + backward once, replay on new inputs
copied into the captured buffers, and compare with eager calls."""
import pytest

import workloads as W
from msda_testutil import f64, rel_l2, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(dtype, seed):
    wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, B=2, Q=120, seed=seed)
    return wl, to_torch(W.make_inputs(wl), dtype, DEV)


@pytest.mark.parametrize("dtype,accum", [("bf16", "native"), ("bf16", "fp32"), ("f32", "auto")])
def test_graph_replay_matches_eager(dtype, accum):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    wl, t = _inputs(dtype, 31)
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
        _, fresh = _inputs(dtype, seed)
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
