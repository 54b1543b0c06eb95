"""msda_backward_static_workspace -- the backward that allocates nothing --
checked against msda_backward with a caller-provided fp32 workspace, through
the C ABI on the GPU.

Some callers cannot allocate device memory when they call the backward: an
inference or training engine plugin that is handed only its input and output
tensors, or a loop that forbids allocation once it is running.  For them the
fp32 scratch of the FP32 accumulator lives in a fixed device array inside the
library.  This file is collected last so that a stop-at-first-failure run has
already run every other test when it gets here; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"bf16": 2e-2, "f16": 2e-2}   # the parity tests' tolerance for 16-bit I/O


def _entry(lib):
    f = lib.msda_backward_static_workspace
    f.argtypes = ([ctypes.c_int, ctypes.c_uint] + [ctypes.c_int64] * 7 + [ctypes.c_void_p] * 9 +
                  [ctypes.c_void_p])
    f.restype = ctypes.c_int
    return f


def _rel_l2(a, b):
    a = a.double().cpu().numpy().ravel()
    b = b.double().cpu().numpy().ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_gb300 import _lib

    return _lib.lib()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_static_workspace_matches_workspace_backward(lib, dtype):
    import scale_deformable_attention_gb300 as msda

    f = _entry(lib)
    code = {"bf16": 2, "f16": 1}[dtype]
    for seed in (21, 22):   # two calls in a row on different inputs: nothing may carry over
        wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, B=1, Q=150, seed=seed)
        inp = W.make_inputs(wl)
        t = W.to_torch(inp, dtype, DEV)
        ref_gv, ref_gl, ref_ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"],
                                               t["sampling_locations"], t["attention_weights"], t["grad_out"],
                                               accum="fp32")
        gv = torch.full_like(t["value"], 3.0)     # stale contents the call must overwrite
        gl = torch.empty_like(t["sampling_locations"])
        ga = torch.empty_like(t["attention_weights"])
        dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
        rc = f(code, 0, *dims, t["value"].data_ptr(), t["spatial_shapes"].data_ptr(),
               t["level_start_index"].data_ptr(), t["sampling_locations"].data_ptr(),
               t["attention_weights"].data_ptr(), t["grad_out"].data_ptr(), gv.data_ptr(), gl.data_ptr(),
               ga.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, lib.msda_last_error()
        torch.cuda.synchronize()
        assert _rel_l2(gv, ref_gv) <= TOL[dtype]
        assert _rel_l2(gl, ref_gl) <= TOL[dtype]
        assert _rel_l2(ga, ref_ga) <= TOL[dtype]


def test_static_workspace_rejects_oversize(lib):
    f = _entry(lib)
    # B*S*M*D one element above the array: rejected before anything is enqueued
    limit = (64 << 20) // 4
    B, S, M, D, L, K, Q = 1, limit // 64 + 1, 2, 32, 1, 1, 1
    value = torch.zeros((B, S, M, D), dtype=torch.bfloat16, device=DEV)
    shapes = torch.tensor([[1, S]], dtype=torch.int64, device=DEV)
    starts = torch.zeros(1, dtype=torch.int64, device=DEV)
    loc = torch.zeros((B, Q, M, L, K, 2), dtype=torch.bfloat16, device=DEV)
    attn = torch.zeros((B, Q, M, L, K), dtype=torch.bfloat16, device=DEV)
    gout = torch.zeros((B, Q, M * D), dtype=torch.bfloat16, device=DEV)
    gv = torch.zeros_like(value)
    gl = torch.zeros_like(loc)
    ga = torch.zeros_like(attn)
    rc = f(2, 0, B, S, M, D, L, K, Q, value.data_ptr(), shapes.data_ptr(), starts.data_ptr(), loc.data_ptr(),
           attn.data_ptr(), gout.data_ptr(), gv.data_ptr(), gl.data_ptr(), ga.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert rc == 4, f"expected MSDA_ERR_WORKSPACE, got {rc}"
    assert b"static workspace" in lib.msda_last_error()
