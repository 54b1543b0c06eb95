"""msda_backward_static_workspace -- the backward that allocates nothing --
checked through the C ABI on the GPU against the fp64 oracle and against
msda_backward with a caller-provided workspace.

Some callers cannot allocate device memory when they call the backward: an
inference or training engine plugin that is handed only its input and output
tensors, or a loop that forbids allocation once it is running.  For them the
scratch of the FP32 accumulator lives in a fixed device array inside the
library.  This file is collected last so that a stop-at-first-failure run has
already run every other test when it gets here; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from msda_testutil import f64, rel_l2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"bf16": 2e-2, "f16": 2e-2, "f32": 1e-4}   # the parity tests' gradient tolerances
CODE = {"f32": 0, "f16": 1, "bf16": 2}
LIMIT = 64 << 20                                  # MSDA_STATIC_WORKSPACE_BYTES
ERR_WORKSPACE = 4


def _entry(lib):
    f = lib.msda_backward_static_workspace
    f.argtypes = ([ctypes.c_int, ctypes.c_uint] + [ctypes.c_int64] * 7 + [ctypes.c_void_p] * 9 +
                  [ctypes.c_void_p])
    f.restype = ctypes.c_int
    return f


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_gb300 import _lib

    return _lib.lib()


def _call(f, dtype, flags, dims, t, gv, gl, ga):
    return f(CODE[dtype], flags, *dims, t["value"].data_ptr(), t["spatial_shapes"].data_ptr(),
             t["level_start_index"].data_ptr(), t["sampling_locations"].data_ptr(),
             t["attention_weights"].data_ptr(), t["grad_out"].data_ptr(), gv.data_ptr(), gl.data_ptr(),
             ga.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _need(lib, dtype, dims):
    """Scratch the static array must hold: the FP32 accumulator's fp32 sums,
    B*S*M*D*4 bytes for fp16/bf16 I/O (the touch classes that
    msda_backward_workspace_size adds are optional), none for fp32 I/O."""
    from scale_deformable_attention_gb300 import _lib

    full = int(lib.msda_backward_workspace_size(CODE[dtype], _lib.ACCUM["fp32"], *dims))
    if full == 0:
        return 0
    B, S, M, D = dims[:4]
    assert full >= B * S * M * D * 4
    return B * S * M * D * 4


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_static_workspace_matches_oracle_and_workspace_backward(lib, dtype):
    """Two calls in a row on different inputs (nothing may carry over in the
    shared array), each against the oracle and against msda_backward with the
    FP32 accumulator and a torch-allocated workspace.  fp32 I/O takes the
    branch that needs no scratch."""
    import scale_deformable_attention_gb300 as msda

    f = _entry(lib)
    for seed in (21, 22):
        wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, B=1, Q=150, seed=seed)
        inp = W.make_inputs(wl)
        t = W.to_torch(inp, dtype, DEV)
        dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
        assert (_need(lib, dtype, dims) > 0) == (dtype != "f32")
        ref_gv, ref_gl, ref_ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"],
                                               t["sampling_locations"], t["attention_weights"], t["grad_out"],
                                               accum="fp32")
        gv = torch.full_like(t["value"], 3.0)     # stale contents the call must overwrite
        gl = torch.empty_like(t["sampling_locations"])
        ga = torch.empty_like(t["attention_weights"])
        rc = _call(f, dtype, 0, dims, t, gv, gl, ga)
        assert rc == 0, lib.msda_last_error()
        torch.cuda.synchronize()
        o_gv, o_gl, o_ga = oracle.backward(inp, dtype)
        for got, want, name in ((gv, o_gv, "grad_value"), (gl, o_gl, "grad_loc"), (ga, o_ga, "grad_attn")):
            e = rel_l2(f64(got), want)
            assert e <= TOL[dtype], f"{dtype} seed {seed} {name} vs oracle: rel-L2 {e:.3e}"
        assert rel_l2(f64(gv), f64(ref_gv)) <= TOL[dtype]
        assert torch.equal(gl, ref_gl) and torch.equal(ga, ref_ga)


def test_static_workspace_accumulates(lib):
    """MSDA_BWD_ACCUMULATE adds into the caller's grad_value (widened into the
    shared array first): twice in a row from a known non-zero start, each
    against that start plus the oracle's grad_value."""
    import scale_deformable_attention_gb300 as msda

    f = _entry(lib)
    wl = W.WORKLOADS["decoder_bf16"].with_(B=1, Q=150, seed=23)
    inp = W.make_inputs(wl)
    t = W.to_torch(inp, "bf16", DEV)
    dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
    start = torch.randn(t["value"].shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(DEV)
    o_gv, _, _ = oracle.backward(inp, "bf16")
    gv = start.clone()
    gl = torch.empty_like(t["sampling_locations"])
    ga = torch.empty_like(t["attention_weights"])
    for n in (1, 2):
        assert _call(f, "bf16", msda.BWD_ACCUMULATE, dims, t, gv, gl, ga) == 0, lib.msda_last_error()
        torch.cuda.synchronize()
        want = f64(start) + n * o_gv
        e = rel_l2(f64(gv), want)
        assert e <= TOL["bf16"], f"accumulate call {n}: rel-L2 {e:.3e}"
    ref = start.clone()
    msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                  t["attention_weights"], t["grad_out"], accum="fp32", grad_value=ref, accumulate=True)
    msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                  t["attention_weights"], t["grad_out"], accum="fp32", grad_value=ref, accumulate=True)
    torch.cuda.synchronize()
    assert rel_l2(f64(gv), f64(ref)) <= TOL["bf16"]


def test_static_workspace_size_boundary(lib):
    """A call whose scratch is exactly the array's size is accepted and
    correct; one element more is rejected with MSDA_ERR_WORKSPACE before
    anything is enqueued (the outputs keep their contents).  One channel per
    head (D = 1) takes the FP32 accumulator with an fp32 mirror of grad_value,
    B*S*M*D*4 bytes."""
    import scale_deformable_attention_gb300 as msda

    f = _entry(lib)
    # accepted at the boundary: 2^24 rows of one bf16 channel (32 MiB of value), 64 MiB of fp32 scratch
    side = 4096
    wl = W.Workload("boundary", B=1, M=1, D=1, K=2, shapes=((side, side),), Q=300, dtype="bf16", loc="uniform01",
                    logits="uniform01", seed=24)
    dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
    assert _need(lib, "bf16", dims) == LIMIT
    inp = W.make_inputs(wl)
    t = W.to_torch(inp, "bf16", DEV)
    gv = torch.full_like(t["value"], 3.0)
    gl = torch.empty_like(t["sampling_locations"])
    ga = torch.empty_like(t["attention_weights"])
    assert _call(f, "bf16", 0, dims, t, gv, gl, ga) == 0, lib.msda_last_error()
    torch.cuda.synchronize()
    o_gv, o_gl, o_ga = oracle.backward(inp, "bf16")
    for got, want, name in ((gv, o_gv, "grad_value"), (gl, o_gl, "grad_loc"), (ga, o_ga, "grad_attn")):
        e = rel_l2(f64(got), want)
        assert e <= TOL["bf16"], f"at the size limit, {name} vs oracle: rel-L2 {e:.3e}"
    ref_gv, _, _ = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                 t["attention_weights"], t["grad_out"], accum="fp32")
    torch.cuda.synchronize()
    assert rel_l2(f64(gv), f64(ref_gv)) <= TOL["bf16"]
    del t, gv, gl, ga, inp, ref_gv

    # rejected one element above
    M, D, Q = 1, 1, 1
    S = LIMIT // 4 + 1
    dims = (1, S, M, D, 1, 1, Q)
    assert _need(lib, "bf16", dims) == LIMIT + 4
    value = torch.zeros((1, S, M, D), dtype=torch.bfloat16, device=DEV)
    z = {"value": value, "spatial_shapes": torch.tensor([[1, S]], dtype=torch.int64, device=DEV),
         "level_start_index": torch.zeros(1, dtype=torch.int64, device=DEV),
         "sampling_locations": torch.full((1, Q, M, 1, 1, 2), 0.5, dtype=torch.bfloat16, device=DEV),
         "attention_weights": torch.ones((1, Q, M, 1, 1), dtype=torch.bfloat16, device=DEV),
         "grad_out": torch.ones((1, Q, M * D), dtype=torch.bfloat16, device=DEV)}
    gv = torch.full_like(value, 3.0)
    gl = torch.full_like(z["sampling_locations"], 3.0)
    ga = torch.full_like(z["attention_weights"], 3.0)
    rc = _call(f, "bf16", 0, dims, z, gv, gl, ga)
    assert rc == ERR_WORKSPACE, f"expected MSDA_ERR_WORKSPACE, got {rc}"
    assert b"static workspace" in lib.msda_last_error()
    torch.cuda.synchronize()
    assert bool((gv == 3.0).all()) and bool((gl == 3.0).all()) and bool((ga == 3.0).all()), \
        "a rejected call wrote its outputs"


def test_static_workspace_argument_errors_match_backward(lib):
    """Invalid arguments get msda_backward's own status, not the size error,
    even when the sizes are also above the limit."""
    f = _entry(lib)
    S = LIMIT // 4 + 1
    nul = ctypes.c_void_p(0)
    st = torch.cuda.current_stream().cuda_stream
    rc = f(2, 0, 1, S, 1, 1, 0, 1, 1, *([nul] * 9), st)          # L = 0
    assert rc == 1, f"expected MSDA_ERR_INVALID_ARG, got {rc}"
    rc = f(2, 0, 1, S, 1, 1, 1, 1, 1, *([nul] * 9), st)          # NULL pointers
    assert rc == 1, f"expected MSDA_ERR_INVALID_ARG, got {rc}"
    rc = f(2, 0, 1, S, 1, 0, 1, 1, 1, *([nul] * 9), st)          # D = 0 and value too large: nothing to sample
    assert rc != ERR_WORKSPACE
