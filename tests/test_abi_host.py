"""The C-ABI library on the host, without a GPU: it loads, exports every
function include/msda.h declares, and rejects invalid calls with the right
status before any CUDA call.  (No call here reaches a kernel launch: every
fake pointer below fails validation first.)"""
import ctypes
import os
import re
import subprocess
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msda.h")


@pytest.fixture(scope="module")
def lib():
    from scale_deformable_attention_gb300 import _lib, build

    build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(msda_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("msda_forward", "msda_backward", "msda_backward_workspace_size", "msda_last_error",
              "msda_resolve_accum", "msda_device_errors", "msda_trace_enable", "msda_trace_read",
              "msda_forward_fused", "msda_backward_fused", "msda_backward_static_workspace"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    from scale_deformable_attention_gb300 import _lib

    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\b[TW] (msda_\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def declared_arity():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(msda_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argtypes_match_the_header(lib):
    arity = declared_arity()
    assert "msda_backward_fused" in arity
    for name, n in arity.items():
        fn = getattr(lib, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, f"{name}: header has {n} parameters, binding declares {len(fn.argtypes)}"


F32, F16, BF16 = 0, 1, 2
GOOD = dict(B=2, S=60, M=2, D=8, L=2, K=2, Q=10)
FAKE = 0x10000  # aligned, never dereferenced: every call using it fails validation


def fwd(lib, dt=F32, ptrs=None, **kw):
    d = dict(GOOD)
    d.update(kw)
    p = [FAKE] * 6 if ptrs is None else ptrs
    return lib.msda_forward(dt, d["B"], d["S"], d["M"], d["D"], d["L"], d["K"], d["Q"], *p, None)


def bwd(lib, dt=F32, mode=0, flags=0, ptrs=None, ws=None, ws_bytes=0, **kw):
    d = dict(GOOD)
    d.update(kw)
    p = [FAKE] * 9 if ptrs is None else ptrs
    return lib.msda_backward(dt, mode, flags, d["B"], d["S"], d["M"], d["D"], d["L"], d["K"], d["Q"], *p, ws,
                             ws_bytes, None)


def msg(lib):
    return lib.msda_last_error().decode()


@pytest.mark.parametrize("kw,status,text", [
    (dict(B=-1), 1, "negative"),
    (dict(L=0), 1, "L and K"),
    (dict(K=0), 1, "L and K"),
    (dict(L=17), 2, "L=17"),
    (dict(K=65), 2, "K=65"),
    (dict(L=16, K=17), 2, "L*K"),
    (dict(D=1025), 2, "D=1025"),
    (dict(B=1 << 40, Q=1 << 40), 1, "overflow"),
])
def test_forward_rejects_sizes(lib, kw, status, text):
    assert fwd(lib, **kw) == status
    assert text in msg(lib)


def test_forward_rejects_bad_dtype(lib):
    assert fwd(lib, dt=7) == 1
    assert "dtype" in msg(lib)


@pytest.mark.parametrize("idx,name", [(0, "value"), (1, "spatial_shapes"), (2, "level_start_index"),
                                      (3, "sampling_locations"), (4, "attention_weights"), (5, "out")])
def test_forward_rejects_null(lib, idx, name):
    p = [FAKE] * 6
    p[idx] = None
    assert fwd(lib, ptrs=p) == 1
    assert name in msg(lib) and "NULL" in msg(lib)


@pytest.mark.parametrize("dt,idx,off", [(F32, 0, 2), (F16, 3, 1), (BF16, 5, 1), (F32, 1, 4)])
def test_forward_rejects_misaligned(lib, dt, idx, off):
    p = [FAKE] * 6
    p[idx] = FAKE + off
    assert fwd(lib, dt=dt, ptrs=p) == 3
    assert "aligned" in msg(lib)


@pytest.mark.parametrize("kw", [dict(B=0), dict(Q=0), dict(M=0), dict(D=0)])
def test_forward_empty_is_ok_without_launch(lib, kw):
    # empty output: validated, nothing enqueued, no CUDA call (works without a GPU)
    assert fwd(lib, ptrs=[None] * 6, **kw) == 0


def test_backward_rejects_mode_and_flags(lib):
    assert bwd(lib, mode=5) == 1 and "accumulator" in msg(lib)
    assert bwd(lib, flags=4) == 1 and "flags" in msg(lib)
    assert bwd(lib, flags=8) == 1 and "flags" in msg(lib)


def test_backward_deterministic_needs_workspace(lib):
    assert bwd(lib, dt=F32, mode=3) == 4 and "deterministic" in msg(lib)
    n = GOOD["B"] * GOOD["S"] * GOOD["M"] * GOOD["D"]
    assert bwd(lib, dt=BF16, mode=3, ws=FAKE, ws_bytes=256 + 8 * n - 1) == 4


def test_backward_null_grad_value(lib):
    p = [FAKE] * 9
    p[6] = None
    assert bwd(lib, ptrs=p) == 1 and "grad_value" in msg(lib)


def test_backward_workspace_required(lib):
    # bf16 with the FP32 accumulator and no / short / misaligned workspace
    assert bwd(lib, dt=BF16, mode=2) == 4 and "workspace" in msg(lib)
    need = GOOD["B"] * GOOD["S"] * GOOD["M"] * GOOD["D"] * 4
    assert bwd(lib, dt=BF16, mode=2, ws=FAKE, ws_bytes=need - 1) == 4
    assert bwd(lib, dt=BF16, mode=2, ws=FAKE + 8, ws_bytes=need) == 4 and "16-byte" in msg(lib)


def test_backward_empty_value_and_queries_ok(lib):
    assert bwd(lib, ptrs=[None] * 9, B=0) == 0


def test_workspace_size_and_resolution(lib):
    dims = (GOOD["B"], GOOD["S"], GOOD["M"], GOOD["D"], GOOD["L"], GOOD["K"], GOOD["Q"])
    n = GOOD["B"] * GOOD["S"] * GOOD["M"] * GOOD["D"]
    assert lib.msda_backward_workspace_size(F32, 2, *dims) == 0
    assert lib.msda_backward_workspace_size(BF16, 1, *dims) == 0
    # fp32 sums, then 2 bits per (b, pixel, head) row of touch classes (16-byte aligned)
    rows = GOOD["B"] * GOOD["S"] * GOOD["M"]
    fp32 = (4 * n + 15) // 16 * 16 + (rows + 63) // 64 * 16
    assert lib.msda_backward_workspace_size(BF16, 2, *dims) == fp32
    assert lib.msda_backward_workspace_size(F16, 2, *dims) == fp32
    assert lib.msda_resolve_accum(F32, 2, *dims) == 1
    assert lib.msda_resolve_accum(BF16, 1, *dims) == 1
    assert lib.msda_resolve_accum(BF16, 2, *dims) == 2
    assert lib.msda_resolve_accum(F16, 0, *dims) in (1, 2)
    # deterministic accumulator: any dtype, 256-byte header + int64 sums
    for dt in (F32, F16, BF16):
        assert lib.msda_backward_workspace_size(dt, 3, *dims) == 256 + 8 * n
        assert lib.msda_resolve_accum(dt, 3, *dims) == 3
    # many samples per pixel: bf16 AUTO goes to the fp32 accumulator
    dense = (2, 22223, 8, 32, 4, 4, 22223)
    assert lib.msda_resolve_accum(BF16, 0, *dense) == 2


def fused_fwd(lib, dt=F32, ptrs=None, **kw):
    d = dict(GOOD)
    d.update(kw)
    p = [FAKE] * 7 if ptrs is None else ptrs
    return lib.msda_forward_fused(dt, d["B"], d["S"], d["M"], d["D"], d["L"], d["K"], d["Q"], *p, None)


def fused_bwd(lib, dt=F32, mode=0, flags=0, ptrs=None, **kw):
    d = dict(GOOD)
    d.update(kw)
    p = [FAKE] * 11 if ptrs is None else ptrs
    return lib.msda_backward_fused(dt, mode, flags, d["B"], d["S"], d["M"], d["D"], d["L"], d["K"], d["Q"], *p,
                                   None, 0, None)


@pytest.mark.parametrize("idx,name", [(0, "value"), (3, "reference_points"), (4, "sampling_offsets"),
                                      (5, "attention_logits"), (6, "out")])
def test_fused_forward_rejects_null(lib, idx, name):
    p = [FAKE] * 7
    p[idx] = None
    assert fused_fwd(lib, ptrs=p) == 1
    assert name in msg(lib) and "NULL" in msg(lib)


@pytest.mark.parametrize("idx,name", [(3, "reference_points"), (4, "sampling_offsets"), (5, "attention_logits"),
                                      (6, "grad_out"), (7, "grad_value"), (8, "grad_reference_points"),
                                      (9, "grad_sampling_offsets"), (10, "grad_attention_logits")])
def test_fused_backward_rejects_null(lib, idx, name):
    p = [FAKE] * 11
    p[idx] = None
    assert fused_bwd(lib, ptrs=p) == 1
    assert name in msg(lib) and "NULL" in msg(lib)


def test_fused_rejects_sizes_and_modes(lib):
    assert fused_fwd(lib, K=65) == 2 and "K=65" in msg(lib)
    assert fused_bwd(lib, mode=9) == 1 and "accumulator" in msg(lib)
    assert fused_bwd(lib, dt=BF16, mode=3) == 4 and "deterministic" in msg(lib)


@pytest.mark.parametrize("kw", [dict(B=0), dict(Q=0)])
def test_fused_empty_is_ok_without_launch(lib, kw):
    assert fused_fwd(lib, ptrs=[None] * 7, **kw) == 0
    if "B" in kw:  # nothing to zero either
        assert fused_bwd(lib, ptrs=[None] * 11, **kw) == 0


def test_status_strings_version_kernel_names(lib):
    assert lib.msda_status_string(0) == b"MSDA_OK"
    assert lib.msda_status_string(4) == b"MSDA_ERR_WORKSPACE"
    assert lib.msda_version() >= 100
    assert [lib.msda_kernel_name(i) for i in range(4)] == [b"forward", b"backward", b"zero", b"convert"]


def test_last_error_is_per_thread(lib):
    assert fwd(lib, B=-1) == 1
    seen = []
    t = threading.Thread(target=lambda: seen.append(lib.msda_last_error()))
    t.start()
    t.join()
    assert seen == [b""]
    assert b"negative" in lib.msda_last_error()


def test_binding_refuses_cpu_tensors():
    import torch

    import scale_deformable_attention_gb300 as msda

    v = torch.zeros(1, 60, 2, 8)
    loc = torch.zeros(1, 10, 2, 2, 2, 2)
    attn = torch.zeros(1, 10, 2, 2, 2)
    ss = torch.tensor([[6, 8], [3, 4]])
    with pytest.raises(ValueError, match="CUDA"):
        msda.forward(v, ss, None, loc, attn)


def test_reduction_ceiling_rejects_bad_arguments(lib):
    out = ctypes.c_double(0.0)
    mib = 1 << 20
    assert lib.msda_reduction_ceiling(0, 64, 8, 5, None, 64 * mib, ctypes.byref(out), None) == 1
    assert "scratch" in msg(lib)
    assert lib.msda_reduction_ceiling(0, 64, 8, 5, FAKE, mib - 1, ctypes.byref(out), None) == 1
    assert lib.msda_reduction_ceiling(0, 64, 8, 5, FAKE + 8, 64 * mib, ctypes.byref(out), None) == 1
    assert lib.msda_reduction_ceiling(3, 64, 8, 5, FAKE, 64 * mib, ctypes.byref(out), None) == 1 and "kind" in msg(lib)
    assert lib.msda_reduction_ceiling(0, 48, 8, 5, FAKE, 64 * mib, ctypes.byref(out), None) == 1 and "row_bytes" in msg(lib)
    assert lib.msda_reduction_ceiling(0, 1024, 8, 5, FAKE, 64 * mib, ctypes.byref(out), None) == 1
    assert lib.msda_reduction_ceiling(0, 64, 0, 5, FAKE, 64 * mib, ctypes.byref(out), None) == 1
    assert lib.msda_reduction_ceiling(0, 64, 8, 101, FAKE, 64 * mib, ctypes.byref(out), None) == 1
    assert lib.msda_reduction_ceiling(0, 64, 8, 5, FAKE, 64 * mib, None, None) == 1

def test_static_workspace_rejects_zeroed_flag(lib):
    """The allocation-free backward clears its own array on every call; the
    flag by which a caller vouches for a zeroed workspace does not apply."""
    f = lib.msda_backward_static_workspace
    f.argtypes = ([ctypes.c_int, ctypes.c_uint] + [ctypes.c_int64] * 7 + [ctypes.c_void_p] * 9 + [ctypes.c_void_p])
    f.restype = ctypes.c_int
    p = [FAKE] * 9
    assert f(2, 2, 1, 4, 1, 32, 1, 1, 1, *p, None) == 1 and "ZEROED" in msg(lib)
