"""fp64 CPU oracle for the multi-scale deformable attention sampling core.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path (the
CUDA library and its binding) never does, and shares no code with it.

Three independent formulations live here:

* ``forward`` / ``backward`` (+ the ``*_units`` / ``grad_value_rows`` samplers
  for full-size checks): the C oracle in ``msda_oracle.c``, fp64, OpenMP over
  (b, m) pairs.  It follows the definition of the operator in the msda-triton
  README ("The operator", "Kernel design" on the sampling convention), the
  course's ch. 4 ("Bilinear sampling", "The corner gathers", "Accumulate and
  store") and ch. 5 ("What the backward pass must produce", "Scatter needs
  atomics").
* ``naive_forward`` / ``naive_backward``: a pure-Python loop per sample and
  corner, for tiny inputs (the README's "msda_naive" role, written here from
  the definition).
* ``gridsample_forward``: the same operator restated with
  ``torch.nn.functional.grid_sample(mode="bilinear", padding_mode="zeros",
  align_corners=False)`` in fp64 on the CPU, the identity the README states
  for its sampling convention; its autograd gives reference gradients.

``coord_mode``: 1 (default) takes the integer cell decision on the fp32 pixel
coordinate ``fma(x, W, -0.5)`` rounded to binary32, as the kernel does; 0 uses
the exact fp64 coordinate (used by the mathematical pins).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msda_oracle.c")
_LIB = os.path.join(_HERE, "libmsda_oracle.so")
_DT = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3}
_lock = threading.Lock()
_lib_handle = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: no -march, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-fopenmp", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load(path: str):
    lib = ctypes.CDLL(path)
    i64, vp, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
    prob = [ip, ip] + [i64] * 7 + [vp, vp, vp, vp, vp]
    lib.msda_oracle_forward.argtypes = prob + [dp, ip]
    lib.msda_oracle_forward_units.argtypes = prob + [vp, i64, dp, ip]
    lib.msda_oracle_backward.argtypes = prob + [vp, dp, dp, dp, ip]
    lib.msda_oracle_backward_units.argtypes = prob + [vp, vp, i64, dp, dp, ip]
    lib.msda_oracle_grad_value_rows.argtypes = prob + [vp, vp, i64, dp, ip]
    for f in ("msda_oracle_forward", "msda_oracle_forward_units", "msda_oracle_backward",
              "msda_oracle_backward_units", "msda_oracle_grad_value_rows"):
        getattr(lib, f).restype = ip
    lib.msda_oracle_num_threads.restype = ip
    lib.msda_oracle_fused_locations.argtypes = [ip] + [i64] * 5 + [vp, vp, vp, vp]
    lib.msda_oracle_fused_locations.restype = ip
    return lib


class using_library:
    """Context manager: route the wrappers below to another build of the C
    oracle (the mutation test uses it to run the pins against planted mistakes)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib_handle
        _lib()
        self._saved = _lib_handle
        _lib_handle = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib_handle
        _lib_handle = self._saved
        return False


def _lib():
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            _lib_handle = _load(build())
    return _lib_handle


def num_threads() -> int:
    return int(_lib().msda_oracle_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _prob(inp: Dict[str, np.ndarray], dtype: str, coord_mode: int, param_dtype: str = ""):
    value = np.ascontiguousarray(inp["value"])
    shapes = np.ascontiguousarray(inp["spatial_shapes"], dtype=np.int64)
    starts = np.ascontiguousarray(inp["level_start_index"], dtype=np.int64)
    loc = np.ascontiguousarray(inp["sampling_locations"])
    attn = np.ascontiguousarray(inp["attention_weights"])
    B, S, M, D = value.shape
    L = shapes.shape[0]
    Q, K = loc.shape[1], loc.shape[4]
    dims = (B, S, M, D, L, K, Q)
    keep = (value, shapes, starts, loc, attn)
    code = _DT[dtype] | ((_DT[param_dtype] + 1) << 8 if param_dtype else 0)
    args = [code, int(coord_mode), *dims, _ptr(value), _ptr(shapes), _ptr(starts), _ptr(loc), _ptr(attn)]
    return dims, args, keep


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid problem (code {rc})")


def forward(inp, dtype: str, coord_mode: int = 1, nthreads: int = 0, param_dtype: str = "") -> np.ndarray:
    """out [B, Q, M*D] in fp64 (param_dtype: storage of loc / attn when it differs from value's)."""
    (B, S, M, D, L, K, Q), args, keep = _prob(inp, dtype, coord_mode, param_dtype)
    out = np.zeros((B, Q, M * D), dtype=np.float64)
    _check(_lib().msda_oracle_forward(*args, _ptr(out), nthreads), "forward")
    return out


def forward_units(inp, dtype: str, units: np.ndarray, coord_mode: int = 1, nthreads: int = 0) -> np.ndarray:
    """out rows [n, D] of the flat units u = (b*Q + q)*M + m."""
    (B, S, M, D, L, K, Q), args, keep = _prob(inp, dtype, coord_mode)
    units = np.ascontiguousarray(units, dtype=np.int64)
    out = np.zeros((units.size, D), dtype=np.float64)
    _check(_lib().msda_oracle_forward_units(*args, _ptr(units), units.size, _ptr(out), nthreads), "forward_units")
    return out


def backward(inp, dtype: str, coord_mode: int = 1, nthreads: int = 0, param_dtype: str = ""
             ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(grad_value [B,S,M,D], grad_loc [B,Q,M,L,K,2], grad_attn [B,Q,M,L,K]) in fp64."""
    (B, S, M, D, L, K, Q), args, keep = _prob(inp, dtype, coord_mode, param_dtype)
    gout = np.ascontiguousarray(inp["grad_out"])
    gv = np.zeros((B, S, M, D), dtype=np.float64)
    gl = np.zeros((B, Q, M, L, K, 2), dtype=np.float64)
    ga = np.zeros((B, Q, M, L, K), dtype=np.float64)
    _check(_lib().msda_oracle_backward(*args, _ptr(gout), _ptr(gv), _ptr(gl), _ptr(ga), nthreads), "backward")
    return gv, gl, ga


def backward_units(inp, dtype: str, units: np.ndarray, coord_mode: int = 1, nthreads: int = 0):
    """(grad_loc [n, L*K*2], grad_attn [n, L*K]) of the flat units."""
    (B, S, M, D, L, K, Q), args, keep = _prob(inp, dtype, coord_mode)
    gout = np.ascontiguousarray(inp["grad_out"])
    units = np.ascontiguousarray(units, dtype=np.int64)
    gl = np.zeros((units.size, L * K * 2), dtype=np.float64)
    ga = np.zeros((units.size, L * K), dtype=np.float64)
    _check(_lib().msda_oracle_backward_units(*args, _ptr(gout), _ptr(units), units.size, _ptr(gl), _ptr(ga),
                                             nthreads), "backward_units")
    return gl, ga


def grad_value_rows(inp, dtype: str, rows: np.ndarray, coord_mode: int = 1, nthreads: int = 0) -> np.ndarray:
    """grad_value rows [n, D] of the flat rows r = (b*S + pixel)*M + m."""
    (B, S, M, D, L, K, Q), args, keep = _prob(inp, dtype, coord_mode)
    gout = np.ascontiguousarray(inp["grad_out"])
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, D), dtype=np.float64)
    _check(_lib().msda_oracle_grad_value_rows(*args, _ptr(gout), _ptr(rows), rows.size, _ptr(out), nthreads),
           "grad_value_rows")
    return out


# ---------------------------------------------------------------------------
# fused operator: softmax of the attention logits and the sampling locations
# from reference points and pixel offsets, around the same core
#
# msda-triton README, "The operator": A is softmax-normalised over the L*K
# (level, point) pairs of a query and head; the location is the reference
# point mapped to level l plus the learned offset.  Reading taken: offsets are
# in pixels of level l, so loc = ref + offset / (W_l, H_l) (x by W, y by H).

def fused_locations(ref: np.ndarray, off: np.ndarray, shapes: np.ndarray, coord_mode: int = 1) -> np.ndarray:
    """Sampling locations [B,Q,M,L,K,2] of the fused operator from fp64 reference
    points [B,Q,L,2] and pixel offsets [B,Q,M,L,K,2] (C oracle):
    loc = ref + off / (W_l, H_l), in binary32 with one rounding per operation
    (coord_mode 1, as the kernels) or in fp64 (coord_mode 0)."""
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    off = np.ascontiguousarray(off, dtype=np.float64)
    shapes = np.ascontiguousarray(shapes, dtype=np.int64)
    B, Q, M, L, K, _ = off.shape
    if ref.shape != (B, Q, L, 2) or shapes.shape != (L, 2):
        raise ValueError("fused_locations: reference points must be [B,Q,L,2] and shapes [L,2]")
    loc = np.zeros(off.shape, dtype=np.float64)
    _check(_lib().msda_oracle_fused_locations(int(coord_mode), B, Q, M, L, K, _ptr(shapes), _ptr(ref), _ptr(off),
                                              _ptr(loc)), "fused_locations")
    return loc


def fused_core_inputs(inp, dtype: str, coord_mode: int = 1):
    """(core inputs with fp64 loc / attn, A [B,Q,M,L,K], normaliser [L,2]) of a
    fused problem.  The locations come from ``fused_locations`` (binary32 in
    coord_mode 1, fp64 in coord_mode 0); A is the fp64 softmax."""
    from workloads import to_f64

    ref = to_f64(inp["reference_points"], dtype)        # [B,Q,L,2]
    off = to_f64(inp["sampling_offsets"], dtype)        # [B,Q,M,L,K,2]
    logits = to_f64(inp["attention_logits"], dtype)     # [B,Q,M,L*K]
    shapes = np.asarray(inp["spatial_shapes"], dtype=np.int64)
    B, Q, M, L, K, _ = off.shape
    norm = np.stack([shapes[:, 1], shapes[:, 0]], axis=-1).astype(np.float64)   # [L,2] = (W, H)
    loc = fused_locations(ref, off, shapes, coord_mode)
    z = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(z)
    A = (e / e.sum(axis=-1, keepdims=True)).reshape(B, Q, M, L, K)
    core = {"value": inp["value"], "spatial_shapes": shapes, "level_start_index": inp["level_start_index"],
            "sampling_locations": np.ascontiguousarray(loc), "attention_weights": np.ascontiguousarray(A)}
    if "grad_out" in inp:
        core["grad_out"] = inp["grad_out"]
    return core, A, norm


def fused_forward(inp, dtype: str, coord_mode: int = 1, nthreads: int = 0) -> np.ndarray:
    core, _, _ = fused_core_inputs(inp, dtype, coord_mode)
    return forward(core, dtype, coord_mode, nthreads, param_dtype="f64")


def fused_backward(inp, dtype: str, coord_mode: int = 1, nthreads: int = 0):
    """(grad_value, grad_reference_points [B,Q,L,2], grad_sampling_offsets [B,Q,M,L,K,2],
    grad_attention_logits [B,Q,M,L*K]) by the chain rule through the core:
    d loc / d offset = 1 / (W_l, H_l), d loc / d ref = 1 (summed over heads and
    points), and the softmax backward A * (gA - <A, gA>)."""
    core, A, norm = fused_core_inputs(inp, dtype, coord_mode)
    gv, gl, ga = backward(core, dtype, coord_mode, nthreads, param_dtype="f64")
    B, Q, M, L, K, _ = gl.shape
    g_off = gl / norm[None, None, None, :, None, :]
    g_ref = gl.sum(axis=(2, 4))
    A2 = A.reshape(B, Q, M, L * K)
    ga2 = ga.reshape(B, Q, M, L * K)
    g_logit = A2 * (ga2 - (A2 * ga2).sum(axis=-1, keepdims=True))
    return gv, g_ref, g_off, g_logit


# ---------------------------------------------------------------------------
# pure-Python brute force (tiny inputs only)
# ---------------------------------------------------------------------------

def _f64_inputs(inp, dtype):
    from workloads import to_f64  # storage decoding only
    return (to_f64(inp["value"], dtype), np.asarray(inp["spatial_shapes"]), np.asarray(inp["level_start_index"]),
            to_f64(inp["sampling_locations"], dtype), to_f64(inp["attention_weights"], dtype))


def _pixel_coord(u: float, n: int, coord_mode: int) -> float:
    """Pixel coordinate u*n - 0.5; coord_mode 1 rounds it once to binary32.

    For a binary32 ``u`` and an integer ``n <= 8192`` the fp64 value of
    ``u*n - 0.5`` is exact whenever it is >= -0.25 (at most 38 significant
    bits), so one rounding to binary32 equals the fused multiply-add rounding;
    below -0.25 both roundings floor to -1.
    """
    x = u * n - 0.5
    if coord_mode == 1:
        if n > 8192:
            raise ValueError("brute-force fp32 coordinate mode supports levels up to 8192 pixels wide")
        return float(np.float32(x))
    return x


def naive_forward(inp, dtype: str, coord_mode: int = 0) -> np.ndarray:
    value, shapes, starts, loc, attn = _f64_inputs(inp, dtype)
    B, S, M, D = value.shape
    Q, L, K = loc.shape[1], loc.shape[3], loc.shape[4]
    out = np.zeros((B, Q, M, D))
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                for l in range(L):
                    h, w = int(shapes[l, 0]), int(shapes[l, 1])
                    for k in range(K):
                        x = _pixel_coord(loc[b, q, m, l, k, 0], w, coord_mode)
                        y = _pixel_coord(loc[b, q, m, l, k, 1], h, coord_mode)
                        a = attn[b, q, m, l, k]
                        xf, yf = np.floor(x), np.floor(y)
                        fx, fy = x - xf, y - yf
                        for yy, wy in ((yf, 1 - fy), (yf + 1, fy)):
                            for xx, wx in ((xf, 1 - fx), (xf + 1, fx)):
                                if 0 <= xx < w and 0 <= yy < h:
                                    pix = int(starts[l]) + int(yy) * w + int(xx)
                                    out[b, q, m] += a * wy * wx * value[b, pix, m]
    return out.reshape(B, Q, M * D)


def naive_backward(inp, dtype: str, coord_mode: int = 0):
    value, shapes, starts, loc, attn = _f64_inputs(inp, dtype)
    from workloads import to_f64
    g_all = to_f64(inp["grad_out"], dtype)
    B, S, M, D = value.shape
    Q, L, K = loc.shape[1], loc.shape[3], loc.shape[4]
    g_all = g_all.reshape(B, Q, M, D)
    gv = np.zeros_like(value)
    gl = np.zeros(loc.shape)
    ga = np.zeros(attn.shape)
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                g = g_all[b, q, m]
                for l in range(L):
                    h, w = int(shapes[l, 0]), int(shapes[l, 1])
                    for k in range(K):
                        x = _pixel_coord(loc[b, q, m, l, k, 0], w, coord_mode)
                        y = _pixel_coord(loc[b, q, m, l, k, 1], h, coord_mode)
                        a = attn[b, q, m, l, k]
                        xf, yf = np.floor(x), np.floor(y)
                        fx, fy = x - xf, y - yf
                        sampled = np.zeros(D)
                        dsdx = np.zeros(D)
                        dsdy = np.zeros(D)
                        # (y offset, x offset): weight and its partial derivatives
                        for di, wy, dwy in ((0, 1 - fy, -1.0), (1, fy, 1.0)):
                            for dj, wx, dwx in ((0, 1 - fx, -1.0), (1, fx, 1.0)):
                                yy, xx = yf + di, xf + dj
                                if not (0 <= xx < w and 0 <= yy < h):
                                    continue
                                pix = int(starts[l]) + int(yy) * w + int(xx)
                                v = value[b, pix, m]
                                sampled += wy * wx * v
                                dsdx += wy * dwx * v
                                dsdy += dwy * wx * v
                                gv[b, pix, m] += a * wy * wx * g
                        ga[b, q, m, l, k] = g @ sampled
                        gl[b, q, m, l, k, 0] = a * w * (g @ dsdx)
                        gl[b, q, m, l, k, 1] = a * h * (g @ dsdy)
    return gv, gl, ga


# ---------------------------------------------------------------------------
# grid_sample restatement (library routine, fp64, CPU)
# ---------------------------------------------------------------------------

def gridsample_forward(value, shapes, starts, loc, attn):
    """The operator as a weighted sum of torch grid_sample lookups.

    Arguments are fp64 torch CPU tensors in the operator's layouts; the result
    is differentiable with torch autograd.  Returns out [B, Q, M*D].
    """
    import torch
    import torch.nn.functional as F

    B, S, M, D = value.shape
    Q, L, K = loc.shape[1], loc.shape[3], loc.shape[4]
    out = torch.zeros(B * M, D, Q, dtype=value.dtype)
    for l in range(L):
        h, w = int(shapes[l, 0]), int(shapes[l, 1])
        st = int(starts[l])
        v_l = value[:, st:st + h * w].reshape(B, h, w, M, D).permute(0, 3, 4, 1, 2).reshape(B * M, D, h, w)
        grid = 2.0 * loc[:, :, :, l] - 1.0                        # [B,Q,M,K,2], (x, y) in [-1, 1]
        grid = grid.permute(0, 2, 1, 3, 4).reshape(B * M, Q, K, 2)
        s = F.grid_sample(v_l, grid, mode="bilinear", padding_mode="zeros", align_corners=False)  # [BM,D,Q,K]
        a = attn[:, :, :, l].permute(0, 2, 1, 3).reshape(B * M, 1, Q, K)
        out = out + (s * a).sum(-1)
    return out.reshape(B, M, D, Q).permute(0, 3, 1, 2).reshape(B, Q, M * D)
