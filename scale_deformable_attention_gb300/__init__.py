"""GB300 (sm_103a) multi-scale deformable attention sampling core.

The bracketed term of MSDA(q) = sum_m W_m [sum_l sum_k A_mlqk x_l(phi_l(p_q) + dp_mlqk)]
(msda-triton README, "The operator") and its three gradients, computed by the
hand-written CUDA kernels of ``libmsda.so`` behind the C ABI of
``include/msda.h``.  This module only marshals torch tensors into that ABI:
it checks shapes, dtypes and devices, makes inputs contiguous, allocates
outputs (and the fp32 workspace of the FP32 accumulator) with torch, and
passes raw pointers and the current CUDA stream.

Entry points:

* ``multi_scale_deformable_attention(value, spatial_shapes, level_start_index,
  sampling_locations, attention_weights, fp32_grad_accum=None)`` -- the
  differentiable operator (signature of the README's quickstart);
* ``forward(...)`` / ``backward(...)`` -- the two C-ABI calls;
* ``multi_scale_deformable_attention_fused(...)``, ``forward_fused(...)`` /
  ``backward_fused(...)`` -- the fused operator (softmax of the attention
  logits and reference point + offset / (W, H) inside the kernels);
* ``device_errors()``, ``trace_enable()`` / ``trace_read()`` -- diagnostics;
* ``reduction_ceiling()`` -- the L2's rate for the backward's reduction
  traffic, for roofline reporting.
"""
from __future__ import annotations

import ctypes
import threading
import weakref
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import ACCUM, BWD_ACCUMULATE, BWD_WORKSPACE_ZEROED, MsdaError

__all__ = ["multi_scale_deformable_attention", "multi_scale_deformable_attention_fused", "forward", "backward",
           "forward_fused", "backward_fused", "workspace_size", "resolve_accum",
           "device_errors", "trace_enable", "trace_pause", "trace_read", "MsdaError", "DTYPE_CODE"]

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


# Host-side checks of spatial_shapes without a per-call host synchronisation.
# A CPU tensor is checked directly and copied to the device once; a device
# tensor is read back once, the first time it is seen.  Both results are
# remembered per tensor object and its version counter (an in-place change
# invalidates them), and forgotten when the tensor is freed.  The kernels check
# every level on the device as well, so a shape that escapes these host checks
# reads nothing out of bounds: it is treated as empty and raises device error
# bit 0.
_seen_lock = threading.Lock()
_shapes_ok = {}      # id(tensor) -> (weakref, version, S)
_device_copy = {}    # (id(tensor), device) -> (weakref, version, device tensor)
_lsi_of = {}         # id(device spatial_shapes) -> (weakref, version, its level_start_index)
_CACHE_MAX = 256


def _remember(table, key, t, payload):
    with _seen_lock:
        if len(table) >= _CACHE_MAX:
            table.clear()
        table[key] = (weakref.ref(t), t._version, payload)


def _recall(table, key, t):
    with _seen_lock:
        e = table.get(key)
    if e is not None and e[0]() is t and e[1] == t._version:
        return e[2]
    return None


def _check_shapes(spatial_shapes: torch.Tensor, S: int) -> None:
    if spatial_shapes.device.type != "cpu" and _recall(_shapes_ok, id(spatial_shapes), spatial_shapes) == S:
        return
    if spatial_shapes.device.type != "cpu" and torch.cuda.is_current_stream_capturing():
        raise RuntimeError("spatial_shapes on the device cannot be checked while a CUDA graph is being captured: "
                           "make one call with it before capturing, or pass validate=False")
    hw = spatial_shapes.to("cpu", torch.int64)     # a device tensor syncs here, once
    if bool((hw <= 0).any()):
        raise ValueError(f"spatial_shapes must be positive, got {hw.tolist()}")
    tot = int((hw[:, 0] * hw[:, 1]).sum())
    if tot != S:
        raise ValueError(f"value has S={S} rows but sum(H*W) over spatial_shapes is {tot}")
    if spatial_shapes.device.type != "cpu":
        _remember(_shapes_ok, id(spatial_shapes), spatial_shapes, S)


def _on_device(t: torch.Tensor, dev: torch.device) -> torch.Tensor:
    """``t`` as a contiguous int64 tensor on ``dev``; a CPU tensor is copied once
    (a copy from pageable host memory waits for the stream) and reused."""
    if t.device == dev and t.dtype == torch.int64 and t.is_contiguous():
        return t
    if t.device.type == "cpu":
        key = (id(t), str(dev))
        hit = _recall(_device_copy, key, t)
        if hit is not None:
            return hit
        d = t.to(dev, torch.int64).contiguous()
        _remember(_device_copy, key, t, d)
        return d
    return t.to(dev, torch.int64).contiguous()


def level_start_index_of(spatial_shapes: torch.Tensor) -> torch.Tensor:
    """Exclusive prefix sum of H_l * W_l (what the README's wrapper computes when
    level_start_index is None)."""
    hw = spatial_shapes[:, 0] * spatial_shapes[:, 1]
    return torch.cat([hw.new_zeros(1), hw.cumsum(0)[:-1]])


def _prepare(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, validate: bool):
    if value.dim() != 4:
        raise ValueError(f"value must be [B, S, M, D], got shape {tuple(value.shape)}")
    B, S, M, D = value.shape
    if sampling_locations.dim() != 6 or sampling_locations.shape[-1] != 2:
        raise ValueError(f"sampling_locations must be [B, Q, M, L, K, 2], got {tuple(sampling_locations.shape)}")
    Q, L, K = sampling_locations.shape[1], sampling_locations.shape[3], sampling_locations.shape[4]
    if tuple(sampling_locations.shape) != (B, Q, M, L, K, 2):
        raise ValueError(f"sampling_locations shape {tuple(sampling_locations.shape)} does not match value "
                         f"[B={B}, S, M={M}, D]")
    if tuple(attention_weights.shape) != (B, Q, M, L, K):
        raise ValueError(f"attention_weights must be {(B, Q, M, L, K)}, got {tuple(attention_weights.shape)}")
    if value.dtype not in DTYPE_CODE:
        raise TypeError(f"unsupported dtype {value.dtype}; use float32, float16 or bfloat16")
    for name, t in (("sampling_locations", sampling_locations), ("attention_weights", attention_weights)):
        if t.dtype != value.dtype:
            raise TypeError(f"{name} is {t.dtype} but value is {value.dtype}; all float tensors share one dtype")
    dev = value.device
    if dev.type != "cuda":
        raise ValueError("the operator runs on CUDA tensors only (there is no CPU implementation)")
    for name, t in (("sampling_locations", sampling_locations), ("attention_weights", attention_weights)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, value on {dev}")
    if spatial_shapes.dim() != 2 or spatial_shapes.shape != (L, 2):
        raise ValueError(f"spatial_shapes must be [L={L}, 2], got {tuple(spatial_shapes.shape)}")
    if validate:
        _check_shapes(spatial_shapes, S)
    spatial_shapes = _on_device(spatial_shapes, dev)
    if level_start_index is None:
        level_start_index = _recall(_lsi_of, id(spatial_shapes), spatial_shapes)
        if level_start_index is None:
            level_start_index = level_start_index_of(spatial_shapes)
            _remember(_lsi_of, id(spatial_shapes), spatial_shapes, level_start_index)
    else:
        if level_start_index.shape != (L,):
            raise ValueError(f"level_start_index must be [L={L}], got {tuple(level_start_index.shape)}")
        level_start_index = _on_device(level_start_index, dev)
    dims = (B, S, M, D, L, K, Q)
    return (value.contiguous(), spatial_shapes, level_start_index, sampling_locations.contiguous(),
            attention_weights.contiguous(), dims)


def forward(value: torch.Tensor, spatial_shapes: torch.Tensor, level_start_index: Optional[torch.Tensor],
            sampling_locations: torch.Tensor, attention_weights: torch.Tensor, *, out: Optional[torch.Tensor] = None,
            validate: bool = True) -> torch.Tensor:
    """out[B, Q, M*D] on the current stream (C ABI ``msda_forward``)."""
    value, ss, lsi, loc, attn, dims = _prepare(value, spatial_shapes, level_start_index, sampling_locations,
                                               attention_weights, validate)
    B, S, M, D, L, K, Q = dims
    if out is None:
        out = torch.empty((B, Q, M * D), dtype=value.dtype, device=value.device)
    elif out.shape != (B, Q, M * D) or out.dtype != value.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, Q, M*D] tensor of value's dtype")
    with torch.cuda.device(value.device):
        _lib.check(_lib.lib().msda_forward(DTYPE_CODE[value.dtype], *dims, _ptr(value), _ptr(ss), _ptr(lsi),
                                           _ptr(loc), _ptr(attn), _ptr(out), _stream(value.device)))
    return out


def resolve_accum(dtype: torch.dtype, accum: str, dims) -> str:
    """Which grad_value accumulator ("native", "fp32" or "deterministic") the backward uses."""
    r = _lib.lib().msda_resolve_accum(DTYPE_CODE[dtype], ACCUM[accum], *dims)
    return _lib.ACCUM_NAMES[r]


def workspace_size(dtype: torch.dtype, accum: str, dims, aligned: bool = True) -> int:
    """Bytes of workspace the backward needs (C ABI ``msda_backward_workspace_size``).
    The FP32 accumulator's figure assumes 16-byte aligned value, grad_out and
    grad_value; ``aligned=False`` gives what it needs otherwise (the fp32
    mirror of grad_value, B*S*M*D*4 bytes, when that is larger)."""
    n = int(_lib.lib().msda_backward_workspace_size(DTYPE_CODE[dtype], ACCUM[accum], *dims))
    if n and not aligned and resolve_accum(dtype, accum, dims) == "fp32":
        B, S, M, D = dims[:4]
        n = max(n, B * S * M * D * 4)
    return n


def _aligned16(*ts) -> bool:
    return all(t.data_ptr() % 16 == 0 for t in ts)


def backward(value: torch.Tensor, spatial_shapes: torch.Tensor, level_start_index: Optional[torch.Tensor],
             sampling_locations: torch.Tensor, attention_weights: torch.Tensor, grad_out: torch.Tensor, *,
             accum: str = "auto", grad_value: Optional[torch.Tensor] = None, accumulate: bool = False,
             workspace: Optional[torch.Tensor] = None, workspace_zeroed: bool = False, validate: bool = True
             ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(grad_value, grad_sampling_locations, grad_attention_weights) (C ABI ``msda_backward``).

    ``accum``: "auto" | "native" | "fp32" accumulator of grad_value for fp16 / bf16, or
    "deterministic" (any dtype: run-to-run bit-identical grad_value).
    ``accumulate``: add into the given ``grad_value`` instead of overwriting it.
    ``workspace_zeroed``: the given ``workspace`` holds zeros, and is left holding zeros
    (MSDA_BWD_WORKSPACE_ZEROED: a persistent workspace skips the FP32 accumulator's clearing pass).
    """
    value, ss, lsi, loc, attn, dims = _prepare(value, spatial_shapes, level_start_index, sampling_locations,
                                               attention_weights, validate)
    B, S, M, D, L, K, Q = dims
    if accum not in ACCUM:
        raise ValueError(f"accum must be one of {sorted(ACCUM)}, got {accum!r}")
    if grad_out.shape != (B, Q, M * D) or grad_out.dtype != value.dtype or grad_out.device != value.device:
        raise ValueError(f"grad_out must be a [B, Q, M*D] {value.dtype} tensor on {value.device}")
    grad_out = grad_out.contiguous()
    if grad_value is None:
        if accumulate:
            raise ValueError("accumulate=True needs grad_value")
        grad_value = torch.empty_like(value)
    elif grad_value.shape != value.shape or grad_value.dtype != value.dtype or not grad_value.is_contiguous():
        raise ValueError("grad_value must be a contiguous tensor shaped and typed like value")
    grad_loc = torch.empty_like(loc)
    grad_attn = torch.empty_like(attn)
    need = workspace_size(value.dtype, accum, dims, _aligned16(value, grad_out, grad_value))
    if need and workspace is None:
        workspace = torch.empty((need + 3) // 4, dtype=torch.float32, device=value.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if workspace_zeroed and workspace is None:
        raise ValueError("workspace_zeroed=True needs the workspace it describes")
    flags = (BWD_ACCUMULATE if accumulate else 0) | (BWD_WORKSPACE_ZEROED if workspace_zeroed else 0)
    with torch.cuda.device(value.device):
        _lib.check(_lib.lib().msda_backward(
            DTYPE_CODE[value.dtype], ACCUM[accum], flags, *dims, _ptr(value), _ptr(ss), _ptr(lsi), _ptr(loc),
            _ptr(attn), _ptr(grad_out), _ptr(grad_value), _ptr(grad_loc), _ptr(grad_attn), _ptr(workspace),
            ws_bytes, _stream(value.device)))
    return grad_value, grad_loc, grad_attn


_ws_bytes = {}   # (dtype, accum, dims) -> workspace bytes of an aligned call


def _workspace_for(dtype, accum, dims) -> int:
    key = (dtype, accum, dims)
    n = _ws_bytes.get(key)
    if n is None:
        if len(_ws_bytes) >= _CACHE_MAX:
            _ws_bytes.clear()
        n = _ws_bytes[key] = workspace_size(dtype, accum, dims)
    return n


class _MSDAFunction(torch.autograd.Function):
    """Autograd wrapper (course ch. 5, "The autograd wrapper"): saves the inputs
    and recomputes the bilinear setup in the backward kernel; the backward is
    not itself differentiable.  The inputs are checked once, in the forward;
    both passes then call the C ABI directly (the dispatch cost per call is
    what the README's "Benchmarks" measurement pitfalls are about)."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, sampling_locations, attention_weights, accum):
        value, ss, lsi, loc, attn, dims = _prepare(value, spatial_shapes, level_start_index, sampling_locations,
                                                   attention_weights, True)
        B, S, M, D, L, K, Q = dims
        out = torch.empty((B, Q, M * D), dtype=value.dtype, device=value.device)
        dev = value.device
        with torch.cuda.device(dev):
            _lib.check(_lib.lib().msda_forward(DTYPE_CODE[value.dtype], *dims, _ptr(value), _ptr(ss), _ptr(lsi),
                                               _ptr(loc), _ptr(attn), _ptr(out), _stream(dev)))
        ctx.save_for_backward(value, ss, lsi, loc, attn)
        ctx.accum = accum
        ctx.dims = dims
        return out

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, grad_out):
        value, ss, lsi, loc, attn = ctx.saved_tensors
        dims = ctx.dims
        if grad_out.dtype != value.dtype:
            grad_out = grad_out.to(value.dtype)
        grad_out = grad_out.contiguous()
        gv = torch.empty_like(value)
        gl = torch.empty_like(loc)
        ga = torch.empty_like(attn)
        if _aligned16(value, grad_out, gv):
            need = _workspace_for(value.dtype, ctx.accum, dims)
        else:
            need = workspace_size(value.dtype, ctx.accum, dims, False)
        ws = torch.empty((need + 3) // 4, dtype=torch.float32, device=value.device) if need else None
        dev = value.device
        with torch.cuda.device(dev):
            _lib.check(_lib.lib().msda_backward(
                DTYPE_CODE[value.dtype], ACCUM[ctx.accum], 0, *dims, _ptr(value), _ptr(ss), _ptr(lsi), _ptr(loc),
                _ptr(attn), _ptr(grad_out), _ptr(gv), _ptr(gl), _ptr(ga), _ptr(ws), need, _stream(dev)))
        return gv, None, None, gl, ga, None


def multi_scale_deformable_attention(value: torch.Tensor, spatial_shapes: torch.Tensor,
                                     level_start_index: Optional[torch.Tensor], sampling_locations: torch.Tensor,
                                     attention_weights: torch.Tensor, fp32_grad_accum: Optional[bool] = None
                                     ) -> torch.Tensor:
    """Differentiable MSDA sampling core, out[B, Q, M*D].

    ``fp32_grad_accum``: None lets the library choose the grad_value
    accumulator for fp16 / bf16; True forces the fp32 workspace; False forces
    native 16-bit atomic adds.
    """
    accum = "auto" if fp32_grad_accum is None else ("fp32" if fp32_grad_accum else "native")
    return _MSDAFunction.apply(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, accum)


def _prepare_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets, attention_logits,
                   validate: bool):
    if sampling_offsets.dim() != 6 or sampling_offsets.shape[-1] != 2:
        raise ValueError(f"sampling_offsets must be [B, Q, M, L, K, 2], got {tuple(sampling_offsets.shape)}")
    B, Q, M, L, K, _ = sampling_offsets.shape
    if tuple(attention_logits.shape) != (B, Q, M, L * K):
        raise ValueError(f"attention_logits must be {(B, Q, M, L * K)}, got {tuple(attention_logits.shape)}")
    if tuple(reference_points.shape) != (B, Q, L, 2):
        raise ValueError(f"reference_points must be {(B, Q, L, 2)}, got {tuple(reference_points.shape)}")
    for name, t in (("reference_points", reference_points), ("attention_logits", attention_logits)):
        if t.dtype != value.dtype or t.device != value.device:
            raise TypeError(f"{name} must be a {value.dtype} tensor on {value.device}")
    # the shared checks, with the logits viewed in the weights' layout
    value, ss, lsi, off, logit5, dims = _prepare(value, spatial_shapes, level_start_index, sampling_offsets,
                                                 attention_logits.reshape(B, Q, M, L, K), validate)
    return value, ss, lsi, reference_points.contiguous(), off, logit5.reshape(B, Q, M, L * K), dims


def forward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets, attention_logits, *,
                  out=None, validate: bool = True) -> torch.Tensor:
    """Fused operator (C ABI ``msda_forward_fused``): A = softmax of the logits
    over L*K, loc = reference point + offset / (W_l, H_l), out[B, Q, M*D]."""
    value, ss, lsi, ref, off, logit, dims = _prepare_fused(value, spatial_shapes, level_start_index,
                                                           reference_points, sampling_offsets, attention_logits,
                                                           validate)
    B, S, M, D, L, K, Q = dims
    if out is None:
        out = torch.empty((B, Q, M * D), dtype=value.dtype, device=value.device)
    with torch.cuda.device(value.device):
        _lib.check(_lib.lib().msda_forward_fused(DTYPE_CODE[value.dtype], *dims, _ptr(value), _ptr(ss), _ptr(lsi),
                                                 _ptr(ref), _ptr(off), _ptr(logit), _ptr(out),
                                                 _stream(value.device)))
    return out


def backward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets, attention_logits,
                   grad_out, *, accum: str = "auto", grad_value=None, accumulate: bool = False, workspace=None,
                   validate: bool = True):
    """(grad_value, grad_reference_points, grad_sampling_offsets, grad_attention_logits)
    of the fused operator (C ABI ``msda_backward_fused``)."""
    value, ss, lsi, ref, off, logit, dims = _prepare_fused(value, spatial_shapes, level_start_index,
                                                           reference_points, sampling_offsets, attention_logits,
                                                           validate)
    B, S, M, D, L, K, Q = dims
    if grad_out.shape != (B, Q, M * D) or grad_out.dtype != value.dtype:
        raise ValueError(f"grad_out must be a [B, Q, M*D] {value.dtype} tensor")
    grad_out = grad_out.contiguous()
    if grad_value is None:
        if accumulate:
            raise ValueError("accumulate=True needs grad_value")
        grad_value = torch.empty_like(value)
    g_ref = torch.empty_like(ref)
    g_off = torch.empty_like(off)
    g_logit = torch.empty_like(logit)
    need = workspace_size(value.dtype, accum, dims)
    if need and workspace is None:
        workspace = torch.empty((need + 3) // 4, dtype=torch.float32, device=value.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(value.device):
        _lib.check(_lib.lib().msda_backward_fused(
            DTYPE_CODE[value.dtype], ACCUM[accum], BWD_ACCUMULATE if accumulate else 0, *dims, _ptr(value), _ptr(ss),
            _ptr(lsi), _ptr(ref), _ptr(off), _ptr(logit), _ptr(grad_out), _ptr(grad_value), _ptr(g_ref),
            _ptr(g_off), _ptr(g_logit), _ptr(workspace), ws_bytes, _stream(value.device)))
    return grad_value, g_ref, g_off, g_logit


class _MSDAFusedFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                attention_logits, accum):
        out = forward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                            attention_logits)
        ss = _on_device(spatial_shapes, value.device)
        lsi = level_start_index_of(ss) if level_start_index is None else _on_device(level_start_index, value.device)
        ctx.save_for_backward(value, ss, lsi, reference_points, sampling_offsets, attention_logits)
        ctx.accum = accum
        return out

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, grad_out):
        value, ss, lsi, ref, off, logit = ctx.saved_tensors
        gv, gr, go, gz = backward_fused(value, ss, lsi, ref, off, logit, grad_out, accum=ctx.accum, validate=False)
        return gv, None, None, gr, go, gz, None


def multi_scale_deformable_attention_fused(value, spatial_shapes, level_start_index, reference_points,
                                           sampling_offsets, attention_logits, fp32_grad_accum=None):
    """Differentiable fused operator: softmax of the logits over L*K and
    loc = reference point + offset / (W_l, H_l) taken inside the kernels."""
    accum = "auto" if fp32_grad_accum is None else ("fp32" if fp32_grad_accum else "native")
    return _MSDAFusedFunction.apply(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                                    attention_logits, accum)


REDUCTION_KIND = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}


def reduction_ceiling(dtype=torch.bfloat16, *, row_bytes: int = 64, blocks_per_sm: int = 8, repeats: int = 5,
                      scratch_mib: int = 64, device=None) -> float:
    """32-byte sectors per second the L2 takes for the backward's kind of
    reduction traffic (C ABI ``msda_reduction_ceiling``): rows of ``row_bytes``
    at random places of a ``scratch_mib`` MiB buffer, each row taken by
    row_bytes / 16 lanes with one 16-byte ``dtype`` vector reduction each.
    Synchronises the current stream; a measurement, not an operator."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    scratch = torch.empty(scratch_mib << 20, dtype=torch.uint8, device=device)
    out = ctypes.c_double(0.0)
    with torch.cuda.device(device):
        _lib.check(_lib.lib().msda_reduction_ceiling(REDUCTION_KIND[dtype], row_bytes, blocks_per_sm, repeats,
                                                     _ptr(scratch), scratch.numel(), ctypes.byref(out),
                                                     _stream(device)))
    return out.value


def device_errors(clear: bool = True) -> int:
    """Error bits raised by kernels on the current device (bit 0: a level failed
    its shape check; bit 1: a parameter copy timed out).  Synchronises."""
    v = ctypes.c_uint32(0)
    _lib.check(_lib.lib().msda_device_errors(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def trace_enable(capacity: int) -> None:
    """Bracket every kernel launch by CUDA events (capacity launches; 0 disables)."""
    _lib.check(_lib.lib().msda_trace_enable(int(capacity)))


def trace_pause(paused: bool) -> None:
    """Stop (or resume) recording launches without destroying the trace's events."""
    _lib.lib().msda_trace_pause(1 if paused else 0)


def trace_read(max_records: int = 1 << 16):
    """[(kernel name, ms, work)] of the traced launches since the last read (waits for them)."""
    recs = (_lib.TraceRecord * max_records)()
    dropped = ctypes.c_int(0)
    n = _lib.lib().msda_trace_read(recs, max_records, ctypes.byref(dropped))
    return [(_lib.KERNEL_NAMES.get(r.kernel, str(r.kernel)), float(r.ms), int(r.work)) for r in recs[:n]], dropped.value
