"""Seeded synthetic inputs for the multi-scale deformable attention sampling core.

This module is shared by the fp64 oracle's tests, the GPU parity tests and the
benchmark.  It holds no part of the operator's arithmetic: it only draws random
numbers, shapes them into the operator's tensor layouts and rounds them to the
I/O dtype, so that the oracle and the CUDA path consume byte-identical inputs.

Layouts (msda-triton README, "Quickstart"; course ch. 4, "Setup"):

* ``value``               ``[B, S, M, D]``   S = sum over levels of H_l * W_l
* ``spatial_shapes``      ``[L, 2]`` int64, rows are ``(H_l, W_l)``
* ``level_start_index``   ``[L]`` int64, exclusive prefix sum of H_l * W_l
* ``sampling_locations``  ``[B, Q, M, L, K, 2]``, last axis is ``(x, y)`` in [0, 1]
* ``attention_weights``   ``[B, Q, M, L, K]``
* ``grad_out``            ``[B, Q, M * D]``

Half-precision arrays are stored as raw bits: ``float16`` for fp16 and
``uint16`` holding the upper half of an IEEE binary32 for bf16.

Distributions are those of the five named workloads below (the decoder and
encoder presets mirror the README's "Benchmarks" operating points: an
800x1333 image pyramid, hidden size 256 = 8 heads x 32, L = K = 4).  No trained
weights exist, so learned offsets are replaced by uniform / Gaussian draws.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16")
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes, I/O dtype and input distributions."""

    name: str
    B: int
    M: int
    D: int
    K: int
    shapes: Tuple[Tuple[int, int], ...]
    Q: Optional[int]          # None: one query per pyramid pixel (Q = S)
    dtype: str                # "f32" | "f16" | "bf16"
    loc: str                  # "uniform01" | "uniform_wide" | "pixel_centres"
    logits: str               # "normal" | "uniform01"
    seed: int
    accum: str = "auto"       # grad_value accumulator the workload asks for

    @property
    def L(self) -> int:
        return len(self.shapes)

    @property
    def S(self) -> int:
        return int(sum(h * w for h, w in self.shapes))

    @property
    def Qn(self) -> int:
        return self.S if self.Q is None else int(self.Q)

    @property
    def units(self) -> int:
        """Number of (b, q, m) output vectors."""
        return self.B * self.Qn * self.M

    @property
    def samples(self) -> int:
        return self.units * self.L * self.K

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


_PYRAMID_800x1333 = ((100, 167), (50, 84), (25, 42), (13, 21))

WORKLOADS: Dict[str, Workload] = {
    # small correctness case, exercises out-of-bounds corners
    "tiny_fp32": Workload("tiny_fp32", B=1, M=2, D=8, K=2, shapes=((6, 8), (3, 4)), Q=10,
                          dtype="f32", loc="uniform_wide", logits="normal", seed=0),
    # decoder cross-attention: 300 object queries per image
    "decoder_bf16": Workload("decoder_bf16", B=4, M=8, D=32, K=4, shapes=_PYRAMID_800x1333, Q=300,
                             dtype="bf16", loc="uniform01", logits="uniform01", seed=1),
    # encoder self-attention: every pyramid pixel is a query
    "encoder_fp16": Workload("encoder_fp16", B=2, M=8, D=32, K=4, shapes=_PYRAMID_800x1333, Q=None,
                             dtype="f16", loc="pixel_centres", logits="normal", seed=2),
    # head dim that is not a power of two
    "oddD_fp32": Workload("oddD_fp32", B=8, M=8, D=48, K=4,
                          shapes=((128, 128), (64, 64), (32, 32), (16, 16)), Q=900,
                          dtype="f32", loc="uniform01", logits="normal", seed=3),
    # B*S*M*D*esize far above 2^31 bytes: 64-bit addressing
    "stress_bf16": Workload("stress_bf16", B=8, M=8, D=32, K=4,
                            shapes=((768, 1024), (384, 512), (192, 256), (96, 128)), Q=20000,
                            dtype="bf16", loc="uniform01", logits="uniform01", seed=4, accum="fp32"),
}


# ---------------------------------------------------------------------------
# dtype rounding / decoding (storage only; no operator arithmetic)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round binary32 values to bfloat16 (round to nearest, ties to even); return raw bits."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def cast(x64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> storage array of ``dtype`` (RNE; bf16 goes through binary32)."""
    if dtype == "f32":
        return x64.astype(np.float32)
    if dtype == "f16":
        return x64.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x64.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array of ``dtype`` -> exact fp64 values."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def level_start_index(shapes) -> np.ndarray:
    hw = np.array([h * w for h, w in shapes], dtype=np.int64)
    return np.concatenate([[0], np.cumsum(hw)[:-1]]).astype(np.int64)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def _normal_cast(rng: np.random.Generator, n: int, dtype: str, chunk: int = 1 << 24) -> np.ndarray:
    """n draws of N(0, 1) cast to ``dtype``, generated in chunks to bound host memory."""
    out = np.empty(n, dtype={"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype])
    for i in range(0, n, chunk):
        j = min(n, i + chunk)
        out[i:j] = cast(rng.standard_normal(j - i), dtype)
    return out


def _softmax_lastaxis(z: np.ndarray) -> np.ndarray:
    # Input preparation: attention weights arrive already normalised, as the
    # README's quickstart builds them; the operator itself does not renormalise.
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _pixel_centres(shapes) -> np.ndarray:
    """[S, 2] normalised (x, y) centres of every pyramid pixel, level-major, row-major."""
    pts = []
    for h, w in shapes:
        ii, jj = np.meshgrid(np.arange(h), np.arange(w), indexing="ij")
        pts.append(np.stack([((jj + 0.5) / w).ravel(), ((ii + 0.5) / h).ravel()], axis=-1))
    return np.concatenate(pts, axis=0)


def make_inputs(wl: Workload, *, with_grad: bool = True) -> Dict[str, np.ndarray]:
    """Draw one batch of inputs for ``wl`` (deterministic in ``wl.seed``).

    Draw order from one PCG64 stream: value, sampling locations, attention
    logits, grad_out.  All floats are drawn in fp64 and rounded once to the
    workload's dtype.
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, M, D, L, K, S, Q = wl.B, wl.M, wl.D, wl.L, wl.K, wl.S, wl.Qn
    shapes = np.array(wl.shapes, dtype=np.int64).reshape(L, 2)

    value = _normal_cast(rng, B * S * M * D, wl.dtype).reshape(B, S, M, D)

    n_loc = B * Q * M * L * K
    if wl.loc == "uniform01":
        loc = rng.random(n_loc * 2)
    elif wl.loc == "uniform_wide":
        loc = rng.uniform(-0.1, 1.1, n_loc * 2)
    elif wl.loc == "pixel_centres":
        if Q != S:
            raise ValueError("pixel_centres needs one query per pyramid pixel (Q == S)")
        ref = _pixel_centres(wl.shapes)                       # [S, 2]
        off = rng.normal(0.0, 0.02, (B, Q, M, L, K, 2))
        loc = np.clip(ref[None, :, None, None, None, :] + off, -0.05, 1.05).ravel()
    else:
        raise ValueError(f"unknown location distribution {wl.loc!r}")
    loc = cast(loc, wl.dtype).reshape(B, Q, M, L, K, 2)

    if wl.logits == "normal":
        z = rng.standard_normal((B, Q, M, L * K))
    elif wl.logits == "uniform01":
        z = rng.random((B, Q, M, L * K))
    else:
        raise ValueError(f"unknown logit distribution {wl.logits!r}")
    attn = cast(_softmax_lastaxis(z), wl.dtype).reshape(B, Q, M, L, K)

    out = {
        "value": value,
        "spatial_shapes": shapes,
        "level_start_index": level_start_index(wl.shapes),
        "sampling_locations": loc,
        "attention_weights": attn,
    }
    if with_grad:
        out["grad_out"] = _normal_cast(rng, B * Q * M * D, wl.dtype).reshape(B, Q, M * D)
    return out


def make_fused_inputs(wl: Workload, *, with_grad: bool = True) -> Dict[str, np.ndarray]:
    """Inputs of the fused operator (reference points, pixel offsets, attention
    logits) for ``wl``'s sizes and dtype.  Draw order from one PCG64 stream
    (seed + 100): value, reference points, offsets, logits, grad_out.

    * uniform01 / uniform_wide: reference points ~ U[0,1) / U[-0.1,1.1) per
      (b, q, l); offsets ~ N(0, 2) pixels of level l.
    * pixel_centres: the reference point of query q is pyramid pixel q's centre
      (as the unfused encoder workload); offsets ~ N(0, 0.02 * (W_l, H_l)) pixels.
    * logits as the workload's attention logits.
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed + 100))
    B, M, D, L, K, S, Q = wl.B, wl.M, wl.D, wl.L, wl.K, wl.S, wl.Qn
    shapes = np.array(wl.shapes, dtype=np.int64).reshape(L, 2)
    value = _normal_cast(rng, B * S * M * D, wl.dtype).reshape(B, S, M, D)
    if wl.loc == "pixel_centres":
        if Q != S:
            raise ValueError("pixel_centres needs one query per pyramid pixel (Q == S)")
        ref = np.broadcast_to(_pixel_centres(wl.shapes)[None, :, None, :], (B, Q, L, 2)).copy()
        scale = 0.02 * np.stack([shapes[:, 1], shapes[:, 0]], axis=-1)            # [L,2] (W, H)
        off = rng.standard_normal((B, Q, M, L, K, 2)) * scale[None, None, None, :, None, :]
    else:
        lo, hi = (-0.1, 1.1) if wl.loc == "uniform_wide" else (0.0, 1.0)
        ref = rng.uniform(lo, hi, (B, Q, L, 2))
        off = rng.normal(0.0, 2.0, (B, Q, M, L, K, 2))
    if wl.logits == "normal":
        z = rng.standard_normal((B, Q, M, L * K))
    else:
        z = rng.random((B, Q, M, L * K))
    out = {
        "value": value,
        "spatial_shapes": shapes,
        "level_start_index": level_start_index(wl.shapes),
        "reference_points": cast(ref, wl.dtype).reshape(B, Q, L, 2),
        "sampling_offsets": cast(off, wl.dtype).reshape(B, Q, M, L, K, 2),
        "attention_logits": cast(z, wl.dtype).reshape(B, Q, M, L * K),
    }
    if with_grad:
        out["grad_out"] = _normal_cast(rng, B * Q * M * D, wl.dtype).reshape(B, Q, M * D)
    return out


def scaled(name: str, **kw) -> Workload:
    """A named workload with some sizes overridden (for oracle-sized parity cases)."""
    return WORKLOADS[name].with_(**kw)


FLOAT_KEYS = ("value", "sampling_locations", "attention_weights", "grad_out", "reference_points",
              "sampling_offsets", "attention_logits")


def to_torch(inp: Dict[str, np.ndarray], dtype: str, device):
    """Same bytes as torch tensors on ``device`` (bf16 raw bits viewed as torch.bfloat16)."""
    import torch

    out = {}
    for k, a in inp.items():
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype == "bf16" and k in FLOAT_KEYS:
            t = t.view(torch.bfloat16)
        out[k] = t.to(device)
    return out
