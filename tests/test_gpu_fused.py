"""The fused operator (msda-triton README, "The operator": softmax-normalised
weights over the L*K (level, point) pairs, sampling location = reference point
+ offset / (W_l, H_l)) through the C ABI, against the oracle's chain rule
around its core (``oracle.fused_forward`` / ``oracle.fused_backward``).

Same tolerances as the core's parity tests; covers every dtype and
accumulator, L*K above one team's point lanes, wide logits, ragged tails,
empty inputs, accumulation, autograd and the unsupported-row error.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
import workloads as W
from msda_testutil import assert_forward, assert_grad, f64, rel_l2, to_torch

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
    assert msda.device_errors(clear=True) == 0, "a kernel raised a device error bit"


def _msda():
    import scale_deformable_attention_gb300 as msda

    return msda


@functools.lru_cache(maxsize=None)
def _case(name: str, items=()):
    wl = W.WORKLOADS[name].with_(**dict(items)) if items else W.WORKLOADS[name]
    return wl, W.make_fused_inputs(wl)


def _args(t):
    return (t["value"], t["spatial_shapes"], t["level_start_index"], t["reference_points"], t["sampling_offsets"],
            t["attention_logits"])


def _run(wl, inp, accum):
    msda = _msda()
    t = to_torch(inp, wl.dtype, DEV)
    out = msda.forward_fused(*_args(t))
    grads = msda.backward_fused(*_args(t), t["grad_out"], accum=accum)
    torch.cuda.synchronize()
    return out, grads


def _check(wl, inp, accum, what):
    out, (gv, gr, go, gz) = _run(wl, inp, accum)
    assert_forward(wl.dtype, f64(out), oracle.fused_forward(inp, wl.dtype), f"{what} out")
    rgv, rgr, rgo, rgz = oracle.fused_backward(inp, wl.dtype)
    assert_grad(wl.dtype, f64(gz), rgz, f"{what} grad_attention_logits")
    assert_grad(wl.dtype, f64(go), rgo, f"{what} grad_sampling_offsets")
    assert_grad(wl.dtype, f64(gr), rgr, f"{what} grad_reference_points")
    assert_grad(wl.dtype, f64(gv), rgv, f"{what} grad_value")


CASES = [
    ("tiny_fp32", (("D", 16), ("B", 2), ("Q", 37)), "auto"),
    ("tiny_fp32", (("D", 32), ("dtype", "bf16")), "native"),
    ("tiny_fp32", (("D", 32), ("dtype", "f16")), "fp32"),
    ("tiny_fp32", (("D", 48), ("B", 3), ("Q", 261)), "deterministic"),   # several blocks + ragged tail
    ("decoder_bf16", (), "native"),
    ("decoder_bf16", (), "fp32"),
    ("decoder_bf16", (), "deterministic"),
    ("decoder_bf16", (("Q", 301), ("B", 3)), "auto"),
    ("decoder_bf16", (("dtype", "f32"), ("B", 2)), "auto"),
    ("decoder_bf16", (("dtype", "f16"), ("B", 2), ("D", 64)), "native"),
    ("decoder_bf16", (("D", 96), ("B", 2)), "fp32"),
    ("decoder_bf16", (("D", 128), ("B", 2)), "native"),                 # 256-byte rows
    ("decoder_bf16", (("D", 64), ("B", 2), ("dtype", "f32")), "auto"),
    ("decoder_bf16", (("D", 128), ("B", 2), ("dtype", "f16")), "fp32"),
    ("decoder_bf16", (("D", 128), ("B", 2)), "deterministic"),
    ("encoder_fp16", (("B", 1),), "native"),
    ("encoder_fp16", (("B", 1),), "deterministic"),
    ("oddD_fp32", (("B", 2),), "auto"),
]


@pytest.mark.parametrize("name,items,accum", CASES, ids=[f"{n}-{dict(i)}-{a}" for n, i, a in CASES])
def test_fused_parity(name, items, accum):
    wl, inp = _case(name, items)
    _check(wl, inp, accum, name)


@pytest.mark.parametrize("dtype,D,L,K", [("f32", 16, 1, 1), ("bf16", 32, 3, 5), ("f32", 32, 4, 16),
                                         ("bf16", 32, 16, 16), ("f16", 64, 4, 64), ("bf16", 96, 2, 3)])
def test_fused_levels_points(dtype, D, L, K):
    """L*K from 1 to 256: the softmax over L*K spans several rounds of a
    team's point lanes, and L*K need not divide them."""
    shapes = tuple((max(2, 24 >> l), max(2, 32 >> l)) for l in range(L))
    wl = W.WORKLOADS["tiny_fp32"].with_(dtype=dtype, D=D, K=K, shapes=shapes, B=2, Q=45, M=3)
    _check(wl, W.make_fused_inputs(wl), "auto", f"L={L} K={K}")


def test_fused_wide_logits():
    """Logits of magnitude ~100: the softmax must subtract its maximum."""
    wl = W.WORKLOADS["tiny_fp32"].with_(D=16, B=2, Q=64, M=4, K=4)
    inp = dict(W.make_fused_inputs(wl))
    inp["attention_logits"] = (inp["attention_logits"] * 60.0).astype(np.float32)
    _check(wl, inp, "auto", "wide logits")


def test_fused_accumulate_and_autograd():
    msda = _msda()
    wl, inp = _case("decoder_bf16", (("dtype", "f32"), ("B", 1), ("Q", 77)))
    t = to_torch(inp, wl.dtype, DEV)
    gv, gr, go, gz = msda.backward_fused(*_args(t), t["grad_out"])
    base = torch.randn_like(t["value"])
    acc = base.clone()
    msda.backward_fused(*_args(t), t["grad_out"], grad_value=acc, accumulate=True)
    assert rel_l2(f64(acc), f64(base) + f64(gv)) <= 1e-5

    leaves = [t[k].clone().requires_grad_(True) for k in ("value", "reference_points", "sampling_offsets",
                                                          "attention_logits")]
    out = msda.multi_scale_deformable_attention_fused(leaves[0], t["spatial_shapes"], t["level_start_index"],
                                                      *leaves[1:])
    assert torch.equal(out, msda.forward_fused(*_args(t)))
    out.backward(t["grad_out"])
    # per-sample gradients are written once, in a fixed order: equal bits
    assert torch.equal(leaves[1].grad, gr)
    assert torch.equal(leaves[2].grad, go)
    assert torch.equal(leaves[3].grad, gz)
    assert rel_l2(f64(leaves[0].grad), f64(gv)) <= 1e-6


def test_fused_deterministic_repeats_bitwise():
    msda = _msda()
    wl, inp = _case("decoder_bf16", ())
    t = to_torch(inp, wl.dtype, DEV)
    first = msda.backward_fused(*_args(t), t["grad_out"], accum="deterministic")
    for _ in range(2):
        again = msda.backward_fused(*_args(t), t["grad_out"], accum="deterministic")
        for a, b in zip(first, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("over", [dict(B=0), dict(Q=0)])
def test_fused_empty(over):
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"].with_(D=16, **over)
    t = to_torch(W.make_fused_inputs(wl), wl.dtype, DEV)
    out = msda.forward_fused(*_args(t))
    assert out.numel() == 0
    gv, gr, go, gz = msda.backward_fused(*_args(t), t["grad_out"])
    torch.cuda.synchronize()
    assert gv.abs().sum().item() == 0 and gr.numel() == 0 and go.numel() == 0 and gz.numel() == 0


@pytest.mark.parametrize("dtype,D", [("f32", 8), ("bf16", 16), ("f32", 80), ("bf16", 5), ("bf16", 160)])
def test_fused_rejects_rows_it_cannot_vectorise(dtype, D):
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"].with_(dtype=dtype, D=D)
    t = to_torch(W.make_fused_inputs(wl), wl.dtype, DEV)
    with pytest.raises(msda._lib.MsdaError, match="fused operator"):
        msda.forward_fused(*_args(t))
    with pytest.raises(msda._lib.MsdaError, match="fused operator"):
        msda.backward_fused(*_args(t), t["grad_out"])


@pytest.mark.parametrize("M", [1, 16, 32])
def test_fused_head_counts(M):
    """grad_reference_points is reduced inside the backward when a block holds
    whole queries (units per block a multiple of M), else by a separate
    kernel: single head, many heads, and more heads than a block's units."""
    wl = W.WORKLOADS["decoder_bf16"].with_(B=2, Q=37, M=M, shapes=((30, 40), (15, 20), (8, 10), (4, 5)))
    _check(wl, W.make_fused_inputs(wl), "auto", f"M={M}")
