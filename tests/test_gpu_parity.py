"""CUDA path vs the fp64 oracle on identical seeded inputs, through the C ABI.

Element-by-element parity on every named workload (full size where the oracle
finishes in seconds; the stress workload on sampled outputs plus size-free
properties), plus edge cases: ragged query tails, element-wise (non 16-byte)
rows, misaligned pointers, empty inputs, all-outside samples, pixel centres,
maximum L*K, large D, device-side shape checks, accumulation and autograd.
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

    msda._lib.lib()  # raises when the library is not built: no fallback exists
    msda.device_errors(clear=True)
    yield
    assert msda.device_errors(clear=True) == 0, "a kernel raised a device error bit"


def _msda():
    import scale_deformable_attention_gb300 as msda

    return msda


@functools.lru_cache(maxsize=None)
def _case(name: str, **over):
    wl = W.WORKLOADS[name].with_(**over) if over else W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    return wl, inp


@functools.lru_cache(maxsize=None)
def _oracle(name: str, items=()):
    wl, inp = _case(name, **dict(items))
    out = oracle.forward(inp, wl.dtype)
    gv, gl, ga = oracle.backward(inp, wl.dtype)
    return out, gv, gl, ga


def _run(wl, inp, accum="auto"):
    msda = _msda()
    t = to_torch(inp, wl.dtype, DEV)
    out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                       t["attention_weights"])
    gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                               t["attention_weights"], t["grad_out"], accum=accum)
    torch.cuda.synchronize()
    return out, gv, gl, ga


def _check(name, items, accum):
    wl, inp = _case(name, **dict(items))
    out, gv, gl, ga = _run(wl, inp, accum)
    rout, rgv, rgl, rga = _oracle(name, items)
    assert_forward(wl.dtype, f64(out), rout, f"{name} out")
    assert_grad(wl.dtype, f64(ga), rga, f"{name} grad_attn")
    assert_grad(wl.dtype, f64(gl), rgl, f"{name} grad_loc")
    assert_grad(wl.dtype, f64(gv), rgv, f"{name} grad_value")


# name, overrides (as a tuple of pairs, hashable), accumulator
CASES = [
    ("tiny_fp32", (), "auto"),
    ("tiny_fp32", (("dtype", "bf16"),), "native"),
    ("tiny_fp32", (("dtype", "bf16"),), "fp32"),
    ("tiny_fp32", (("dtype", "f16"),), "native"),
    ("tiny_fp32", (("B", 3), ("Q", 257)), "auto"),                      # several blocks + ragged tail
    ("decoder_bf16", (), "fp32"),
    ("decoder_bf16", (), "native"),
    ("decoder_bf16", (("Q", 301), ("B", 3)), "fp32"),                   # ragged tail
    ("decoder_bf16", (("dtype", "f32"), ("B", 2)), "auto"),
    ("decoder_bf16", (("dtype", "f16"), ("B", 2)), "native"),
    ("encoder_fp16", (), "native"),
    ("encoder_fp16", (), "fp32"),
    ("oddD_fp32", (), "auto"),
    ("oddD_fp32", (("dtype", "bf16"), ("B", 2)), "fp32"),
    ("stress_bf16", (("B", 1), ("Q", 3000), ("shapes", ((96, 128), (48, 64), (24, 32), (12, 16)))), "fp32"),
    # sparse samples, wider rows (two and three 16-byte vectors per lane) with the FP32 accumulator
    ("stress_bf16", (("B", 2), ("Q", 2000), ("shapes", ((96, 128), (48, 64), (24, 32), (12, 16)))), "fp32"),
    ("decoder_bf16", (("dtype", "f16"), ("D", 64), ("B", 2)), "fp32"),
    ("decoder_bf16", (("D", 96), ("B", 1), ("Q", 77)), "fp32"),
]


@pytest.mark.parametrize("name,items,accum", CASES, ids=[f"{n}-{dict(i)}-{a}" for n, i, a in CASES])
def test_parity(name, items, accum):
    _check(name, items, accum)


@pytest.mark.parametrize("dtype,D", [("f32", 5), ("bf16", 6), ("f16", 3), ("f32", 48), ("bf16", 256),
                                     ("bf16", 1024), ("f32", 512), ("f16", 100)])
def test_channel_widths(dtype, D):
    """Element-wise rows (D*esize not a multiple of 16) and wide rows."""
    wl = W.WORKLOADS["tiny_fp32"].with_(dtype=dtype, D=D, B=2, Q=19, M=3)
    inp = W.make_inputs(wl)
    out, gv, gl, ga = _run(wl, inp, "auto")
    assert_forward(dtype, f64(out), oracle.forward(inp, dtype), f"D={D}")
    rgv, rgl, rga = oracle.backward(inp, dtype)
    assert_grad(dtype, f64(gv), rgv, f"D={D} grad_value")
    assert_grad(dtype, f64(gl), rgl, f"D={D} grad_loc")
    assert_grad(dtype, f64(ga), rga, f"D={D} grad_attn")


@pytest.mark.parametrize("L,K", [(1, 1), (16, 16), (3, 5), (4, 64)])
def test_levels_points(L, K):
    shapes = tuple((3 + l, 4 + 2 * l) for l in range(L))
    wl = W.WORKLOADS["tiny_fp32"].with_(shapes=shapes, K=K, B=2, Q=7, M=2, D=8)
    inp = W.make_inputs(wl)
    out, gv, gl, ga = _run(wl, inp)
    assert_forward("f32", f64(out), oracle.forward(inp, "f32"))
    rgv, rgl, rga = oracle.backward(inp, "f32")
    assert_grad("f32", f64(gv), rgv, "grad_value")
    assert_grad("f32", f64(gl), rgl, "grad_loc")
    assert_grad("f32", f64(ga), rga, "grad_attn")


@pytest.mark.parametrize("dtype,D,K", [("bf16", 32, 1), ("bf16", 32, 2), ("bf16", 32, 8), ("f16", 64, 2),
                                       ("f32", 48, 1), ("f32", 32, 8), ("bf16", 96, 4)])
def test_forward_widths_and_point_counts(dtype, D, K):
    """Whole 16-byte rows with L*K in {4, 8, 16, 32} (the TMA-gather forward)
    and ragged unit counts."""
    wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, D=D, K=K, B=2, Q=37, M=3,
                                           shapes=((11, 13), (6, 7), (3, 5), (2, 2)))
    inp = W.make_inputs(wl)
    out, gv, gl, ga = _run(wl, inp, "native" if dtype != "f32" else "auto")
    assert_forward(dtype, f64(out), oracle.forward(inp, dtype), f"D={D} K={K}")
    rgv, rgl, rga = oracle.backward(inp, dtype)
    assert_grad(dtype, f64(gv), rgv, "grad_value")
    assert_grad(dtype, f64(gl), rgl, "grad_loc")
    assert_grad(dtype, f64(ga), rga, "grad_attn")


def test_misaligned_pointers_take_elementwise_path():
    """value / grad_out starting 2 bytes past a 16-byte boundary: same results."""
    msda = _msda()
    wl = W.WORKLOADS["decoder_bf16"].with_(B=1, Q=50)
    inp = W.make_inputs(wl)
    t = to_torch(inp, "bf16", DEV)
    buf = torch.empty(t["value"].numel() + 1, dtype=torch.bfloat16, device=DEV)
    v = buf[1:].view(t["value"].shape)
    v.copy_(t["value"])
    assert v.data_ptr() % 16 != 0
    out = msda.forward(v, t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                       t["attention_weights"])
    gbuf = torch.empty(t["grad_out"].numel() + 1, dtype=torch.bfloat16, device=DEV)
    g = gbuf[1:].view(t["grad_out"].shape)
    g.copy_(t["grad_out"])
    gv, gl, ga = msda.backward(v, t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                               t["attention_weights"], g, accum="native")
    torch.cuda.synchronize()
    assert_forward("bf16", f64(out), oracle.forward(inp, "bf16"))
    rgv, rgl, rga = oracle.backward(inp, "bf16")
    assert_grad("bf16", f64(gv), rgv, "grad_value")
    assert_grad("bf16", f64(gl), rgl, "grad_loc")


def test_empty_inputs():
    msda = _msda()
    for over in (dict(B=0), dict(Q=0)):
        wl = W.WORKLOADS["tiny_fp32"].with_(**over)
        inp = W.make_inputs(wl)
        t = to_torch(inp, "f32", DEV)
        out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                           t["attention_weights"])
        assert out.numel() == 0
        gv = torch.full_like(t["value"], 7.0)
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], t["grad_out"], grad_value=gv)
        torch.cuda.synchronize()
        assert gl.numel() == 0 and ga.numel() == 0
        assert bool((gv == 0).all()), "the gradient of an empty sum is zero"


def test_all_outside_and_pixel_centres():
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"].with_(B=1, Q=6, M=2, D=8)
    inp = W.make_inputs(wl)
    loc = inp["sampling_locations"].copy()
    loc[:, :3] = np.array([-3.0, 0.5], dtype=np.float32)       # far outside: x_im < -1
    loc[:, 3, :, 0, :, 0] = (2 + 0.5) / 8                         # pixel centres of level 0
    loc[:, 3, :, 0, :, 1] = (1 + 0.5) / 6
    loc[:, 4] = np.float32(np.nan)                                 # non-finite: no corner inside
    inp = dict(inp, sampling_locations=loc)
    out, gv, gl, ga = _run(wl, inp)
    out = f64(out).reshape(1, 6, 2, 8)
    assert np.all(out[:, :3] == 0) and np.all(out[:, 4] == 0)
    assert np.all(f64(gl)[:, :3] == 0) and np.all(f64(ga)[:, :3] == 0)
    assert np.all(f64(gl)[:, 4] == 0) and np.all(f64(ga)[:, 4] == 0)
    ref = oracle.forward(inp, "f32").reshape(1, 6, 2, 8)
    assert_forward("f32", out, ref)
    rgv, rgl, rga = oracle.backward(inp, "f32")
    assert_grad("f32", f64(gv), rgv, "grad_value")
    assert_grad("f32", f64(gl), rgl, "grad_loc")


def test_bad_device_shapes_are_contained():
    """A level whose start + H*W exceeds S (skipping the host check) reads
    nothing, gets zero gradient and raises device error bit 0."""
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"]
    inp = W.make_inputs(wl)
    t = to_torch(inp, "f32", DEV)
    bad_starts = torch.tensor([0, 50], dtype=torch.int64, device=DEV)   # level 1 (3x4) would end at 62 > 60
    out = msda.forward(t["value"], t["spatial_shapes"], bad_starts, t["sampling_locations"], t["attention_weights"],
                       validate=False)
    torch.cuda.synchronize()
    assert msda.device_errors(clear=True) & 1
    # equals the oracle with level 1 removed from every sample (its attention weights zeroed)
    attn = inp["attention_weights"].copy()
    attn[:, :, :, 1] = 0
    ref = oracle.forward(dict(inp, attention_weights=attn), "f32")
    assert_forward("f32", f64(out), ref)


def test_forward_is_deterministic():
    msda = _msda()
    wl, inp = _case("decoder_bf16")
    t = to_torch(inp, "bf16", DEV)
    args = (t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"], t["attention_weights"])
    a = msda.forward(*args)
    b = msda.forward(*args)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,accum,dense", [("f32", "auto", False), ("bf16", "fp32", False), ("f16", "native", False),
                                               ("bf16", "fp32", True), ("f16", "native", True)])
def test_accumulate_doubles(dtype, accum, dense):
    """Backward into the previous call's grad_value adds the same gradient again
    (up to summation order).  Dense cases (many samples per pixel) run with the
    backward's corner merge on."""
    msda = _msda()
    over = dict(shapes=((20, 24), (10, 12), (5, 6), (3, 3))) if dense else {}
    wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, B=1, Q=120, **over)
    assert (4.0 * wl.Qn * wl.L * wl.K / wl.S >= 2.0) == dense
    inp = W.make_inputs(wl)
    t = to_torch(inp, dtype, DEV)
    args = (t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"], t["attention_weights"],
            t["grad_out"])
    gv1, _, _ = msda.backward(*args, accum=accum)
    once = gv1.clone()
    gv2, _, _ = msda.backward(*args, accum=accum, grad_value=gv1, accumulate=True)
    torch.cuda.synchronize()
    lim = 1e-6 if dtype == "f32" else 1e-2
    assert rel_l2(f64(gv2), 2 * f64(once)) <= lim


def test_autograd_matches_direct_calls():
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"].with_(B=2, Q=33)
    inp = W.make_inputs(wl)
    t = to_torch(inp, "f32", DEV)
    v = t["value"].clone().requires_grad_(True)
    loc = t["sampling_locations"].clone().requires_grad_(True)
    attn = t["attention_weights"].clone().requires_grad_(True)
    out = msda.multi_scale_deformable_attention(v, t["spatial_shapes"], None, loc, attn)
    out.backward(t["grad_out"])
    gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], None, t["sampling_locations"],
                               t["attention_weights"], t["grad_out"])
    assert rel_l2(f64(v.grad), f64(gv)) <= 1e-6
    assert torch.equal(loc.grad, gl) and torch.equal(attn.grad, ga)


def test_noncontiguous_inputs():
    msda = _msda()
    wl = W.WORKLOADS["tiny_fp32"].with_(B=2, Q=21)
    inp = W.make_inputs(wl)
    t = to_torch(inp, "f32", DEV)
    # same values, permuted storage
    loc_nc = t["sampling_locations"].permute(1, 0, 2, 3, 4, 5).contiguous().permute(1, 0, 2, 3, 4, 5)
    assert not loc_nc.is_contiguous()
    out = msda.forward(t["value"], t["spatial_shapes"], None, loc_nc, t["attention_weights"])
    assert_forward("f32", f64(out), oracle.forward(inp, "f32"))


def test_adjoint_identity_on_gpu_outputs():
    """<g, out> = <grad_value, value> = <grad_attn, A> holds at any size."""
    wl, inp = _case("encoder_fp16")
    out, gv, gl, ga = _run(wl, inp, "fp32")
    g = W.to_f64(inp["grad_out"], "f16")
    lhs = float(np.sum(g * f64(out)))
    r1 = float(np.sum(f64(gv) * W.to_f64(inp["value"], "f16")))
    r2 = float(np.sum(f64(ga) * W.to_f64(inp["attention_weights"], "f16")))
    scale = float(np.sqrt(np.sum(g ** 2) * np.sum(f64(out) ** 2)))
    assert abs(lhs - r1) <= 1e-2 * scale and abs(lhs - r2) <= 1e-2 * scale


@pytest.mark.slow
def test_stress_full_size_sampled():
    """The stress workload at full size (B*S*M*D*2 bytes > 2^32): sampled
    outputs against the oracle, computed one by one."""
    msda = _msda()
    wl = W.WORKLOADS["stress_bf16"]
    inp = W.make_inputs(wl)
    t = to_torch(inp, "bf16", DEV)
    out = msda.forward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                       t["attention_weights"])
    gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                               t["attention_weights"], t["grad_out"], accum="fp32")
    torch.cuda.synchronize()
    rng = np.random.default_rng(123)
    n_units = wl.units
    units = np.unique(np.concatenate([rng.choice(n_units, 3000, replace=False), [0, n_units - 1]]))
    ref = oracle.forward_units(inp, "bf16", units)
    got = f64(out.view(n_units, wl.D)[torch.from_numpy(units).to(DEV)])
    assert_forward("bf16", got, ref, "stress out (sampled)")
    rgl, rga = oracle.backward_units(inp, "bf16", units)
    LK = wl.L * wl.K
    idx = torch.from_numpy(units).to(DEV)
    assert_grad("bf16", f64(gl.view(n_units, LK * 2)[idx]), rgl, "stress grad_loc (sampled)")
    assert_grad("bf16", f64(ga.view(n_units, LK)[idx]), rga, "stress grad_attn (sampled)")
    # grad_value rows: the last batch (highest byte offsets) and a spread of the rest
    n_rows = wl.B * wl.S * wl.M
    rows = np.unique(np.concatenate([rng.choice(n_rows, 1500, replace=False),
                                     rng.integers(n_rows - wl.S * wl.M, n_rows, 500)]))
    rgv = oracle.grad_value_rows(inp, "bf16", rows)
    got = f64(gv.view(n_rows, wl.D)[torch.from_numpy(rows).to(DEV)])
    assert_grad("bf16", got, rgv, "stress grad_value (sampled rows)")


@pytest.mark.slow
def test_stress_nine_batches_element_index_beyond_2_31():
    """The stress shapes at B=9: B*S*M*D = 2.41e9 elements, so element
    indices of the last batch pass 2^31 (not only byte offsets).  Batch 0 is
    built by the workload's generator and copied to all nine batches on the
    device; every batch must give the same forward and parameter-gradient
    bits, and the last batch must match the oracle on the one-batch problem
    (sampled units and grad_value rows)."""
    msda = _msda()
    wl1 = W.WORKLOADS["stress_bf16"].with_(B=1)
    inp = W.make_inputs(wl1)
    t1 = to_torch(inp, "bf16", DEV)
    B = 9
    assert B * wl1.S * wl1.M * wl1.D > 2 ** 31

    def rep(x):
        return x.expand(B, *x.shape[1:]).contiguous()

    value, loc, attn, g = (rep(t1[k]) for k in ("value", "sampling_locations", "attention_weights", "grad_out"))
    out = msda.forward(value, t1["spatial_shapes"], t1["level_start_index"], loc, attn)
    gv, gl, ga = msda.backward(value, t1["spatial_shapes"], t1["level_start_index"], loc, attn, g, accum="fp32")
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[B - 1]) and torch.equal(gl[0], gl[B - 1]) and torch.equal(ga[0], ga[B - 1])
    del value, loc, attn, g
    rng = np.random.default_rng(9)
    n1 = wl1.units
    units = np.unique(np.concatenate([rng.choice(n1, 2000, replace=False), [0, n1 - 1]]))
    idx = torch.from_numpy(units).to(DEV)
    assert_forward("bf16", f64(out[B - 1].reshape(n1, wl1.D)[idx]), oracle.forward_units(inp, "bf16", units),
                   "last batch out (sampled)")
    rgl, rga = oracle.backward_units(inp, "bf16", units)
    LK = wl1.L * wl1.K
    assert_grad("bf16", f64(gl[B - 1].reshape(n1, LK * 2)[idx]), rgl, "last batch grad_loc (sampled)")
    assert_grad("bf16", f64(ga[B - 1].reshape(n1, LK)[idx]), rga, "last batch grad_attn (sampled)")
    rows1 = wl1.S * wl1.M
    rows = np.unique(rng.choice(rows1, 2000, replace=False))
    got = f64(gv[B - 1].reshape(rows1, wl1.D)[torch.from_numpy(rows).to(DEV)])
    assert_grad("bf16", got, oracle.grad_value_rows(inp, "bf16", rows), "last batch grad_value (sampled rows)")


@pytest.mark.parametrize("dtype,accum,tune_merge", [("f32", "auto", True), ("bf16", "native", True),
                                                    ("bf16", "fp32", True), ("f16", "deterministic", True),
                                                    ("f32", "deterministic", True), ("bf16", "native", False)])
def test_clustered_samples_merge(dtype, accum, tune_merge):
    """Each unit's points at a level lie within about a pixel of each other,
    on levels 11, 3 and 1 pixels wide: the backward's corner merge sees
    coinciding, edge- and corner-adjacent cells and chains of them (and skips
    the narrow levels).  The inputs are dense (4*Q*L*K/S well above 2), so the
    merge is on; the last case turns the density low so it is off."""
    shapes = ((9, 11), (4, 3), (6, 1)) if tune_merge else ((60, 70), (40, 50), (30, 20))
    wl = W.WORKLOADS["tiny_fp32"].with_(dtype=dtype, D=32 if dtype != "f32" else 16, B=2, Q=64 if tune_merge else 5,
                                        M=3, K=4, shapes=shapes)
    inp = dict(W.make_inputs(wl))
    rng = np.random.default_rng(77)
    L = len(shapes)
    wh = np.array([[w, h] for h, w in shapes], dtype=np.float64)               # [L, 2] = (W, H)
    centre = rng.uniform(0.0, 1.0, (wl.B, wl.Qn, wl.M, L, 1, 2))
    loc = centre + rng.normal(0.0, 0.6, (wl.B, wl.Qn, wl.M, L, wl.K, 2)) / wh[None, None, None, :, None, :]
    inp["sampling_locations"] = W.cast(loc, dtype).reshape(loc.shape)
    msda = _msda()
    assert (4.0 * wl.Qn * wl.L * wl.K / wl.S >= 2.0) == tune_merge
    out, gv, gl, ga = _run(wl, inp, accum)
    assert_forward(dtype, f64(out), oracle.forward(inp, dtype), "clustered out")
    rgv, rgl, rga = oracle.backward(inp, dtype)
    assert_grad(dtype, f64(gv), rgv, "clustered grad_value")
    assert_grad(dtype, f64(gl), rgl, "clustered grad_loc")
    assert_grad(dtype, f64(ga), rga, "clustered grad_attn")
    assert msda.device_errors(clear=False) == 0


@pytest.mark.parametrize("dtype,accumulate", [("bf16", False), ("f16", False), ("bf16", True)])
def test_workspace_zeroed_flag(dtype, accumulate):
    """MSDA_BWD_WORKSPACE_ZEROED: a persistent fp32 workspace, cleared once,
    passed to three calls in a row on different inputs.  Each call matches the
    oracle and leaves the workspace holding zeros for the next one."""
    msda = _msda()
    ws = None
    for seed in (41, 42, 43):
        wl = W.WORKLOADS["decoder_bf16"].with_(dtype=dtype, B=2, Q=120, seed=seed)
        inp = W.make_inputs(wl)
        t = to_torch(inp, dtype, DEV)
        dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
        if ws is None:
            ws = torch.zeros(msda.workspace_size(t["value"].dtype, "fp32", dims) // 4, dtype=torch.float32,
                             device=DEV)
            assert ws.numel() * 4 >= wl.B * wl.S * wl.M * wl.D * 4
        start = torch.randn(t["value"].shape, generator=torch.Generator().manual_seed(seed)).to(DEV).to(
            t["value"].dtype) if accumulate else None
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], t["grad_out"], accum="fp32",
                                   grad_value=start.clone() if accumulate else None, accumulate=accumulate,
                                   workspace=ws, workspace_zeroed=True)
        torch.cuda.synchronize()
        rgv, rgl, rga = oracle.backward(inp, dtype)
        want = rgv + (f64(start) if accumulate else 0.0)
        assert_grad(dtype, f64(gv), want, f"zeroed workspace seed {seed} grad_value")
        assert_grad(dtype, f64(gl), rgl, f"zeroed workspace seed {seed} grad_loc")
        assert_grad(dtype, f64(ga), rga, f"zeroed workspace seed {seed} grad_attn")
        assert int(torch.count_nonzero(ws)) == 0, "the workspace must hold zeros after the call"


@pytest.mark.parametrize("zeroed", [False, True])
def test_level_passes_accumulate(zeroed):
    """MSDA_BWD_ACCUMULATE on a problem with one backward pass per level: the
    workspace starts from the widened grad_value (no touch classes then: every
    row goes through the workspace), the passes add to it, the rounding adds
    nothing more.  Against the oracle plus the starting values."""
    msda = _msda()
    shapes = ((256, 256), (128, 128), (64, 64), (32, 32))
    wl = W.WORKLOADS["decoder_bf16"].with_(B=2, Q=15000, shapes=shapes, seed=52)
    inp = W.make_inputs(wl)
    t = to_torch(inp, "bf16", DEV)
    dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
    ws = torch.zeros(msda.workspace_size(torch.bfloat16, "fp32", dims) // 4, dtype=torch.float32, device=DEV)
    start = torch.randn(t["value"].shape, generator=torch.Generator().manual_seed(52)).to(DEV).to(torch.bfloat16)
    gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                               t["attention_weights"], t["grad_out"], accum="fp32", grad_value=start.clone(),
                               accumulate=True, workspace=ws, workspace_zeroed=zeroed)
    torch.cuda.synchronize()
    if zeroed:
        assert int(torch.count_nonzero(ws)) == 0
    rgv, rgl, rga = oracle.backward(inp, "bf16")
    assert_grad("bf16", f64(gv), rgv + f64(start), "grad_value")
    assert_grad("bf16", f64(gl), rgl, "grad_loc")
    assert_grad("bf16", f64(ga), rga, "grad_attn")


@pytest.mark.parametrize("levels_reversed,zeroed,big0", [(False, False, False), (True, False, False),
                                                          (False, True, False), (False, False, True),
                                                          (True, True, True)])
def test_level_passes_round_finished_rows(levels_reversed, zeroed, big0):
    """A problem large enough for one backward pass per level (the fp32
    workspace exceeds the L2, and there are many units): the passes of the
    coarse levels round the workspace rows below the first row of level 2.
    With the levels stored in reverse order in the pyramid that cut is row 0,
    so every row is left to the rounding pass.  Level 0 is sparse (3.7
    corners a row and head; 0.9 with big0, where most of its rows take none
    or one): its rows with one contribution are written directly.  Against
    the oracle, with and without a workspace that holds zeros on entry (and
    must on return)."""
    msda = _msda()
    shapes = ((512 if big0 else 256, 512 if big0 else 256), (128, 128), (64, 64), (32, 32))
    wl = W.WORKLOADS["decoder_bf16"].with_(B=2, Q=15000, shapes=shapes, seed=51)
    assert wl.B * wl.S * wl.M * wl.D * 4 > 160e6 and wl.units * 4 > 8 * 152 * 768
    inp = dict(W.make_inputs(wl))
    if levels_reversed:
        hw = [h * w for h, w in shapes]
        inp["level_start_index"] = np.array([sum(hw[l + 1:]) for l in range(4)], dtype=np.int64)
    t = to_torch(inp, "bf16", DEV)
    dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
    ws = torch.zeros(msda.workspace_size(torch.bfloat16, "fp32", dims) // 4, dtype=torch.float32, device=DEV)
    for _ in range(2):
        gv, gl, ga = msda.backward(t["value"], t["spatial_shapes"], t["level_start_index"], t["sampling_locations"],
                                   t["attention_weights"], t["grad_out"], accum="fp32", workspace=ws,
                                   workspace_zeroed=zeroed)
        torch.cuda.synchronize()
        if zeroed:
            assert int(torch.count_nonzero(ws)) == 0
    rgv, rgl, rga = oracle.backward(inp, "bf16")
    assert_grad("bf16", f64(gv), rgv, "grad_value")
    assert_grad("bf16", f64(gl), rgl, "grad_loc")
    assert_grad("bf16", f64(ga), rga, "grad_attn")
