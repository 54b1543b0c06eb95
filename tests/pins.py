"""Checks that pin the fp64 oracle to facts the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle disagrees.  They
take no arguments and call the ``oracle`` package, so the mutation test can
run them against a copy of the C oracle with a planted mistake.

Facts used (msda-triton README "The operator" and "Kernel design"; course
ch. 4 "Bilinear sampling", "The corner gathers"; course ch. 5 "What the
backward pass must produce"):
  * sampling convention x_im = x*W_l - 0.5 (the grid_sample align_corners=False
    convention), zero padding outside the level;
  * bilinear interpolation reproduces constant and linear fields exactly and
    returns the pixel at its centre;
  * the output is linear in value and in the attention weights, hence the
    adjoint identities <g, out> = <grad_value, value> = <grad_attn, A>;
  * the location gradient is the derivative of the interpolant, checked by
    central finite differences.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _inputs(value, shapes, loc, attn, grad_out=None):
    shapes = np.asarray(shapes, dtype=np.int64).reshape(-1, 2)
    d = {
        "value": np.ascontiguousarray(value, dtype=np.float64),
        "spatial_shapes": shapes,
        "level_start_index": W.level_start_index([tuple(r) for r in shapes]),
        "sampling_locations": np.ascontiguousarray(loc, dtype=np.float64),
        "attention_weights": np.ascontiguousarray(attn, dtype=np.float64),
    }
    if grad_out is not None:
        d["grad_out"] = np.ascontiguousarray(grad_out, dtype=np.float64)
    return d


def _softmax(z):
    e = np.exp(z - z.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def _interior_locs(rng, shapes, B, Q, M, K, margin=0.05):
    """Locations whose four corners are all inside their level: x_im in [0, W-1)."""
    L = len(shapes)
    loc = np.empty((B, Q, M, L, K, 2))
    for l, (h, w) in enumerate(shapes):
        xi = rng.uniform(margin, w - 1 - margin, (B, Q, M, K))
        yi = rng.uniform(margin, h - 1 - margin, (B, Q, M, K))
        loc[:, :, :, l, :, 0] = (xi + 0.5) / w
        loc[:, :, :, l, :, 1] = (yi + 0.5) / h
    return loc


def _rand_problem(rng, B=2, Q=5, M=2, D=3, K=2, shapes=((4, 5), (3, 3), (2, 6)), lo=-0.2, hi=1.2):
    S = sum(h * w for h, w in shapes)
    L = len(shapes)
    value = rng.standard_normal((B, S, M, D))
    loc = rng.uniform(lo, hi, (B, Q, M, L, K, 2))
    attn = rng.uniform(-1, 1, (B, Q, M, L, K))
    g = rng.standard_normal((B, Q, M * D))
    return _inputs(value, shapes, loc, attn, g)


def _away_from_kinks(inp, tol=1e-4):
    """True when no pixel coordinate lies within ``tol`` of an integer."""
    loc = inp["sampling_locations"]
    sh = inp["spatial_shapes"]
    for l in range(sh.shape[0]):
        h, w = sh[l]
        x = loc[:, :, :, l, :, 0] * w - 0.5
        y = loc[:, :, :, l, :, 1] * h - 0.5
        for c in (x, y):
            if np.min(np.abs(c - np.round(c))) < tol:
                return False
    return True


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(np.max(np.abs(b)) if b.size else 0.0, 1e-300)
    assert err <= rtol * scale + atol, f"{what}: max|err| {err:.3e} vs scale {scale:.3e}"


# ---------------------------------------------------------------------------


def pin_hand_worked():
    """A two-level example worked by hand (tests/golden/hand_worked_2level.json)."""
    with open(os.path.join(GOLDEN, "hand_worked_2level.json")) as f:
        gj = json.load(f)
    inp = _inputs(gj["value"], gj["spatial_shapes"], gj["sampling_locations"], gj["attention_weights"],
                  gj["grad_out"])
    assert list(inp["level_start_index"]) == gj["level_start_index"]
    ex = gj["expected"]
    for mode in (0, 1):
        out = oracle.forward(inp, "f64", coord_mode=mode)
        _close(out, np.array(ex["out"]).reshape(out.shape), 1e-14, what="hand-worked out")
        gv, gl, ga = oracle.backward(inp, "f64", coord_mode=mode)
        _close(ga, np.array(ex["grad_attn"]).reshape(ga.shape), 1e-14, what="hand-worked grad_attn")
        _close(gl, np.array(ex["grad_loc"]).reshape(gl.shape), 1e-14, what="hand-worked grad_loc")
        _close(gv, np.array(ex["grad_value"]).reshape(gv.shape), 1e-14, what="hand-worked grad_value")


def pin_constant_field():
    """value == c(b,m,d) everywhere and sum A = 1, all corners inside -> out == c."""
    rng = np.random.default_rng(11)
    shapes = ((5, 7), (3, 4))
    B, Q, M, D, K = 2, 6, 3, 4, 3
    S = sum(h * w for h, w in shapes)
    c = rng.standard_normal((B, 1, M, D))
    value = np.broadcast_to(c, (B, S, M, D)).copy()
    loc = _interior_locs(rng, shapes, B, Q, M, K)
    attn = _softmax(rng.standard_normal((B, Q, M, len(shapes) * K))).reshape(B, Q, M, len(shapes), K)
    out = oracle.forward(_inputs(value, shapes, loc, attn), "f64", coord_mode=0).reshape(B, Q, M, D)
    _close(out, np.broadcast_to(c, (B, Q, M, D)), 1e-13, what="constant field")


def pin_linear_field():
    """value = alpha*x_pix + beta*y_pix + gamma is reproduced exactly by bilinear
    interpolation; its x / y slopes give grad_loc = (A*W*<g,alpha>, A*H*<g,beta>)."""
    rng = np.random.default_rng(12)
    shapes = ((6, 9), (4, 3))
    B, Q, M, D, K = 2, 5, 2, 3, 2
    L = len(shapes)
    S = sum(h * w for h, w in shapes)
    alpha = rng.standard_normal((L, B, M, D))
    beta = rng.standard_normal((L, B, M, D))
    gamma = rng.standard_normal((L, B, M, D))
    value = np.zeros((B, S, M, D))
    st = 0
    for l, (h, w) in enumerate(shapes):
        ii, jj = np.meshgrid(np.arange(h), np.arange(w), indexing="ij")
        px = jj.ravel()[None, :, None, None]
        py = ii.ravel()[None, :, None, None]
        value[:, st:st + h * w] = (alpha[l][:, None] * px + beta[l][:, None] * py + gamma[l][:, None])
        st += h * w
    loc = _interior_locs(rng, shapes, B, Q, M, K)
    attn = rng.uniform(-1, 1, (B, Q, M, L, K))
    g = rng.standard_normal((B, Q, M, D))
    inp = _inputs(value, shapes, loc, attn, g.reshape(B, Q, M * D))
    out = oracle.forward(inp, "f64", coord_mode=0).reshape(B, Q, M, D)
    exp = np.zeros((B, Q, M, D))
    egl = np.zeros((B, Q, M, L, K, 2))
    ega = np.zeros((B, Q, M, L, K))
    for l, (h, w) in enumerate(shapes):
        x = loc[:, :, :, l, :, 0] * w - 0.5               # [B,Q,M,K]
        y = loc[:, :, :, l, :, 1] * h - 0.5
        a = attn[:, :, :, l, :]
        al = alpha[l][:, None, :, None, :]                # [B,1,M,1,D]
        be = beta[l][:, None, :, None, :]
        ga_ = gamma[l][:, None, :, None, :]
        samp = al * x[..., None] + be * y[..., None] + ga_  # [B,Q,M,K,D]
        exp += (a[..., None] * samp).sum(3)
        ega[:, :, :, l, :] = (g[:, :, :, None, :] * samp).sum(-1)
        egl[:, :, :, l, :, 0] = a * w * (g[:, :, :, None, :] * al).sum(-1)
        egl[:, :, :, l, :, 1] = a * h * (g[:, :, :, None, :] * be).sum(-1)
    _close(out, exp, 1e-12, what="linear field out")
    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    _close(gl, egl, 1e-11, what="linear field grad_loc")
    _close(ga, ega, 1e-12, what="linear field grad_attn")


def pin_pixel_centres():
    """loc at pixel centres ((j+0.5)/W, (i+0.5)/H): lx = ly = 0, out = sum A*value[pixel]."""
    rng = np.random.default_rng(13)
    shapes = ((4, 6), (3, 5), (2, 2))
    B, Q, M, D, K = 2, 4, 2, 5, 3
    L = len(shapes)
    S = sum(h * w for h, w in shapes)
    starts = W.level_start_index(shapes)
    value = rng.standard_normal((B, S, M, D))
    loc = np.empty((B, Q, M, L, K, 2))
    pix = np.empty((B, Q, M, L, K), dtype=np.int64)
    for l, (h, w) in enumerate(shapes):
        i = rng.integers(0, h, (B, Q, M, K))
        j = rng.integers(0, w, (B, Q, M, K))
        loc[:, :, :, l, :, 0] = (j + 0.5) / w
        loc[:, :, :, l, :, 1] = (i + 0.5) / h
        pix[:, :, :, l, :] = starts[l] + i * w + j
    attn = rng.uniform(-1, 1, (B, Q, M, L, K))
    out = oracle.forward(_inputs(value, shapes, loc, attn), "f64", coord_mode=0).reshape(B, Q, M, D)
    exp = np.zeros((B, Q, M, D))
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                for l in range(L):
                    for k in range(K):
                        exp[b, q, m] += attn[b, q, m, l, k] * value[b, pix[b, q, m, l, k], m]
    _close(out, exp, 1e-13, what="pixel centres")


def pin_zero_padding():
    """Corners outside the level contribute nothing; a sample with no corner
    inside yields zero output and zero gradients; half-outside samples get
    exactly half the edge pixel."""
    rng = np.random.default_rng(14)
    shapes = ((4, 5),)
    B, Q, M, D, K = 1, 6, 1, 3, 1
    S = 20
    value = rng.standard_normal((B, S, M, D))
    v = value[0, :, 0].reshape(4, 5, D)
    i = 2
    cy = (i + 0.5) / 4
    locs = [
        (-1.0, 0.5),        # far left
        (2.0, 0.5),         # far right
        (0.5, -0.6),        # far above: y_im = -2.9, both rows outside
        (0.0, cy),          # x_im = -0.5 on pixel row i: 0.5 * v[i, 0]
        (1.0, cy),          # x_im = W - 0.5 on row i: 0.5 * v[i, W-1]
        ((3 + 0.5) / 5, 1.0),  # y_im = H - 0.5 on column 3: 0.5 * v[H-1, 3]
    ]
    loc = np.array(locs).reshape(B, Q, M, 1, K, 2)
    attn = np.ones((B, Q, M, 1, K))
    g = rng.standard_normal((B, Q, M * D))
    inp = _inputs(value, shapes, loc, attn, g)
    out = oracle.forward(inp, "f64", coord_mode=0).reshape(Q, D)
    exp = np.zeros((Q, D))
    exp[3] = 0.5 * v[i, 0]
    exp[4] = 0.5 * v[i, 4]
    exp[5] = 0.5 * v[3, 3]
    _close(out, exp, 1e-15, atol=0.0, what="zero padding out")
    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    assert np.all(gl[0, :3] == 0.0) and np.all(ga[0, :3] == 0.0), "fully outside samples must get zero gradient"
    # the edge samples: grad_attn = <g, 0.5 v>, and only the inside pixel receives 0.5*g
    gq = g.reshape(Q, D)
    _close(ga[0, 3:, 0, 0, 0], np.array([gq[3] @ exp[3], gq[4] @ exp[4], gq[5] @ exp[5]]), 1e-14,
           what="edge grad_attn")
    ev = np.zeros((4, 5, D))
    ev[i, 0] += 0.5 * gq[3]
    ev[i, 4] += 0.5 * gq[4]
    ev[3, 3] += 0.5 * gq[5]
    _close(gv[0, :, 0].reshape(4, 5, D), ev, 1e-15, what="edge grad_value")


def pin_thin_levels():
    """Levels one pixel high or wide (msda-triton README "The operator": the
    corners of x*W - 0.5 with zero padding).  On a 1x1 level bilinear
    sampling with zero padding is the tent (1 - |x_im|)(1 - |y_im|) times the
    pixel, so grad_attn = tent * <g, v>, grad_value = A * tent * g and the
    location gradient is A * <g, v> times -sign(x_im) * W (y: -sign(y_im) * H)
    times the other axis' tent.  On a level one pixel high the x axis is
    piecewise-linear interpolation of the row padded with zeros (np.interp)
    times the y tent.  Samples keep clear of the kinks (x_im, y_im in
    {-1, 0, 1} and the integers of the row)."""
    rng = np.random.default_rng(21)
    Q, D = 40, 3
    g = rng.standard_normal((1, Q, D))
    a = rng.uniform(-1, 1, (1, Q, 1, 1, 1))

    def away(n):   # locations in [-0.3, 1.3] at least 0.02 from the kinks of a level n pixels across
        u = rng.uniform(-0.3, 1.3, 4 * Q)
        t = u * n - 0.5
        keep = np.abs(t - np.round(t)) > 0.02
        return u[keep][:Q]

    # 1x1: the tent on both axes
    v = rng.standard_normal((1, 1, 1, D))
    loc = np.stack([away(1), away(1)], -1).reshape(1, Q, 1, 1, 1, 2)
    inp = _inputs(v, ((1, 1),), loc, a, g)
    xi, yi = loc[0, :, 0, 0, 0, 0] - 0.5, loc[0, :, 0, 0, 0, 1] - 0.5
    tx, ty = np.maximum(0.0, 1 - np.abs(xi)), np.maximum(0.0, 1 - np.abs(yi))
    A = a.reshape(Q)
    out = oracle.forward(inp, "f64", coord_mode=0).reshape(Q, D)
    _close(out, (A * tx * ty)[:, None] * v.reshape(1, D), 1e-14, what="1x1 level out")
    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    gvv = g.reshape(Q, D) @ v.reshape(D)
    _close(ga.reshape(Q), tx * ty * gvv, 1e-14, what="1x1 level grad_attn")
    _close(gv.reshape(D), ((A * tx * ty)[:, None] * g.reshape(Q, D)).sum(0), 1e-14, what="1x1 level grad_value")
    sx = np.where(np.abs(xi) < 1, -np.sign(xi), 0.0)
    sy = np.where(np.abs(yi) < 1, -np.sign(yi), 0.0)
    _close(gl.reshape(Q, 2), np.stack([A * gvv * sx * ty, A * gvv * sy * tx], -1), 1e-14,
           what="1x1 level grad_loc")

    # one pixel high, five wide: np.interp along x, the tent along y
    Wd = 5
    v = rng.standard_normal((1, Wd, 1, D))
    loc = np.stack([away(Wd), away(1)], -1).reshape(1, Q, 1, 1, 1, 2)
    inp = _inputs(v, ((1, Wd),), loc, a)
    xi, yi = loc[0, :, 0, 0, 0, 0] * Wd - 0.5, loc[0, :, 0, 0, 0, 1] - 0.5
    ty = np.maximum(0.0, 1 - np.abs(yi))
    xs = np.arange(-1, Wd + 1)
    row = np.zeros((Wd + 2, D))
    row[1:-1] = v.reshape(Wd, D)
    exp = np.stack([np.interp(xi, xs, row[:, d]) for d in range(D)], -1) * (A * ty)[:, None]
    out = oracle.forward(inp, "f64", coord_mode=0).reshape(Q, D)
    _close(out, exp, 1e-14, what="one-pixel-high level out")

    # one pixel wide, four high: the same with the axes exchanged; the location
    # gradient from the interpolant's slope (a central difference of np.interp
    # inside one linear piece is exact) and the x tent's
    Hd = 4
    v = rng.standard_normal((1, Hd, 1, D))
    loc = np.stack([away(1), away(Hd)], -1).reshape(1, Q, 1, 1, 1, 2)
    inp = _inputs(v, ((Hd, 1),), loc, a, g)
    xi, yi = loc[0, :, 0, 0, 0, 0] - 0.5, loc[0, :, 0, 0, 0, 1] * Hd - 0.5
    tx = np.maximum(0.0, 1 - np.abs(xi))
    ys = np.arange(-1, Hd + 1)
    col = np.zeros((Hd + 2, D))
    col[1:-1] = v.reshape(Hd, D)
    iy = np.stack([np.interp(yi, ys, col[:, d]) for d in range(D)], -1)
    exp = iy * (A * tx)[:, None]
    out = oracle.forward(inp, "f64", coord_mode=0).reshape(Q, D)
    _close(out, exp, 1e-14, what="one-pixel-wide level out")
    h = 0.01
    slope = np.stack([(np.interp(yi + h, ys, col[:, d]) - np.interp(yi - h, ys, col[:, d])) / (2 * h)
                      for d in range(D)], -1)
    gq = g.reshape(Q, D)
    sx = np.where(np.abs(xi) < 1, -np.sign(xi), 0.0)
    egl = np.stack([A * 1 * sx * (gq * iy).sum(-1), A * Hd * tx * (gq * slope).sum(-1)], -1)
    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    _close(gl.reshape(Q, 2), egl, 1e-12, what="one-pixel-wide level grad_loc")


def pin_convexity():
    """sum A = 1, A >= 0, corners inside: each output channel lies within the
    range of the corner values the unit read."""
    rng = np.random.default_rng(15)
    shapes = ((7, 9), (4, 5))
    B, Q, M, D, K = 2, 8, 2, 4, 3
    L = len(shapes)
    S = sum(h * w for h, w in shapes)
    starts = W.level_start_index(shapes)
    value = rng.standard_normal((B, S, M, D))
    loc = _interior_locs(rng, shapes, B, Q, M, K)
    attn = _softmax(rng.standard_normal((B, Q, M, L * K))).reshape(B, Q, M, L, K)
    out = oracle.forward(_inputs(value, shapes, loc, attn), "f64", coord_mode=0).reshape(B, Q, M, D)
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                rows = []
                for l, (h, w) in enumerate(shapes):
                    for k in range(K):
                        x0 = int(np.floor(loc[b, q, m, l, k, 0] * w - 0.5))
                        y0 = int(np.floor(loc[b, q, m, l, k, 1] * h - 0.5))
                        for yy in (y0, y0 + 1):
                            for xx in (x0, x0 + 1):
                                rows.append(value[b, starts[l] + yy * w + xx, m])
                rows = np.array(rows)
                lo, hi = rows.min(0), rows.max(0)
                assert np.all(out[b, q, m] >= lo - 1e-12) and np.all(out[b, q, m] <= hi + 1e-12), "convexity"


def pin_gridsample():
    """Forward and all three gradients equal the torch grid_sample restatement (fp64)."""
    import torch

    rng = np.random.default_rng(16)
    for trial in range(4):
        inp = _rand_problem(rng)
        if not _away_from_kinks(inp):
            continue
        t = {k: torch.tensor(v) for k, v in inp.items()}
        for k in ("value", "sampling_locations", "attention_weights"):
            t[k].requires_grad_(True)
        ref = oracle.gridsample_forward(t["value"], inp["spatial_shapes"], inp["level_start_index"],
                                        t["sampling_locations"], t["attention_weights"])
        (ref * t["grad_out"]).sum().backward()
        out = oracle.forward(inp, "f64", coord_mode=0)
        _close(out, ref.detach().numpy(), 1e-12, what="grid_sample out")
        gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
        _close(gv, t["value"].grad.numpy(), 1e-12, what="grid_sample grad_value")
        _close(gl, t["sampling_locations"].grad.numpy(), 1e-11, what="grid_sample grad_loc")
        _close(ga, t["attention_weights"].grad.numpy(), 1e-12, what="grid_sample grad_attn")


def pin_brute_force():
    """The C oracle equals the pure-Python loop on the tiny workload, in both coordinate modes."""
    inp = W.make_inputs(W.WORKLOADS["tiny_fp32"])
    for mode in (0, 1):
        out = oracle.forward(inp, "f32", coord_mode=mode)
        _close(out, oracle.naive_forward(inp, "f32", coord_mode=mode), 1e-13, what=f"brute force out mode {mode}")
        gv, gl, ga = oracle.backward(inp, "f32", coord_mode=mode)
        ngv, ngl, nga = oracle.naive_backward(inp, "f32", coord_mode=mode)
        _close(gv, ngv, 1e-13, what="brute force grad_value")
        _close(gl, ngl, 1e-13, what="brute force grad_loc")
        _close(ga, nga, 1e-13, what="brute force grad_attn")


def pin_finite_differences():
    """Central differences (fp64, h = 1e-6, away from kinks) of <g, out> match
    all three analytic gradients."""
    rng = np.random.default_rng(17)
    for trial in range(20):
        inp = _rand_problem(rng, B=1, Q=3, M=2, D=3, K=2, shapes=((4, 5), (3, 3)))
        if _away_from_kinks(inp, tol=1e-3):
            break
    else:
        raise AssertionError("could not draw a kink-free problem")
    g = inp["grad_out"]

    def loss(d):
        return float(np.sum(oracle.forward(d, "f64", coord_mode=0) * g))

    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    h = 1e-6
    for key, grad in (("sampling_locations", gl), ("attention_weights", ga), ("value", gv)):
        base = inp[key]
        flat = base.reshape(-1)
        idx = np.arange(flat.size) if flat.size <= 200 else rng.choice(flat.size, 200, replace=False)
        fd = np.empty(idx.size)
        for n, i in enumerate(idx):
            plus = dict(inp)
            minus = dict(inp)
            p = flat.copy()
            p[i] += h
            plus[key] = p.reshape(base.shape)
            mm = flat.copy()
            mm[i] -= h
            minus[key] = mm.reshape(base.shape)
            fd[n] = (loss(plus) - loss(minus)) / (2 * h)
        _close(grad.reshape(-1)[idx], fd, 1e-6, atol=1e-8, what=f"finite differences {key}")


def pin_adjoint():
    """<g, out> = <grad_value, value> = <grad_attn, A> (out is linear in value and in A)."""
    rng = np.random.default_rng(18)
    inp = _rand_problem(rng, B=2, Q=9, M=3, D=4, K=3)
    out = oracle.forward(inp, "f64", coord_mode=0)
    gv, gl, ga = oracle.backward(inp, "f64", coord_mode=0)
    lhs = float(np.sum(inp["grad_out"] * out))
    r1 = float(np.sum(gv * inp["value"]))
    r2 = float(np.sum(ga * inp["attention_weights"]))
    assert abs(lhs - r1) <= 1e-12 * max(1.0, abs(lhs)), f"adjoint value {lhs} vs {r1}"
    assert abs(lhs - r2) <= 1e-12 * max(1.0, abs(lhs)), f"adjoint attn {lhs} vs {r2}"


def pin_scatter_total():
    """With every corner inside, the weights of a sample sum to 1, so for each
    (b, m, d): sum over pixels of grad_value = sum over (q, l, k) of A * g."""
    rng = np.random.default_rng(19)
    shapes = ((6, 5), (3, 7))
    B, Q, M, D, K = 2, 7, 3, 2, 2
    L = len(shapes)
    S = sum(h * w for h, w in shapes)
    value = rng.standard_normal((B, S, M, D))
    loc = _interior_locs(rng, shapes, B, Q, M, K)
    attn = rng.uniform(-1, 1, (B, Q, M, L, K))
    g = rng.standard_normal((B, Q, M, D))
    gv, _, _ = oracle.backward(_inputs(value, shapes, loc, attn, g.reshape(B, Q, M * D)), "f64", coord_mode=0)
    tot = gv.sum(1)                                    # [B, M, D]
    exp = np.einsum("bqmlk,bqmd->bmd", attn, g)
    _close(tot, exp, 1e-12, what="scatter total")


def pin_fp32_coordinate():
    """coord_mode 1 takes the cell from the binary32 pixel coordinate.  A fp32
    location whose exact x*W - 0.5 lies just below an integer n, but rounds to
    n in binary32, must use the cell [n, n+1]; on a quadratic field the two
    cells' slopes differ, which fixes grad_loc."""
    Wd = 1000
    # every binary32 x in [0.5, 0.6): find one whose exact x*W - 0.5 (exact in
    # fp64: 24 + 10 significant bits) floors differently from its binary32 rounding
    lo = np.array([0.5], dtype=np.float32).view(np.uint32)[0]
    hi = np.array([0.6], dtype=np.float32).view(np.uint32)[0]
    xs = np.arange(lo, hi, dtype=np.uint32).view(np.float32)
    exact = xs.astype(np.float64) * Wd - 0.5
    r32 = exact.astype(np.float32).astype(np.float64)
    hit = np.nonzero(np.floor(exact) != np.floor(r32))[0]
    assert hit.size > 0, "no rounding-crossing location found"
    found = (xs[hit[0]], exact[hit[0]], r32[hit[0]])
    x, exact, r32 = found
    n = int(np.floor(r32))
    shapes = ((1, Wd),)
    value = (np.arange(Wd, dtype=np.float64) ** 2).reshape(1, Wd, 1, 1)
    loc = np.array([float(x), 0.5]).reshape(1, 1, 1, 1, 1, 2)
    attn = np.ones((1, 1, 1, 1, 1))
    g = np.ones((1, 1, 1))
    inp = _inputs(value, shapes, loc, attn, g)
    _, gl1, _ = oracle.backward(inp, "f64", coord_mode=1)
    _, gl0, _ = oracle.backward(inp, "f64", coord_mode=0)
    # cell [n, n+1]: slope (n+1)^2 - n^2 = 2n + 1;  cell [n-1, n]: 2n - 1
    assert gl1[0, 0, 0, 0, 0, 0] == Wd * (2 * n + 1), f"fp32 cell: {gl1.ravel()}"
    assert gl0[0, 0, 0, 0, 0, 0] == Wd * (2 * n - 1), f"fp64 cell: {gl0.ravel()}"


def pin_coordinate_modes_agree():
    """For bf16 / f16 inputs the pixel coordinate is exact in binary32, so both
    modes agree bit for bit; for fp32 inputs the forward agrees to 1e-6."""
    for name in ("tiny_fp32",):
        base = W.WORKLOADS[name]
        for dt in ("bf16", "f16"):
            wl = base.with_(dtype=dt)
            inp = W.make_inputs(wl)
            a = oracle.forward(inp, dt, coord_mode=0)
            b = oracle.forward(inp, dt, coord_mode=1)
            assert np.array_equal(a, b), f"{dt}: modes differ"
        inp = W.make_inputs(base)
        _close(oracle.forward(inp, "f32", coord_mode=1), oracle.forward(inp, "f32", coord_mode=0), 1e-6,
               what="fp32 coordinate modes")


def pin_samplers():
    """The sampled entry points equal the matching slices of the full results."""
    wl = W.scaled("decoder_bf16", B=2, Q=13, M=3, shapes=((9, 11), (5, 6)))
    inp = W.make_inputs(wl)
    out = oracle.forward(inp, "bf16").reshape(-1, wl.D)
    gv, gl, ga = oracle.backward(inp, "bf16")
    rng = np.random.default_rng(20)
    units = rng.choice(wl.units, 17, replace=False)
    assert np.array_equal(oracle.forward_units(inp, "bf16", units), out[units])
    sgl, sga = oracle.backward_units(inp, "bf16", units)
    assert np.array_equal(sgl, gl.reshape(wl.units, -1)[units])
    assert np.array_equal(sga, ga.reshape(wl.units, -1)[units])
    rows = rng.choice(wl.B * wl.S * wl.M, 40, replace=False)
    rows = np.concatenate([rows, rows[:3]])
    _close(oracle.grad_value_rows(inp, "bf16", rows), gv.reshape(-1, wl.D)[rows], 1e-13, what="grad_value rows")


def _fused_problem(rng, B=2, Q=4, M=2, D=3, K=2, shapes=((4, 6), (3, 5)), spread=2.0):
    L = len(shapes)
    S = sum(h * w for h, w in shapes)
    sh = np.asarray(shapes, dtype=np.int64)
    return {
        "value": rng.standard_normal((B, S, M, D)),
        "spatial_shapes": sh,
        "level_start_index": W.level_start_index(shapes),
        "reference_points": rng.uniform(0.1, 0.9, (B, Q, L, 2)),
        "sampling_offsets": rng.normal(0.0, spread, (B, Q, M, L, K, 2)),
        "attention_logits": rng.standard_normal((B, Q, M, L * K)),
        "grad_out": rng.standard_normal((B, Q, M * D)),
    }


def pin_fused_special_cases():
    """Zero offsets and equal logits: the fused operator is the core with
    loc = reference point and A = 1/(L*K).  Offsets of (dx*W, dy*H) pixels move
    the sample by exactly (dx, dy) in normalised coordinates (x by W, y by H;
    the levels have W != H).  A constant added to a row of logits changes
    nothing."""
    rng = np.random.default_rng(31)
    f = _fused_problem(rng)
    B, Q, M, L, K = 2, 4, 2, 2, 2
    f0 = dict(f, sampling_offsets=np.zeros((B, Q, M, L, K, 2)), attention_logits=np.full((B, Q, M, L * K), 0.7))
    core = _inputs(f["value"], f["spatial_shapes"],
                   np.broadcast_to(f["reference_points"][:, :, None, :, None, :], (B, Q, M, L, K, 2)),
                   np.full((B, Q, M, L, K), 1.0 / (L * K)))
    _close(oracle.fused_forward(f0, "f64", coord_mode=0), oracle.forward(core, "f64", coord_mode=0), 1e-13,
           what="fused with zero offsets")
    d = rng.uniform(-0.05, 0.05, (B, Q, M, L, K, 2))
    wh = np.stack([f["spatial_shapes"][:, 1], f["spatial_shapes"][:, 0]], axis=-1).astype(np.float64)
    f1 = dict(f0, sampling_offsets=d * wh[None, None, None, :, None, :])
    core1 = dict(core, sampling_locations=f["reference_points"][:, :, None, :, None, :] + d)
    _close(oracle.fused_forward(f1, "f64", coord_mode=0), oracle.forward(core1, "f64", coord_mode=0), 1e-12,
           what="fused offsets normalised by (W, H)")
    shift = rng.uniform(-3, 3, (B, Q, M, 1))
    _close(oracle.fused_forward(dict(f, attention_logits=f["attention_logits"] + shift), "f64", coord_mode=0),
           oracle.fused_forward(f, "f64", coord_mode=0), 1e-12, what="softmax shift invariance")
    _, _, _, gz = oracle.fused_backward(f, "f64", coord_mode=0)
    assert np.max(np.abs(gz.sum(-1))) < 1e-12, "logit gradients of a row must sum to zero"


def pin_fused_torch_restatement():
    """The fused operator and its three input gradients equal torch softmax +
    grid_sample with autograd (fp64, CPU)."""
    import torch

    rng = np.random.default_rng(32)
    for _ in range(4):
        f = _fused_problem(rng)
        core, _, _ = oracle.fused_core_inputs(f, "f64", coord_mode=0)
        if _away_from_kinks(core):
            break
    t = {k: torch.tensor(v) for k, v in f.items()}
    for k in ("reference_points", "sampling_offsets", "attention_logits"):
        t[k].requires_grad_(True)
    B, Q, M, L, K = 2, 4, 2, 2, 2
    wh = torch.stack([t["spatial_shapes"][:, 1], t["spatial_shapes"][:, 0]], dim=-1).double()
    loc = t["reference_points"][:, :, None, :, None, :] + t["sampling_offsets"] / wh[None, None, None, :, None, :]
    A = torch.softmax(t["attention_logits"], dim=-1).view(B, Q, M, L, K)
    ref_out = oracle.gridsample_forward(t["value"], f["spatial_shapes"], f["level_start_index"], loc, A)
    (ref_out * t["grad_out"]).sum().backward()
    _close(oracle.fused_forward(f, "f64", coord_mode=0), ref_out.detach().numpy(), 1e-12, what="fused out")
    gv, gr, go, gz = oracle.fused_backward(f, "f64", coord_mode=0)
    _close(gr, t["reference_points"].grad.numpy(), 1e-11, what="fused grad_reference_points")
    _close(go, t["sampling_offsets"].grad.numpy(), 1e-11, what="fused grad_sampling_offsets")
    _close(gz, t["attention_logits"].grad.numpy(), 1e-11, what="fused grad_attention_logits")


def pin_fused_finite_differences():
    """Central differences of <g, out> in fp64 against the fused gradients."""
    rng = np.random.default_rng(33)
    for _ in range(20):
        f = _fused_problem(rng, B=1, Q=2, M=2, D=2, K=2)
        core, _, _ = oracle.fused_core_inputs(f, "f64", coord_mode=0)
        if _away_from_kinks(core, tol=1e-3):
            break
    else:
        raise AssertionError("could not draw a kink-free problem")
    g = f["grad_out"]
    _, gr, go, gz = oracle.fused_backward(f, "f64", coord_mode=0)
    h = 1e-6
    for key, grad in (("reference_points", gr), ("sampling_offsets", go), ("attention_logits", gz)):
        base = f[key].reshape(-1)
        fd = np.empty(base.size)
        for i in range(base.size):
            p, m = base.copy(), base.copy()
            p[i] += h
            m[i] -= h
            lp = float(np.sum(oracle.fused_forward(dict(f, **{key: p.reshape(f[key].shape)}), "f64", coord_mode=0) * g))
            lm = float(np.sum(oracle.fused_forward(dict(f, **{key: m.reshape(f[key].shape)}), "f64", coord_mode=0) * g))
            fd[i] = (lp - lm) / (2 * h)
        _close(grad.reshape(-1), fd, 1e-6, atol=1e-8, what=f"fused finite differences {key}")


def pin_fused_coordinate_modes_agree():
    """The fused locations in binary32 (coord_mode 1, the kernels' arithmetic)
    agree with the fp64 ones (coord_mode 0) to binary32 rounding: a location
    moves by at most a few units of 2^-24, i.e. a few 1e-5 pixels on a level
    167 pixels wide, so the fused forward of a tiny and of a decoder-shaped
    problem (levels with W != H) match to 2e-5 relative L2.  Dividing by
    (H, W), or summing before dividing, moves samples by whole pixels and
    fails this."""
    rng = np.random.default_rng(34)
    cases = [_fused_problem(rng),
             _fused_problem(rng, B=1, Q=24, M=4, D=4, K=4, shapes=((100, 167), (50, 84), (25, 42), (13, 21)),
                            spread=3.0)]
    for f in cases:
        f = {k: (v.astype(np.float32).astype(np.float64) if v.dtype == np.float64 else v) for k, v in f.items()}
        a = oracle.fused_forward(f, "f64", coord_mode=1)
        b = oracle.fused_forward(f, "f64", coord_mode=0)
        err = float(np.linalg.norm(a - b) / np.linalg.norm(b))
        assert err <= 2e-5, f"fused coordinate modes differ: rel-L2 {err:.3e}"
        la = oracle.fused_locations(f["reference_points"], f["sampling_offsets"], f["spatial_shapes"], 1)
        lb = oracle.fused_locations(f["reference_points"], f["sampling_offsets"], f["spatial_shapes"], 0)
        assert np.max(np.abs(la - lb)) <= 2.0 ** -20, "binary32 fused locations far from the fp64 ones"


def pin_fused_fp32_location():
    """coord_mode 1 forms loc = ref + off / W with two binary32 roundings (the
    quotient, then the sum).  For ref = 0.70616740 and off = -0.61850226 on a
    level three pixels wide (both binary32 values), the quotient rounds to the
    nearest binary32 and the sum then rounds to exactly 0.5, the centre of
    pixel 1, so the fused output is A * value[pixel 1] = 20 exactly.  The exact
    fp64 location, and a single rounding of it, are both just below 0.5 and
    pick the cell [0, 1].  The same values on the y axis of a level three
    pixels high fix the division by H."""
    r = float(np.float32(0.7061673998832703))
    o = float(np.float32(-0.6185022592544556))
    value = np.array([10.0, 20.0, 40.0]).reshape(1, 3, 1, 1)
    for axis, shapes in ((0, ((1, 3),)), (1, ((3, 1),))):
        ref = np.full((1, 1, 1, 2), 0.5)
        off = np.zeros((1, 1, 1, 1, 1, 2))
        ref[..., axis] = r
        off[..., axis] = o
        f = {"value": value, "spatial_shapes": np.asarray(shapes, dtype=np.int64),
             "level_start_index": np.zeros(1, dtype=np.int64), "reference_points": ref, "sampling_offsets": off,
             "attention_logits": np.zeros((1, 1, 1, 1)), "grad_out": np.ones((1, 1, 1))}
        loc = oracle.fused_locations(ref, off, f["spatial_shapes"], 1)
        assert loc[0, 0, 0, 0, 0, axis] == 0.5, f"binary32 fused location {loc.ravel()}"
        out1 = oracle.fused_forward(f, "f64", coord_mode=1)
        assert out1.ravel()[0] == 20.0, f"axis {axis}: fused binary32 output {out1.ravel()}"
        out0 = oracle.fused_forward(f, "f64", coord_mode=0)
        assert 19.99 < out0.ravel()[0] < 20.0, f"axis {axis}: fused fp64 output {out0.ravel()}"


ALL_PINS = [
    pin_hand_worked, pin_constant_field, pin_linear_field, pin_pixel_centres, pin_zero_padding,
    pin_thin_levels, pin_convexity, pin_gridsample, pin_brute_force, pin_finite_differences, pin_adjoint,
    pin_scatter_total, pin_fp32_coordinate, pin_coordinate_modes_agree, pin_samplers,
    pin_fused_special_cases, pin_fused_torch_restatement, pin_fused_finite_differences,
    pin_fused_coordinate_modes_agree, pin_fused_fp32_location,
]
