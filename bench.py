"""Benchmark of the MSDA sampling core (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload stress_bf16] [--accum fp32|native|auto|deterministic]
                    [--all] [--fused] [--no-configs]

One step = one pass of the whole hot path over one batch: forward
(msda_forward), then backward (msda_backward: zero or widen of the grad_value
accumulator, gather + scatter kernel, and for the fp32 accumulator the
rounding pass).  Inputs are resident in HBM; the L2 is flushed (a read of a
512 MB buffer) between steps, outside the timed events.  The metric is (b, q, m)
output vectors per second over the timed steps (higher is better).

The contract line runs the largest single-GPU workload, stress_bf16 (B=8,
Q=20000, a 768x1024 pyramid of 4 levels, M=8, D=32, L=K=4, bf16) with the
FP32 grad_value accumulator it asks for.  Its K timed steps run untraced;
per-kernel durations (`kernels`, `roofline`) come from a separate traced pass
after them.  `all_configs` holds the other named workloads, each timed on its
own inputs, and `dispatch` the host time per call of the autograd operator.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(weak scaling, no data-path collective: the path shards over batches); the
step time is the max over ranks and the value is the units of all ranks over
that time.

--impl reference times the fp64 CPU oracle (test infrastructure) on the host
cores on a bounded sample of the same workload.
--all prints one extra JSON line per named workload with every accumulator
(not the contract line); --fused the fused operator against PyTorch ops
around the core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MSDA fwd+bwd ms and (b,q,m) outputs/s; achieved HBM GB/s vs GB300 peak"
UNIT = "(b,q,m) outputs/s"
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# byte models (algorithmic bytes per launch): per-corner (every in-level
# corner row counted each time) and unique (each distinct value row once)

_corner_memo = {}


def corner_counts(wl: W.Workload, inp, unique: bool = True):
    """(in-bounds (sample, corner) pairs, distinct value rows they touch), on
    the binary32 pixel coordinate the kernels use.  A value row is one
    (b, pixel, m): D contiguous channels.  Remembered per workload and input
    set within the run."""
    key = (wl, id(inp["sampling_locations"]), unique)
    if key not in _corner_memo:
        _corner_memo.clear()
        _corner_memo[key] = _corner_counts(wl, inp, unique)
    return _corner_memo[key]


def _corner_counts(wl: W.Workload, inp, unique: bool):
    loc = W.to_f64(inp["sampling_locations"], wl.dtype)         # [B,Q,M,L,K,2]
    B, Q, M = loc.shape[:3]
    starts = W.level_start_index(wl.shapes)
    b_idx = np.arange(B, dtype=np.int64)[:, None, None, None]
    m_idx = np.arange(M, dtype=np.int64)[None, None, :, None]
    n = 0
    rows = []
    for l, (h, w) in enumerate(wl.shapes):
        # exact in fp64 for binary32 inputs and sides <= 8192, then one rounding
        x = np.floor((loc[:, :, :, l, :, 0] * w - 0.5).astype(np.float32)).astype(np.int64)
        y = np.floor((loc[:, :, :, l, :, 1] * h - 0.5).astype(np.float32)).astype(np.int64)
        for dy in (0, 1):
            for dx in (0, 1):
                xx, yy = x + dx, y + dy
                ok = (xx >= 0) & (xx < w) & (yy >= 0) & (yy < h)
                n += int(np.count_nonzero(ok))
                if unique:
                    r = ((b_idx * wl.S + starts[l] + yy * w + xx) * M + m_idx)
                    rows.append(np.unique(r[ok]))
    u = int(np.unique(np.concatenate(rows)).size) if unique and rows else None
    return n, u


def inbounds_corners(wl: W.Workload, inp) -> int:
    return corner_counts(wl, inp, unique=False)[0]


def byte_model(wl: W.Workload, corners: int, unique_rows=None) -> dict:
    """Algorithmic bytes per launch.  Per-corner model: every in-bounds corner
    row counted each time it is read (and, in the backward, written by a
    reduction).  Unique (compulsory) model: each distinct value row once."""
    es = W.ESIZE[wl.dtype]
    n_value = wl.B * wl.S * wl.M * wl.D
    loc = wl.samples * 2 * es
    attn = wl.samples * es
    rowio = wl.units * wl.D * es            # out, or grad_out
    gather = corners * wl.D * es
    fwd = gather + loc + attn + rowio
    # backward kernel: corner reads + atomic payload at the value dtype, grad_out, params, param grads
    bwd_kernel = 2 * gather + rowio + 2 * (loc + attn)
    bwd = bwd_kernel + n_value * es          # + one full grad_value write
    out = {"forward": fwd, "backward": bwd_kernel, "bwd_total": bwd, "zero": n_value * es,
           "convert": n_value * (4 + es), "step": fwd + bwd,
           # the FP32 accumulator on chip splits the backward kernel: the gather
           # kernel (corner reads, grad_out, params, param grads) and the
           # accumulate pass (the per-corner payload, summed in shared memory,
           # and one full grad_value write); count and place read the locations
           # (place writes a 4-byte entry per point and tile, about one)
           "backward_gather": gather + rowio + 2 * (loc + attn),
           "tile_accum": gather + n_value * es,
           "tile_count": loc, "tile_place": loc + 4 * wl.samples,
           "tile_scan": 12 * wl.B * wl.M * ((wl.S + 511) // 512),
           # the touch count of the FP32 workspace's rows: the locations, and
           # 2 bits of class per (b, pixel, head) row
           "touch_count": loc + wl.B * wl.S * wl.M // 4}
    if unique_rows is not None:
        urow = unique_rows * wl.D * es
        out["unique_rows"] = unique_rows
        out["forward_unique"] = urow + loc + attn + rowio
        out["bwd_total_unique"] = urow + rowio + 2 * (loc + attn) + n_value * es
    return out


# ---------------------------------------------------------------------------
# helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scale_deformable_attention_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, accum: str):
    """DRAM bytes per step of a kernel (its launches of one step together; per
    launch when it launches once) from a committed ncu capture, if it was
    taken on the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[f"{workload}/{accum}/{kernel}"]
        if e.get("source_hash") == kernel_source_hash():
            return float(e.get("dram_bytes_per_step", e.get("dram_bytes_per_launch")))
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm

class GpuStep:
    """Preallocated buffers and the raw C-ABI calls of one fwd+bwd step."""

    def __init__(self, wl: W.Workload, inp, accum: str, device):
        import torch

        import scale_deformable_attention_gb300 as msda
        from scale_deformable_attention_gb300 import _lib

        self.torch = torch
        self.msda = msda
        self.lib = _lib.lib()
        self.wl = wl
        self.device = device
        t = W.to_torch(inp, wl.dtype, device)
        self.t = t
        self.out = torch.empty((wl.B, wl.Qn, wl.M * wl.D), dtype=t["value"].dtype, device=device)
        self.gv = torch.empty_like(t["value"])
        self.gl = torch.empty_like(t["sampling_locations"])
        self.ga = torch.empty_like(t["attention_weights"])
        self.dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
        self.dt = msda.DTYPE_CODE[t["value"].dtype]
        self.accum = _lib.ACCUM[accum]
        need = int(self.lib.msda_backward_workspace_size(self.dt, self.accum, *self.dims))
        self.resolved = _lib.ACCUM_NAMES[int(self.lib.msda_resolve_accum(self.dt, self.accum, *self.dims))]
        # the FP32 accumulator's workspace is allocated once, cleared once, and
        # passed to every step as holding zeros: each step's rounding pass
        # clears what it used (MSDA_BWD_WORKSPACE_ZEROED)
        self.ws_zeroed = self.resolved == "fp32" and wl.dtype != "f32" and need > 0
        self.ws = torch.zeros(max(need // 4, 1), dtype=torch.float32, device=device)
        self.ws_bytes = need
        p = lambda x: x.data_ptr()  # noqa: E731
        self.fargs = (self.dt, *self.dims, p(t["value"]), p(t["spatial_shapes"]), p(t["level_start_index"]),
                      p(t["sampling_locations"]), p(t["attention_weights"]), p(self.out))
        flags = _lib.BWD_WORKSPACE_ZEROED if self.ws_zeroed else 0
        self.bargs = (self.dt, self.accum, flags, *self.dims, p(t["value"]), p(t["spatial_shapes"]),
                      p(t["level_start_index"]), p(t["sampling_locations"]), p(t["attention_weights"]),
                      p(t["grad_out"]), p(self.gv), p(self.gl), p(self.ga), p(self.ws), self.ws_bytes)
        self.flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def forward(self):
        from scale_deformable_attention_gb300 import _lib

        _lib.check(self.lib.msda_forward(*self.fargs, self.stream()))

    def backward(self):
        from scale_deformable_attention_gb300 import _lib

        _lib.check(self.lib.msda_backward(*self.bargs, self.stream()))

    def step(self):
        self.forward()
        self.backward()

    def flush(self):
        # read (not write) a buffer of 4x the L2: the L2 is left holding clean
        # lines, so the timed kernels neither hit their own data nor pay for
        # writing back someone else's dirty lines
        self.flush_sink = self.flush_buf.sum()

    def timed(self, fn, steps: int):
        """Device time of `fn` per step with the L2 flushed before each one (ms):
        CUDA events on the launching stream around each call, the flush
        outside them."""
        torch = self.torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            self.flush()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def timed_steps(self, steps: int):
        """As timed(step), plus the backward's share of each step: a third
        event between the forward and the backward.  Returns (step ms, backward
        ms) per step."""
        torch = self.torch
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
        for a, m, b in ev:
            self.flush()
            a.record()
            self.forward()
            m.record()
            self.backward()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, m, b in ev], [m.elapsed_time(b) for a, m, b in ev]


def _dist(backend: str = "nccl"):
    import torch.distributed as dist

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist if ws > 1 else None, int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def rank_workload(wl: W.Workload, rank: int) -> W.Workload:
    """Weak scaling: every rank runs the same sizes on its own seeded batch
    (the path shards over batches; no data-path exchange exists)."""
    return wl.with_(seed=wl.seed + 1000 * rank) if rank else wl


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time (barrier-bracketed timings are reduced by MAX)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job (b, q, m) outputs per second: all ranks' units over the max time."""
    return units_per_rank * world * steps / (total_ms / 1e3)


def unique_fractions(model: dict, kernels: dict, peak: float, bwd_wall_ms: float = None):
    """Compulsory-byte (unique value rows) fractions of the measured peak for
    the traced forward and backward (every other kernel of the step: zero,
    backward passes, convert) durations per step; the backward's wall time
    in the timed steps instead when given (its kernels may overlap on two
    streams)."""
    if "forward_unique" not in model or "forward" not in kernels or "backward" not in kernels:
        return None
    tf = kernels["forward"]["ms_per_step"]
    tb = bwd_wall_ms or sum(v["ms_per_step"] for k, v in kernels.items() if k != "forward")
    return {"unique_rows": model["unique_rows"], "forward_bytes": model["forward_unique"],
            "backward_bytes": model["bwd_total_unique"],
            "forward_frac": round(model["forward_unique"] / (tf / 1e3) / 1e9 / peak, 4),
            "backward_frac": round(model["bwd_total_unique"] / (tb / 1e3) / 1e9 / peak, 4),
            "peak": peak, "unit": "GB/s"}


def reduction_row_bytes(wl: W.Workload, accum: str) -> int:
    """Bytes of one corner row as the backward reduces it (D channels at the
    accumulator's width), rounded up to the probe's sizes (16 .. 512)."""
    es_acc = W.ESIZE[wl.dtype] if accum == "native" else 4
    rb = 16
    while rb < min(512, wl.D * es_acc):
        rb *= 2
    return rb


def reduction_ceiling_for(wl: W.Workload, accum: str):
    """32-byte reduction sectors per second the L2 takes for this backward's
    kind of reduction (msda_reduction_ceiling: whole corner rows, 16-byte
    reductions from adjacent lanes), or None (the deterministic accumulator's
    scalar integer reductions are another pattern)."""
    import torch

    import scale_deformable_attention_gb300 as msda

    if accum == "deterministic":
        return None
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[wl.dtype]
    return msda.reduction_ceiling(tdt if accum == "native" else torch.float32,
                                  row_bytes=reduction_row_bytes(wl, accum))


def reduction_roofline(wl: W.Workload, corners: int, accum: str, kernels: dict, ceiling):
    """The backward kernel against the L2's reduction ceiling: algorithmic
    sectors = in-level corner rows x 32-byte sectors per row at the
    accumulator's width (before the corner merge), over the traced kernel time."""
    if not ceiling or "backward" not in kernels:
        return None
    es_acc = W.ESIZE[wl.dtype] if accum == "native" else 4
    sectors = corners * ((wl.D * es_acc + 31) // 32)
    achieved = sectors / (kernels["backward"]["ms_per_step"] / 1e3)
    return {"kernel": "backward", "bound": "l2_reductions", "sectors": sectors,
            "achieved_gsectors_s": round(achieved / 1e9, 2), "ceiling_gsectors_s": round(ceiling / 1e9, 2),
            "frac": round(achieved / ceiling, 4),
            "ceiling_source": f"msda_reduction_ceiling on this GPU (random {reduction_row_bytes(wl, accum)}-byte rows, "
                              "16-byte reductions from adjacent lanes)"}


def graph_cross_check(st, steps: int):
    """The step captured once as a CUDA graph and replayed, timed like the
    bench's steps (L2 flushed, then events around each replay), beside the
    same number of stream-launched steps: a cross-check of the step time."""
    torch = st.torch
    s = torch.cuda.Stream(st.device)
    s.wait_stream(torch.cuda.current_stream(st.device))
    with torch.cuda.stream(s):
        st.step()
    torch.cuda.current_stream(st.device).wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.step()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    replay = st.timed(g.replay, steps)
    stream = st.timed(st.step, steps)
    del g
    return {"steps": steps, "graph_ms_per_step": round(sum(replay) / steps, 5),
            "stream_ms_per_step": round(sum(stream) / steps, 5)}


def l2_bytes(device) -> int:
    import torch

    return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (126 << 20))


def bound_of(kernel: str, wl: W.Workload, accum: str, l2: int, tiled: bool = False) -> str:
    """The ceiling that binds a kernel of this workload: HBM when its gathers
    (value) or its accumulator spill past the L2, else the L2 itself, for the
    backward its rate of reduction operations."""
    es = W.ESIZE[wl.dtype]
    value_bytes = wl.B * wl.S * wl.M * wl.D * es
    acc_bytes = wl.B * wl.S * wl.M * wl.D * (4 if accum == "fp32" else es)
    if kernel in ("zero", "convert"):
        return "hbm" if acc_bytes > l2 else "l2"
    if kernel == "tile_accum":
        return "hbm" if value_bytes > l2 else "l2"
    if kernel.startswith("tile_") or kernel == "touch_count":
        return "hbm" if wl.samples * 3 * es > l2 else "l2"
    if value_bytes > l2 or (kernel == "backward" and acc_bytes > l2):
        return "hbm"
    return "l2_reductions" if kernel == "backward" and not tiled else "l2"


def kernel_table(recs, steps: int):
    """Per-kernel launches, mean duration, time per step (a kernel may launch
    more than once per step: the backward runs one pass per level on large
    problems) and share of a traced pass of `steps` steps."""
    per = {}
    for name, ms, work in recs:
        per.setdefault(name, []).append(ms)
    tot = sum(sum(v) for v in per.values()) or 1.0
    return per, {k: {"launches": len(v), "avg_ms": round(statistics.mean(v), 5),
                     "ms_per_step": round(sum(v) / steps, 5), "share": round(sum(v) / tot, 4)}
                 for k, v in per.items()}


def traced_pass(st, steps: int):
    """Per-kernel durations: `steps` further steps with the library's kernel
    trace on (an event pair around every launch, no programmatic launches).
    Separate from the headline steps, which run untraced."""
    msda = st.msda
    msda.trace_enable(16 * steps + 16)
    st.timed(st.step, steps)
    recs, dropped = msda.trace_read()
    msda.trace_enable(0)
    return recs, dropped


def roofline_of(dom: str, per: dict, wl: W.Workload, model: dict, accum: str, l2: int, kernels: dict,
                bwd_wall_ms: float = None):
    """The dominant kernel against the measured HBM peak: its algorithmic
    bytes per step (per-corner model) over its traced time per step, i.e. the
    per-launch ratio when it launches once per step, and the launch-weighted
    one when it launches once per level.  The FP32 accumulator's backward is
    taken whole (its kernels overlap on two streams): over the wall time of
    the backward call in the timed steps, `bwd_wall_ms`."""
    peak, peak_kind = peaks()
    k = dict(kernels[dom])
    name = dom
    # the backward kernel without its scatter when the accumulate pass holds grad_value
    alg = model["backward_gather"] if dom == "backward" and "tile_accum" in per else model[dom]
    if dom == "backward" and "convert" in kernels and accum == "fp32" and wl.dtype != "f32":
        # FP32 accumulator: the backward passes round most of the workspace
        # themselves (extra blocks in the passes of the coarse levels), so the
        # rounding is counted with them: their bytes and their time together
        name = "backward+convert"
        alg = model["backward"] + model["convert"]
        c = kernels["convert"]
        t = kernels.get("touch_count", {"launches": 0, "ms_per_step": 0.0})
        launches = k["launches"] + c["launches"] + t["launches"]
        traced = k["ms_per_step"] + c["ms_per_step"] + t["ms_per_step"]
        if "touch_count" in kernels:
            alg += model["touch_count"]
        k = {"avg_ms": None, "launches": launches, "steps": k.get("steps", 1),
             "ms_per_step": round(bwd_wall_ms if bwd_wall_ms else traced, 5)}
    achieved = alg / (k["ms_per_step"] / 1e3) / 1e9
    roof = {"kernel": name, "bound": bound_of(dom, wl, accum, l2, "tile_accum" in per),
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(name, wl.name, accum),
            "algorithmic_bytes": alg, "bytes_model": "per-corner (every in-level corner row each time)",
            "avg_launch_ms": k["avg_ms"], "launches_per_step": round(k["launches"] / max(1, k.get("steps", 1)), 3),
            "ms_per_step": k["ms_per_step"], "peak_source": peak_kind, "launches_traced": k["launches"]}
    if name == "backward+convert" and bwd_wall_ms:
        roof["time_source"] = ("wall time of the backward call (every kernel from the touch count to the "
                               "rounding, two streams) in the timed steps, CUDA events on the launching stream")
    uf = unique_fractions(model, kernels, peak, bwd_wall_ms)
    if uf:
        roof["compulsory_frac"] = uf["backward_frac"] if dom != "forward" else uf["forward_frac"]
        roof["compulsory_scope"] = ("backward pass (every kernel after the forward)" if dom != "forward"
                                    else "forward pass")
    return roof


def run_ours(args):
    import torch

    dist, rank, world, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.with_(B=args.batch)
    wl = rank_workload(wl, rank)
    inp = W.make_inputs(wl)
    accum = args.accum or wl.accum
    st = GpuStep(wl, inp, accum, device)
    resolved = st.resolved
    corners, urows = corner_counts(wl, inp)
    model = byte_model(wl, corners, urows)
    red_ceiling = reduction_ceiling_for(wl, resolved)
    l2 = l2_bytes(device)

    for _ in range(max(args.warmup, 3)):
        st.flush()
        st.step()
    torch.cuda.synchronize()
    # launches per step, from one traced step outside the timed region
    msda.trace_enable(64)
    st.step()
    recs, _ = msda.trace_read()
    msda.trace_enable(0)
    launches_per_step = len(recs)

    # headline: the timed steps run untraced, with programmatic launches
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    uuid = str(torch.cuda.get_device_properties(device).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    with ClockSampler(uuid) as clk:
        times, bwd_times = st.timed_steps(args.steps)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(float(sum(times)), dist, device)
    ms_per_step = total_ms / args.steps
    value = job_throughput(wl.units, world, args.steps, total_ms)

    # per-kernel durations from a separate traced pass
    n_traced = max(4, min(args.steps, args.trace_steps))
    recs, dropped = traced_pass(st, n_traced)
    per, kernels = kernel_table(recs, n_traced)
    for v in kernels.values():
        v["steps"] = n_traced
    dom = max(per, key=lambda k: sum(per[k])) if per else None
    roof = roofline_of(dom, per, wl, model, resolved, l2, kernels, statistics.mean(bwd_times)) if dom else None
    peak, _ = peaks()

    graph = graph_cross_check(st, min(args.steps, 2000)) if not args.no_graph else None
    e2e = run_e2e(st, inp, args) if not args.no_e2e else None
    del st
    torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, inp, budget_s=args.cpu_seconds)
    others = None
    dispatch = None
    if rank == 0 and not args.no_configs:
        others = all_configs(args, device, wl.name, inp if wl.name == "stress_bf16" else None)
        dispatch = dispatch_timing(device)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "Q": wl.Qn, "M": wl.M, "D": wl.D, "L": wl.L, "K": wl.K,
                       "S": wl.S, "spatial_shapes": [list(s) for s in wl.shapes], "accum": accum,
                       "accum_resolved": resolved,
                       "workspace": ("allocated and cleared once; each step leaves it cleared "
                                     "(MSDA_BWD_WORKSPACE_ZEROED)") if resolved == "fp32" and wl.dtype != "f32"
                       else "none",
                       "l2": f"flushed between steps (read of a {FLUSH_BYTES >> 20} MB buffer, outside the timed events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "clocks": clk.summary(), "gpu_launches": launches_per_step * args.steps,
            "roofline": roof, "kernels": kernels, "kernels_source": "separate traced pass after the timed steps",
            "bytes_per_step_model": model["step"],
            "unique_model": unique_fractions(model, kernels, peak, statistics.mean(bwd_times)),
            "backward_wall_ms": round(statistics.mean(bwd_times), 5),
            "reduction_roofline": reduction_roofline(wl, corners, resolved, kernels, red_ceiling),
            "step_gbs_model": round(model["step"] / (ms_per_step / 1e3) / 1e9, 1),
            "e2e": e2e, "cpu_baseline": cpu, "trace_dropped": dropped, "graph_cross_check": graph,
            "all_configs": others, "dispatch": dispatch,
        }
        print(json.dumps(line), flush=True)
    if args.all and rank == 0:
        for name in W.WORKLOADS:
            print(json.dumps(run_workload_table(name, args, device)), flush=True)
    if args.fused and rank == 0:
        for name in ("decoder_bf16", "encoder_fp16"):
            print(json.dumps(run_fused_table(name, args, device)), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def config_entry(wl: W.Workload, inp, accum: str, device, n: int, l2: int):
    """Forward, backward and fwd+bwd device times (median of n, L2 flushed) of
    one workload and accumulator, with both byte models' fractions of the
    measured peak and the dominant kernel's bound."""
    import torch

    st = GpuStep(wl, inp, accum, device)
    corners, urows = corner_counts(wl, inp)
    model = byte_model(wl, corners, urows)
    peak, _ = peaks()
    for _ in range(3):
        st.step()
    tf = statistics.median(st.timed(st.forward, n))
    tb = statistics.median(st.timed(st.backward, n))
    ts = statistics.median(st.timed(st.step, n))
    recs, _ = traced_pass(st, 4)
    per, kernels = kernel_table(recs, 4)
    dom = max(per, key=lambda k: sum(per[k])) if per else None
    e = {"accum": accum, "accum_resolved": st.resolved, "fwd_ms": round(tf, 4), "bwd_ms": round(tb, 4),
         "step_ms": round(ts, 4), "step_units_per_s": round(wl.units / (ts / 1e3), 1),
         "fwd_frac_per_corner": round(model["forward"] / (tf / 1e3) / 1e9 / peak, 4),
         "bwd_frac_per_corner": round(model["bwd_total"] / (tb / 1e3) / 1e9 / peak, 4),
         "fwd_frac_compulsory": round(model["forward_unique"] / (tf / 1e3) / 1e9 / peak, 4),
         "bwd_frac_compulsory": round(model["bwd_total_unique"] / (tb / 1e3) / 1e9 / peak, 4),
         "kernels": kernels,
         "dominant": {"kernel": dom, "bound": bound_of(dom, wl, st.resolved, l2, "tile_accum" in per)} if dom else None}
    del st
    torch.cuda.empty_cache()
    return e


def all_configs(args, device, headline: str, headline_inp=None):
    """The other named workloads (and the headline one's other accumulator),
    each with its own inputs: every configuration in one run."""
    l2 = l2_bytes(device)
    res = {}
    for name in ("tiny_fp32", "decoder_bf16", "encoder_fp16", "oddD_fp32", "stress_bf16"):
        wl = W.WORKLOADS[name]
        if name == headline:
            if wl.dtype == "f32":
                continue
            inp = headline_inp if headline_inp is not None else W.make_inputs(wl)
            accums = ["native"] if wl.accum == "fp32" else ["fp32"]
        else:
            inp = W.make_inputs(wl)
            accums = ["auto"] + (["fp32"] if wl.dtype != "f32" else [])
        n = 5 if name == "stress_bf16" else 30
        res[name] = {"units": wl.units,
                     "runs": [config_entry(wl, inp, a, device, n, l2) for a in accums]}
        del inp
    return res


def dispatch_timing(device, calls: int = 200):
    """Dispatch-inclusive time per call on the decoder workload: `calls`
    back-to-back forward + backward calls through the autograd operator
    (multi_scale_deformable_attention, device-resident inputs and shapes, the
    leaves' gradients set to None before each call), one synchronisation at
    the end; beside the same calls through the raw C ABI.
    host_us: time until the loop has enqueued every call; wall_us: until the
    GPU has finished them."""
    import torch

    import scale_deformable_attention_gb300 as msda

    wl = W.WORKLOADS["decoder_bf16"]
    inp = W.make_inputs(wl)
    t = W.to_torch(inp, wl.dtype, device)
    leaves = [t[k].clone().requires_grad_(True) for k in ("value", "sampling_locations", "attention_weights")]
    ss, lsi, g = t["spatial_shapes"], t["level_start_index"], t["grad_out"]

    def autograd_call():
        # a training step's pattern: gradients set to None before each backward
        for v in leaves:
            v.grad = None
        out = msda.multi_scale_deformable_attention(leaves[0], ss, lsi, leaves[1], leaves[2])
        out.backward(g)

    def forward_call():
        with torch.no_grad():
            msda.multi_scale_deformable_attention(leaves[0], ss, lsi, leaves[1], leaves[2])

    st = GpuStep(wl, inp, "auto", device)
    res = {"workload": wl.name, "calls": calls}
    for tag, fn in (("autograd_op", autograd_call), ("autograd_op_forward_only", forward_call),
                    ("c_abi", st.step), ("c_abi_forward_only", st.forward)):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        res[tag] = {"host_us_per_call": round((t1 - t0) / calls * 1e6, 2),
                    "wall_us_per_call": round((t2 - t0) / calls * 1e6, 2)}
    del st
    return res


def run_e2e(st: GpuStep, inp, args):
    """Same metric through the public API with host inputs.  Every step copies
    its inputs host->device from pinned memory, runs forward + backward and
    copies its results (out, grad_value, grad_loc, grad_attn) device->host.
    Steps are double-buffered over three streams -- uploads of step i+1 and
    downloads of step i-1 run while step i computes (the host link is full
    duplex) -- with events ordering each buffer's reuse.  The timed region
    runs from the first upload to the last download."""
    torch = st.torch
    msda = st.msda
    wl = st.wl
    dev = st.device
    host_in = [{k: v.pin_memory() for k, v in W.to_torch(inp, wl.dtype, "cpu").items()} for _ in range(2)]
    out_shapes = {"out": (tuple(st.out.shape), st.out.dtype), "gv": (tuple(st.gv.shape), st.gv.dtype),
                  "gl": (tuple(st.gl.shape), st.gl.dtype), "ga": (tuple(st.ga.shape), st.ga.dtype)}
    host_out = [{k: torch.empty(sh, dtype=dt).pin_memory() for k, (sh, dt) in out_shapes.items()} for _ in range(2)]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in[0].items()} for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in host_in[0].values())
    bo = sum(t.numel() * t.element_size() for t in host_out[0].values())
    accum = st.resolved
    # one persistent workspace, cleared once (the compute stream runs the steps one after another)
    ws = st.ws if st.ws_zeroed else None
    steps = max(10, min(args.e2e_steps, args.steps))
    s_up, s_comp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    down_done = [ev(), ev()]
    consumed = [ev(), ev()]   # compute of buffer j finished reading dev_in[j]
    for e in up_done + comp_done + down_done + consumed:
        e.record(torch.cuda.current_stream(dev))
    results = [None, None]

    def one(i):
        j = i % 2
        with torch.cuda.stream(s_up):
            s_up.wait_event(consumed[j])
            for k in host_in[j]:
                dev_in[j][k].copy_(host_in[j][k], non_blocking=True)
            up_done[j].record(s_up)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(up_done[j])
            s_comp.wait_event(down_done[j])   # results[j] of step i-2 have been downloaded
            d = dev_in[j]
            out = msda.forward(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
                               d["attention_weights"], validate=False)
            gv, gl, ga = msda.backward(d["value"], d["spatial_shapes"], d["level_start_index"],
                                       d["sampling_locations"], d["attention_weights"], d["grad_out"], accum=accum,
                                       workspace=ws, workspace_zeroed=ws is not None, validate=False)
            results[j] = (out, gv, gl, ga)
            consumed[j].record(s_comp)
            comp_done[j].record(s_comp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(comp_done[j])
            for (k, t) in zip(("out", "gv", "gl", "ga"), results[j]):
                host_out[j][k].copy_(t, non_blocking=True)
                t.record_stream(s_down)
            down_done[j].record(s_down)

    for i in range(4):
        one(i)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(steps):
        one(i)
    b.record(s_down)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    return {"value": round(wl.units / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo), "ms_per_step": round(ms, 4), "steps": steps,
            "pipelining": "double-buffered: upload i+1 and download i-1 overlap compute i"}


def oracle_sample(wl: W.Workload, inp, queries: int):
    """Batch 0 and its first `queries` queries: a bounded sample of the
    workload for the oracle (its grad_value is then one batch image)."""
    q = int(max(1, min(wl.Qn, queries)))
    sub = {"value": inp["value"][:1], "spatial_shapes": inp["spatial_shapes"],
           "level_start_index": inp["level_start_index"]}
    for k in ("sampling_locations", "attention_weights", "grad_out"):
        sub[k] = np.ascontiguousarray(inp[k][:1, :q])
    return sub, q, q * wl.M


def cpu_baseline(wl: W.Workload, inp, budget_s: float):
    """The fp64 oracle on the host cores: whole fwd+bwd passes over a bounded
    sample of the same inputs (batch 0, a prefix of its queries sized so one
    pass takes about a second), repeated for about `budget_s` seconds."""
    import oracle

    sub, q, units = oracle_sample(wl, inp, min(wl.Qn, 256))
    t0 = time.perf_counter()
    oracle.forward(sub, wl.dtype)
    oracle.backward(sub, wl.dtype)
    t1 = time.perf_counter() - t0
    sub, q, units = oracle_sample(wl, inp, q * max(1.0, 1.0 / max(t1, 1e-3)))
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(sub, wl.dtype)
        oracle.backward(sub, wl.dtype)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(units * reps / el, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} fwd+bwd passes over batch 0, queries 0..{q - 1} of {wl.Qn} ({units} units each) "
                      f"of {wl.name}, in {el:.1f} s"}


def run_workload_table(name: str, args, device):
    """Forward / backward / fwd+bwd device times of one named workload."""
    import torch

    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    out = {}
    accums = ["native", "fp32", "deterministic"] if wl.dtype != "f32" else ["auto", "deterministic"]
    corners, urows = corner_counts(wl, inp)
    model = byte_model(wl, corners, urows)
    peak, _ = peaks()
    for accum in accums:
        st = GpuStep(wl, inp, accum, device)
        n = 5 if name == "stress_bf16" else 50
        for _ in range(3):
            st.step()
        tf = statistics.median(st.timed(st.forward, n))
        tb = statistics.median(st.timed(st.backward, n))
        ts = statistics.median(st.timed(st.step, n))
        out[accum] = {"fwd_ms": round(tf, 4), "bwd_ms": round(tb, 4), "step_ms": round(ts, 4),
                      "fwd_units_per_s": round(wl.units / (tf / 1e3), 1),
                      "bwd_units_per_s": round(wl.units / (tb / 1e3), 1),
                      "step_units_per_s": round(wl.units / (ts / 1e3), 1),
                      "fwd_frac_of_8TBs": round(model["forward"] / (tf / 1e3) / 8e12, 4),
                      "bwd_frac_of_8TBs": round(model["bwd_total"] / (tb / 1e3) / 8e12, 4),
                      "fwd_frac_of_measured": round(model["forward"] / (tf / 1e3) / 1e9 / peak, 4),
                      "bwd_frac_of_measured": round(model["bwd_total"] / (tb / 1e3) / 1e9 / peak, 4),
                      "fwd_unique_frac_of_8TBs": round(model["forward_unique"] / (tf / 1e3) / 8e12, 4),
                      "bwd_unique_frac_of_8TBs": round(model["bwd_total_unique"] / (tb / 1e3) / 8e12, 4),
                      "fwd_unique_frac_of_measured": round(model["forward_unique"] / (tf / 1e3) / 1e9 / peak, 4),
                      "bwd_unique_frac_of_measured": round(model["bwd_total_unique"] / (tb / 1e3) / 1e9 / peak, 4)}
        del st
        torch.cuda.empty_cache()
    return {"table": name, "units": wl.units, "corners_inside": corners, "bytes_model": model, "results": out}


def run_fused_table(name: str, args, device):
    """Device times of the fused operator (softmax of the logits and
    loc = ref + offset / (W, H) inside the kernels) against the same operator
    built from PyTorch ops around the core kernels, on one named workload."""
    import torch

    import scale_deformable_attention_gb300 as msda
    from scale_deformable_attention_gb300 import _lib

    wl = W.WORKLOADS[name]
    inp = W.make_fused_inputs(wl)
    t = W.to_torch(inp, wl.dtype, device)
    lib = _lib.lib()
    dims = (wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn)
    dt = msda.DTYPE_CODE[t["value"].dtype]
    B, Q, M, L, K = wl.B, wl.Qn, wl.M, wl.L, wl.K
    p = lambda x: x.data_ptr()  # noqa: E731
    out = torch.empty((B, Q, M * wl.D), dtype=t["value"].dtype, device=device)
    gv = torch.empty_like(t["value"])
    gr = torch.empty_like(t["reference_points"])
    go = torch.empty_like(t["sampling_offsets"])
    gz = torch.empty_like(t["attention_logits"])
    ss = t["spatial_shapes"]
    norm = torch.stack([ss[:, 1], ss[:, 0]], -1).to(torch.float32)            # [L, 2] = (W, H)
    flush_buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    st = lambda: torch.cuda.current_stream(device).cuda_stream  # noqa: E731
    # pixel coordinates of the fused locations (binary32, as the kernels) for the byte model
    es = W.ESIZE[wl.dtype]
    ref = W.to_f64(inp["reference_points"], wl.dtype).astype(np.float32)
    off = W.to_f64(inp["sampling_offsets"], wl.dtype).astype(np.float32)
    nrm = np.array([[w, h] for h, w in wl.shapes], dtype=np.float32)
    loc = ref[:, :, None, :, None, :] + off / nrm[None, None, None, :, None, :]
    corners = inbounds_corners(wl.with_(dtype="f32"), {"sampling_locations": loc.astype(np.float32)})
    gather = corners * wl.D * es
    refb = B * Q * L * 2 * es
    params = wl.samples * 3 * es
    rowio = wl.units * wl.D * es
    n_value = wl.B * wl.S * wl.M * wl.D
    model = {"forward": gather + refb + params + rowio,
             "bwd_total": 2 * gather + rowio + refb + 2 * params + n_value * es + wl.samples * 2 * es + refb}
    res = {}
    for accum in (["native", "fp32", "deterministic"] if wl.dtype != "f32" else ["auto", "deterministic"]):
        acc = _lib.ACCUM[accum]
        need = int(lib.msda_backward_workspace_size(dt, acc, *dims))
        ws = torch.empty(max(need // 4, 1), dtype=torch.float32, device=device)

        def fwd():
            _lib.check(lib.msda_forward_fused(dt, *dims, p(t["value"]), p(ss), p(t["level_start_index"]),
                                              p(t["reference_points"]), p(t["sampling_offsets"]),
                                              p(t["attention_logits"]), p(out), st()))

        def bwd():
            _lib.check(lib.msda_backward_fused(dt, acc, 0, *dims, p(t["value"]), p(ss), p(t["level_start_index"]),
                                               p(t["reference_points"]), p(t["sampling_offsets"]),
                                               p(t["attention_logits"]), p(t["grad_out"]), p(gv), p(gr), p(go),
                                               p(gz), p(ws), need, st()))

        # the same operator from PyTorch ops around the core kernels
        saved = {}

        def fwd_torch():
            A = torch.softmax(t["attention_logits"].float(), -1).to(t["value"].dtype).view(B, Q, M, L, K)
            lc = (t["reference_points"].float()[:, :, None, :, None, :] +
                  t["sampling_offsets"].float() / norm[None, None, None, :, None, :]).to(t["value"].dtype)
            saved["A"], saved["loc"] = A, lc
            msda.forward(t["value"], ss, t["level_start_index"], lc, A, out=out, validate=False)

        def bwd_torch():
            A, lc = saved["A"], saved["loc"]
            g_v, g_l, g_a = msda.backward(t["value"], ss, t["level_start_index"], lc, A, t["grad_out"], accum=accum,
                                          grad_value=gv, workspace=ws if need else None, validate=False)
            g_l = g_l.float()
            g_off = (g_l / norm[None, None, None, :, None, :]).to(t["value"].dtype)
            g_ref = g_l.sum(dim=(2, 4)).to(t["value"].dtype)
            a2 = A.float().reshape(B, Q, M, L * K)
            ga2 = g_a.float().reshape(B, Q, M, L * K)
            g_z = (a2 * (ga2 - (a2 * ga2).sum(-1, keepdim=True))).to(t["value"].dtype)
            return g_v, g_ref, g_off, g_z

        def timed(fn, n):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for a, b in ev:
                flush_buf.sum()
                a.record()
                fn()
                b.record()
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ev)

        n = 50
        for _ in range(3):
            fwd(), bwd(), fwd_torch(), bwd_torch()
        r = {}
        for tag, f, b in (("fused", fwd, bwd), ("torch_ops_around_core", fwd_torch, bwd_torch)):
            tf = timed(f, n)
            f()
            tb = timed(b, n)
            ts = timed(lambda: (f(), b()), n)
            r[tag] = {"fwd_ms": round(tf, 4), "bwd_ms": round(tb, 4), "step_ms": round(ts, 4)}
        r["fused"]["fwd_frac_of_measured"] = round(model["forward"] / (r["fused"]["fwd_ms"] / 1e3) / 1e9 / peaks()[0], 4)
        r["fused"]["bwd_frac_of_measured"] = round(model["bwd_total"] / (r["fused"]["bwd_ms"] / 1e3) / 1e9 /
                                                   peaks()[0], 4)
        r["step_speedup"] = round(r["torch_ops_around_core"]["step_ms"] / r["fused"]["step_ms"], 3)
        res[accum] = r
        del ws
    return {"table": "fused", "workload": name, "units": wl.units, "corners_inside": corners, "bytes_model": model,
            "results": res}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    wl = W.WORKLOADS[args.workload]
    inp = W.make_inputs(wl)
    # each step is one fwd+bwd pass of the oracle over batch 0 and a prefix of
    # its queries, sized so that warm-up and timed steps take about ref_budget
    sub, q, units = oracle_sample(wl, inp, min(wl.Qn, 64))
    t0 = time.perf_counter()
    oracle.forward(sub, wl.dtype)
    oracle.backward(sub, wl.dtype)
    t_probe = time.perf_counter() - t0
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    sub, q, units = oracle_sample(wl, inp, q * per_step / max(t_probe, 1e-6))
    for _ in range(args.warmup):
        oracle.forward(sub, wl.dtype)
        oracle.backward(sub, wl.dtype)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(sub, wl.dtype)
        oracle.backward(sub, wl.dtype)
    el = time.perf_counter() - t0
    value = units * args.steps / el
    sample = f"batch 0, queries 0..{q - 1} of {wl.Qn} ({units} (b,q,m) units) per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "Q": wl.Qn, "M": wl.M, "D": wl.D, "L": wl.L, "K": wl.K,
                       "S": wl.S, "spatial_shapes": [list(x) for x in wl.shapes], "accum": "fp64 (oracle)",
                       "parallelism": f"host cores ({oracle.num_threads()} threads), rank 0 only"},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stress_bf16", choices=sorted(W.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size B")
    ap.add_argument("--accum", choices=["auto", "native", "fp32", "deterministic"], default=None,
                    help="grad_value accumulator (default: the workload's)")
    ap.add_argument("--all", action="store_true", help="also print per-workload fwd/bwd tables")
    ap.add_argument("--fused", action="store_true",
                    help="also print fused-operator vs PyTorch-ops-around-the-core tables")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay cross-check")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--trace-steps", type=int, default=16,
                    help="steps of the separate traced pass that gives per-kernel durations")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' entries (all_configs) and the dispatch timing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds of oracle work for --impl reference")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
