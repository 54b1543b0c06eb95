"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2): each
rank gets its own seeded batch of the same sizes (weak scaling, no data-path
exchange), timings reduce by MAX over ranks, and the job throughput counts
every rank's units over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import workloads as W

    d, r, w, local = bench._dist("gloo")
    try:
        wl = bench.rank_workload(W.WORKLOADS["decoder_bf16"], r)
        own_ms = 10.0 + 5.0 * r
        total = bench.max_over_ranks(own_ms, d, "cpu")
        value = bench.job_throughput(wl.units, w, 100, total)
        inp = W.make_inputs(wl.with_(B=1, Q=3))
        q.put((r, w, wl.seed, (wl.B, wl.Qn, wl.M), total, value, inp["value"].tobytes()[:64]))
        d.barrier()
    finally:
        d.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (r0, w0, s0, shp0, t0, v0, b0), (r1, w1, s1, shp1, t1, v1, b1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2
    assert shp0 == shp1                       # same per-rank work
    assert s0 != s1 and b0 != b1              # different batches
    assert t0 == t1 == 15.0                   # MAX over ranks
    assert v0 == v1 == pytest.approx(9600 * 2 * 100 / 0.015)
