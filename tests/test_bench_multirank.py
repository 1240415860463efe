"""bench.py's multi-rank path on CPU: two gloo ranks (world_size 2).

Each rank runs an independent replica; the job's step time is the max over
ranks and ``value`` is all ranks' tokens over that time. Checked here with the
same helpers bench.py uses, on a gloo process group over 127.0.0.1.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local, d = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank) and d is not None
    dev = torch.device("cpu")
    bench.barrier(d, dev)
    step_ms = [2.0, 5.0][rank]                       # rank 1 is the slow one
    ms_max = bench.reduce_max(d, step_ms, dev)
    value = bench.aggregate(ms_max / 1e3, 4096, w)
    out[rank] = (ms_max, value)
    d.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms_max, value = out[0]
    assert ms_max == 5.0
    assert value == pytest.approx(2 * 4096 / 5e-3)


def test_single_process_needs_no_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    r, w, local, d = bench.dist_setup(1)
    assert (r, w, local, d) == (0, 1, 0, None)
    assert bench.reduce_max(None, 3.5, torch.device("cpu")) == 3.5
    assert bench.aggregate(0.5, 100, 1) == 200


def test_gpus_flag_is_never_ignored():
    """--gpus N > 1 without torchrun relaunches N ranks; inside a torchrun job
    WORLD_SIZE must equal N; N < 1 is refused."""
    import bench
    assert bench.launch_plan(1, {}) == "single"
    assert bench.launch_plan(4, {}) == "spawn"
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}) == "rank"
    assert bench.launch_plan(1, {"WORLD_SIZE": "1"}) == "single"
    with pytest.raises(SystemExit):
        bench.launch_plan(8, {"WORLD_SIZE": "2"})
    with pytest.raises(SystemExit):
        bench.launch_plan(0, {})
