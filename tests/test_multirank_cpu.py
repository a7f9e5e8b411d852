"""The multi-rank parts of bench.py on CPU with the gloo backend (world size 2):
the max-over-ranks timing reduction and the whole-job rate.  The codec itself
runs one independent replica per GPU (no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank  # the slower rank decides the job time
        worst = bench.dist_max(ms)
        out[rank] = (worst, bench.whole_job_gbs(world, 1e9, worst))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    assert res[0] == res[1]
    worst, gbs = res[0]
    assert worst == 15.0
    assert gbs == pytest.approx(2 * 1e9 / 15e-3 / 1e9)


def test_single_process_identity():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.dist_max(3.5) == 3.5
    assert bench.whole_job_gbs(1, 2e9, 1000.0) == pytest.approx(2.0)


def test_bench_starts_its_own_ranks(capfd):
    """--gpus 2 without a torchrun environment: bench.launch_ranks starts two
    ranks (torch.distributed.run, gloo on CPU); the stand-in rank reports the
    whole-job line with n_gpus 2 and the slower rank's time."""
    import json
    import sys

    sys.path.insert(0, ROOT)
    import bench

    env_before = os.environ.pop("WORLD_SIZE", None)
    try:
        rc = bench.launch_ranks(2, [], script=os.path.join(ROOT, "tests", "bench_rank_stub.py"))
    finally:
        if env_before is not None:
            os.environ["WORLD_SIZE"] = env_before
    out = capfd.readouterr().out
    assert rc == 0, out
    lines = [json.loads(l) for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["ms_per_step"] == 15.0
    assert lines[0]["value"] == pytest.approx(2 * 1e9 / 15e-3 / 1e9)
