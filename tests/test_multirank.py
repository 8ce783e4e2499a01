"""Host-side logic of the multi-process bench on CPU: two gloo ranks, each a
replica with its own work, combined as (units summed over ranks) / (slowest
rank's time).  The path has no data exchange, so this is the only collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    r, w, local = bench.dist_env()
    ranks = bench.Ranks(w, "gloo")
    ranks.barrier()
    units, seconds = bench.combine(ranks, units=1000.0 * (rank + 1), seconds=0.5 + rank)
    ranks.barrier()
    ranks.close()
    q.put((r, w, local, units, seconds))


def test_two_gloo_ranks_combine():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, units, seconds) in enumerate(out):
        assert (r, w, local) == (rank, world, rank)
        assert units == 3000.0          # 1000 + 2000
        assert seconds == 1.5           # the slower rank


def test_single_process_is_identity():
    import bench
    ranks = bench.Ranks(1, "gloo")
    assert bench.combine(ranks, 42.0, 0.25) == (42.0, 0.25)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank, monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", str(rank))
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 3, 3, 2
    assert bench.reference_arm(A) == 0
    out = capsys.readouterr().out.strip()
    if rank == 0:
        import json
        line = json.loads(out)
        assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
        assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    else:
        assert out == ""
