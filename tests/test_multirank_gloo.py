"""The benchmark's multi-rank host logic on the CPU: two gloo ranks (world size 2).

Every rank runs an independent replica of the workload (heads need no exchange), so
the only cross-rank operations are the barrier and the max / sum of per-rank timings;
the reference arm runs on rank 0 alone."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench

    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    mx = bench.reduce_max(dist, 1.5 + rank)
    sm = bench.reduce_sum(dist, 10.0 * (rank + 1))
    bench.barrier(dist)
    dist.destroy_process_group()
    results[rank] = (mx, sm)


def test_two_gloo_ranks_reduce_timings():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == (2.5, 30.0)


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max(None, 3.25) == 3.25
    assert bench.reduce_sum(None, 3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_config_names_replicas():
    import bench
    import synth

    cfg = bench.config_dict(synth.WORKLOADS[3], 4)
    assert cfg["workload"] == "b2h32_n8192_d128_causal"
    assert "replicas x4" in cfg["parallelism"]
    assert cfg["l2"].startswith("inputs larger than L2")
