"""bench.py's multi-GPU plumbing (independent replicas: a barrier and a
max/sum over ranks of the timing and the work, no data-path collective),
run as two gloo ranks on the CPU."""

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


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    elapsed = 10.0 + 5.0 * rank          # rank 1 is the slower replica
    work = 100.0 * (rank + 1)
    t_max = bench.max_over_ranks(elapsed, w, torch.device("cpu"))
    total = bench.sum_over_ranks(work, w, torch.device("cpu"))
    out[rank] = (t_max, total)
    dist.destroy_process_group()


def test_two_replicas_max_time_and_total_work():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # every rank sees the slowest replica's time and all replicas' work;
    # value = total work / max time
    assert out[0] == out[1] == (15.0, 300.0)


def test_single_process_defaults(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.sum_over_ranks(4.0, 1, None) == 4.0


def test_reference_arm_non_zero_rank_does_no_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("workload", ["small", "int8"])
def test_reference_arm_prints_the_contract_line(monkeypatch, capsys, workload):
    """--impl reference on rank 0 runs the oracle on the host cores (no GPU)
    and prints one JSON line with the base contract's keys, the reference
    arm's e2e and cpu_baseline objects."""
    import json

    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "0",
                "--reference-rows", "4"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"]
