"""The benchmark's multi-GPU path on CPU: N ranks run independent replicas of
the step, the job's time per step is the slowest rank's, and the value counts
the tensors of every rank.  Two gloo ranks stand in for two GPUs; the
reference arm does its work on rank 0 only."""
import json
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = 1.0 + rank * 0.5                     # rank 1 is the slower one
        job_ms = bench.max_over_ranks(ms, "cpu")
        line = bench.step_line(job_ms, ws, steps=10, warmup=3, peak=6771.5)
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"job_ms": job_ms, "line": line}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_tensors(tmp_path):
    ws = 2
    mp.start_processes(_rank, args=(ws, _free_port(), str(tmp_path)), nprocs=ws,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(ws)]
    assert res[0]["job_ms"] == res[1]["job_ms"] == 1.5
    line = res[0]["line"]
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["ms_per_step"] == 1.5
    expect = 2 * 4 * bench.ALG_BYTES / 1.5e-3 / 1e9
    assert line["value"] == pytest.approx(expect, abs=0.01)
    assert line["pct_of_peak"] == pytest.approx(100 * expect / 2 / 6771.5, abs=0.01)


def test_without_a_process_group_the_rank_time_is_the_job_time():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(2.25, "cpu") == 2.25
    line = bench.step_line(2.0, 1, steps=5, warmup=3, peak=6771.5)
    assert line["value"] == pytest.approx(4 * bench.ALG_BYTES / 2e-3 / 1e9, abs=0.01)
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""
