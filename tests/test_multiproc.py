"""The N > 1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py runs one replica per GPU (the path shards by rows, tokens and
sequences with no exchange); the only cross-rank steps are the timing
barrier and the max over ranks, checked here without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, results):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        local_ms = 10.0 + 7.5 * rank  # rank 1 is the slow one
        job = bench._job_time_ms(local_ms, ws, "cpu")
        rate = bench._job_rate(2048, 20, ws, job)
        results[rank] = (job, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(ws, port, results), nprocs=ws, join=True)
        res = dict(results)
    assert set(res) == {0, 1}
    for job, rate in res.values():
        assert job == pytest.approx(17.5)  # the slowest rank's time
        assert rate == pytest.approx(2 * 2048 * 20 / 0.0175)  # whole-job tokens over the job time


def test_single_rank_needs_no_process_group():
    assert bench._job_time_ms(12.5, 1, "cpu") == 12.5
    assert bench._job_rate(2048, 10, 1, 20.0) == pytest.approx(2048 * 10 / 0.02)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # under torchrun every rank calls the reference arm; ranks > 0 exit 0 quietly
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class A:
        gpus, steps, warmup = 2, 1, 3

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    # the one bench arm that needs no GPU: the oracle on the host cores, one
    # bounded sample per step, printed as one JSON line of the bench contract
    import json

    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")

    class A:
        gpus, steps, warmup = 1, 1, 0

    assert bench.run_reference(A()) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["value"] > 0 and d["ms_per_step"] == pytest.approx(1000.0 * bench.M_TOK / d["value"])
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
