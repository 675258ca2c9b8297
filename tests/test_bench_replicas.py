"""The multi-GPU path of bench.py on the CPU: N > 1 runs independent replicas
(each rank its own batch, no data-path collective), and the whole-job figure
takes the slowest rank's time and every rank's work.  Two gloo ranks check the
reduction bench.py applies to its timings (the GPU kernels are not involved).
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402

ELAPSED_MS = (3.0, 5.0)  # per rank
UNITS = (432, 400)       # verified draft tokens per step, per rank
STEPS = 10


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, total = bench.reduce_over_ranks(ELAPSED_MS[rank], UNITS[rank], torch.device("cpu"), world)
        q.put((rank, ms, total, bench.whole_job_rate(total, STEPS, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, ms, total, rate in res:
        assert ms == max(ELAPSED_MS)
        assert total == float(sum(UNITS))
        assert rate == pytest.approx(sum(UNITS) * STEPS / (max(ELAPSED_MS) / 1e3))


def test_one_rank_reports_its_own_figures():
    ms, total = bench.reduce_over_ranks(4.0, 432, None, 1)
    assert (ms, total) == (4.0, 432.0)
    assert bench.whole_job_rate(total, STEPS, ms) == pytest.approx(432 * STEPS / 4e-3)


def test_rank_environment_defaults_to_one_process(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (1, 2, 1)


def test_every_workload_has_a_config_line():
    import sdsynth as S
    for name, w in S.WORKLOADS.items():
        c = bench.config_of(w)
        assert c["workload"] == name
        assert c["mode"] in ("adaptive", "all_slots", "uniform_k")
    assert bench.config_of(S.WORKLOADS["uniform_hc"])["mode"] == "uniform_k"


def test_oracle_all_cores_leg_runs_on_the_host():
    """The all-cores oracle timing (spawned processes, requests dealt
    round-robin) returns a positive rate and the process count it used."""
    import sdsynth as S
    r = bench.oracle_all_cores(S.WORKLOADS["tiny"], 7, 1.0, workers=2)
    assert "error" not in r
    assert r["cores"] == 2 and r["value"] > 0 and r["kind"] == "oracle"
    assert bench.all_cores_or_error(S.WORKLOADS["tiny"].with_(name="no_such_workload"), 7, 1.0)["error"]
