"""Host logic of bench.py, without a GPU: the pass schedule of the timed
region, the per-weight-type workloads, and the multi-process path (N > 1
runs independent replicas: the timing is the slowest rank's, the value the
total over ranks), with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


class FakeModel:
    def __init__(self):
        self.calls = []

    def decode_step(self, token, position):
        self.calls.append(("step", token, position))

    def decode_greedy(self, n):
        self.calls.append(("greedy", n))


@pytest.mark.parametrize("wdtype", ["f32", "int4", "f16"])
def test_step_runner_keeps_the_workload_positions(wdtype):
    bench.set_workload(wdtype)
    prompt_len, cycle = bench.WORKLOADS[wdtype]
    m = FakeModel()
    r = bench.StepRunner(m, first_token=7)
    steps = 2 * cycle + 5
    r.run(steps - 3)
    r.run(3)                                 # split calls continue the cycle
    passes, pos = 0, None
    for c in m.calls:
        if c[0] == "step":
            assert c[1:] == (7, prompt_len)  # each cycle re-enters its first position with its first token
            pos = prompt_len + 1
            passes += 1
        else:
            pos += c[1]
            passes += c[1]
            assert pos <= prompt_len + cycle  # never past the workload's last position
    assert passes == steps
    assert sum(1 for c in m.calls if c[0] == "step") == 3
    bench.set_workload("f32")


def test_workloads_follow_the_configurations():
    assert bench.WORKLOADS["f32"] == (10, 60)
    assert bench.WORKLOADS["int4"] == (10, 128)
    assert bench.WORKLOADS["f16"] == (16, 1008)
    assert sum(bench.WORKLOADS["f16"]) == 1024      # to the full 1024-position cache
    bench.set_workload("int4")
    cfg = bench.workload_config("int4", 1, "f32")
    assert "10-token prompt + 128 greedy decode steps (positions 10..137)" in cfg["workload"]
    bench.set_workload("f32")


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    assert bench.job_throughput(1000, 1, 500.0) == pytest.approx(2000.0)
    assert bench.job_throughput(1000, 4, 500.0) == pytest.approx(8000.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 37.0 * rank                 # rank 1 is the slowest
        slowest = bench.reduce_max(ms, world, "cpu")
        out[rank] = (slowest, bench.job_throughput(50, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_time_and_the_total():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                          # every rank agrees
    slowest, value = res[0]
    assert slowest == pytest.approx(137.0)
    assert value == pytest.approx(50 * 2 / 0.137)


def test_reference_arm_on_other_ranks_exits_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        wdtype, steps, warmup, head = "f32", 5, 3, "f32"

    assert bench.run_reference(A()) == 0
