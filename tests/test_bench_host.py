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
    prompt_len, cycle = bench.WORKLOADS[wdtype]
    m = FakeModel()
    r = bench.StepRunner(m, first_token=7, n_prompt=prompt_len, cycle=cycle)
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
    # the roofline averages over exactly the positions these passes ran
    pos_seen = []
    for c in m.calls:
        if c[0] == "step":
            pos_seen.append(c[2])
        else:
            pos_seen.extend(range(pos_seen[-1] + 1, pos_seen[-1] + 1 + c[1]))
    assert pos_seen == bench.timed_positions(wdtype, steps)


def test_workloads_follow_the_configurations():
    assert bench.WORKLOADS["f32"] == (10, 60)
    assert bench.WORKLOADS["int4"] == (10, 128)
    assert bench.WORKLOADS["f16"] == (16, 1008)
    assert sum(bench.WORKLOADS["f16"]) == 1024      # to the full 1024-position cache
    cfg = bench.workload_config("int4", 1, "f32")
    assert "10-token prompt + 128 greedy decode steps (positions 10..137)" in cfg["workload"]
    # the driver's short run (20 steps) times positions 10..29 only
    assert bench.timed_positions("f32", 20) == list(range(10, 30))


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


def test_traffic_figures_are_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    """A committed DRAM-traffic figure counts only while the kernel sources it
    was captured on are unchanged."""
    import json
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "traffic.json").write_text(json.dumps(
        {"cluster": {"f32": {"bytes": 123, "sources": sha}, "int4": {"bytes": 45, "sources": "0" * 16}}}))
    csrc = tmp_path / "transformer_decode_token_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("cluster.cu", "cluster.h", "common.cuh"):
        src = os.path.join(ROOT, "transformer_decode_token_gb300", "csrc", name)
        (csrc / name).write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("cluster", "f32") == 123
    assert bench.load_traffic("cluster", "int4") is None      # captured on other sources
    assert bench.load_traffic("cluster", "f16") is None       # never captured
    (csrc / "cluster.cu").write_bytes(b"changed")
    assert bench.load_traffic("cluster", "f32") is None


def test_reference_arm_reports_the_same_config_as_ours(monkeypatch, capsys):
    """The reference arm (the oracle) prints the headline's metric, unit and
    config, so the two lines describe the same workload."""
    import json
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: (5, 0.5))
    a = bench.parse(["--impl", "reference", "--steps", "5", "--warmup", "3"])
    assert bench.run_reference(a) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["config"] == bench.workload_config("f32", 1, "f32")
    assert line["value"] == pytest.approx(10.0) and line["cpu_baseline"]["kind"] == "oracle"
