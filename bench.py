#!/usr/bin/env python
"""GPT-2 124M batch-1 greedy decode throughput on GB300.

Workload (default): GPT-2 small (12 layers, n_embd 768, 12 heads, vocab 50257,
1024 positions), fp32 weights drawn from N(0, 0.02) with seed 0, a 10-token
prompt (seed 1) and 60 greedy decode steps at positions 10..69.  With
--wdtype int4 the block matrices are grouped int4 and the workload is a
10-token prompt + 128 steps; with --wdtype f16 they are fp16 and the workload
is a 16-token prompt decoded to the full 1024-position cache (1008 steps),
with tok/s and GB/s also reported per 64 positions ("context_sweep").  A bench
"step" is one decode pass over one token: embedding, 12 blocks, final
LayerNorm, tied head and argmax.  The timed region runs exactly --steps
passes; they cycle through the workload's generation (each cycle re-enters
its first position with the generation's first token, the rest are
device-fed greedy passes), so any step count keeps the workload's positions.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--wdtype f32|f16|int4]
  python bench.py --impl reference ...     # the CPU oracle, same metric

Prints one JSON line on rank 0.  N > 1 runs N independent replicas (one
process per GPU, launched by torchrun); the value is the total over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GPT-2 124M decode tok/s @batch1; achieved HBM GB/s vs GB300 peak"
UNIT = "tok/s"
# The workload of each block-weight type (GPT-2 small; prompt tokens, greedy
# passes): fp32 10 + 60, int4 10 + 128, fp16 16 + 1008 (to the full
# 1024-position cache, with tok/s reported per 64 positions).
WORKLOADS = {"f32": (10, 60), "int4": (10, 128), "f16": (16, 1008)}
PROMPT_LEN, CYCLE = WORKLOADS["f32"]
SWEEP_BUCKET = 64


def set_workload(wdtype: str):
    global PROMPT_LEN, CYCLE
    PROMPT_LEN, CYCLE = WORKLOADS[wdtype]
L2_BYTES = 129 * 1024 * 1024
CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=120)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--wdtype", choices=["f32", "f16", "int4"], default="f32")
    p.add_argument("--head", choices=["f32", "f16", "int4"], default="f32",
                   help="LM head storage: the tied fp32 wte (the configurations), an fp16 copy (README -h) or int4")
    p.add_argument("--e2e-calls", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", choices=["auto", "persistent", "per_kernel"], default="auto",
                   help="auto: the cluster decode kernel where the device allows it")
    a = p.parse_args()
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def workload_config(wdtype: str, world: int, head: str = "f32") -> dict:
    return {"workload": f"GPT-2 small 124M, {wdtype} block weights, {head} LM head, batch 1, {PROMPT_LEN}-token prompt "
                        f"+ {CYCLE} greedy decode steps (positions {PROMPT_LEN}..{PROMPT_LEN + CYCLE - 1}), "
                        "cycled",
            "n_layer": 12, "n_embd": 768, "n_head": 12, "vocab": 50257, "n_positions": 1024,
            "batch": 1, "weights": "synthetic N(0,0.02), seed 0; prompt ids uniform, seed 1",
            "l2": "no flush: every step streams all weights (f32 494.6 MB, f16 324.7 MB, int4 209.3 MB) "
                  "through a 129 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ---- clocks ------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 3.0:
            time.sleep(0.02)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self, t_begin: float, t_end: float):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=3)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [ln for (t, ln) in self.lines if t_begin - 0.05 <= t <= t_end + 0.15]
        if not rows:
            rows = [ln for (_, ln) in self.lines[-3:]]
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def gpu_id_for(torch, dev: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def load_traffic():
    """DRAM bytes per decode pass from the committed ncu summaries, by path and
    weight type ({path: {wdtype: bytes}}), if any."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            return json.load(f)
    except OSError:
        return {}


# ---- CPU oracle timing -------------------------------------------------------

def oracle_sample(cfg, weights, prompt, wdtype, budget_s, max_steps=None, head="f32"):
    """Decode passes of the oracle after an untimed prefill; stops after
    ~budget_s seconds (or max_steps).  Returns (passes, seconds)."""
    from oracle import oracle as orc
    sw = orc.stored_weights(weights, wdtype, head=head)
    m = orc.OracleModel(cfg, sw)
    try:
        tok = None
        for pos, t in enumerate(prompt):
            _, tok = m.forward(int(t), pos)
        n, pos = 0, len(prompt)
        t0 = time.perf_counter()
        while True:
            if pos >= PROMPT_LEN + CYCLE:           # keep the workload's positions
                pos = PROMPT_LEN
            _, tok = m.forward(tok, pos)
            pos += 1
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s or (max_steps is not None and n >= max_steps):
                return n, el
    finally:
        m.close()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from transformer_decode_token_gb300 import synth
    cfg = synth.SMALL
    w = synth.make_weights(cfg, 0)
    prompt = synth.make_prompt(cfg, PROMPT_LEN, 1)
    oracle_sample(cfg, w, prompt, args.wdtype, 1e9, max_steps=min(args.warmup, 3), head=args.head)
    n, el = oracle_sample(cfg, w, prompt, args.wdtype, 60.0, max_steps=args.steps, head=args.head)
    value = n / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args.wdtype, 1, args.head),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n} of the {args.steps} requested decode passes (60 s cap), "
                                       "single-threaded C oracle, after an untimed 10-token prefill"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- our arm -------------------------------------------------------------------

def reduce_max(v: float, world: int, device: str) -> float:
    """The largest of the ranks' values (the slowest rank's time); the
    process group must be initialised when world > 1."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps_per_rank: int, world: int, ms_slowest: float) -> float:
    """Whole-job passes per second: every rank's passes over the slowest
    rank's time (replicas: each rank runs its own sequence)."""
    return steps_per_rank * world / (ms_slowest / 1e3)


class StepRunner:
    """Queues decode passes that cycle through the 60-step generation."""

    def __init__(self, model, first_token: int):
        self.m = model
        self.tok0 = first_token
        self.k = 0
        self.host_steps = 0

    def run(self, n: int):
        while n > 0:
            if self.k % CYCLE == 0:
                self.m.decode_step(self.tok0, PROMPT_LEN)
                self.host_steps += 1
                self.k += 1
                n -= 1
            else:
                c = min(n, CYCLE - self.k % CYCLE)
                self.m.decode_greedy(c)
                self.k += c
                n -= c


def main():
    args = parse()
    set_workload(args.wdtype)
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist
    from transformer_decode_token_gb300 import binding, roofline, synth

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return reduce_max(v, world, "cuda")

    cfg = synth.SMALL
    w = synth.make_weights(cfg, 0)
    prompt = synth.make_prompt(cfg, PROMPT_LEN, 1)
    dw = binding.upload_weights(w)
    model = binding.Model(cfg, dw, args.wdtype, path=args.path, head=args.head)
    del dw
    torch.cuda.empty_cache()
    kps = model.kernels_per_step()
    path = model.path()

    # ---- device-timed value ----
    model.prefill(prompt)
    tok0 = model.argmax()
    runner = StepRunner(model, tok0)
    runner.run(args.warmup)
    model.sync()
    runner = StepRunner(model, tok0)
    sampler = ClockSampler(gpu_id_for(torch, local))
    sampler.start()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    n0 = model.launch_count()
    e0.record(stream)
    runner.run(args.steps)
    e1.record(stream)
    launches = model.launch_count() - n0
    torch.cuda.synchronize()
    t_end = time.time()
    barrier()
    clocks = sampler.stop(t_begin, t_end)
    model.sync()
    ms = max_over_ranks(e0.elapsed_time(e1))
    value = job_throughput(args.steps, world, ms)

    # ---- end to end through gpt2_generate: host prompt in, host ids out ----
    passes_per_call = PROMPT_LEN + CYCLE
    e2e_calls = max(3, min(args.e2e_calls, 3000 // passes_per_call))
    model.generate(prompt, CYCLE)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_calls):
        model.generate(prompt, CYCLE)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    e2e = {"value": e2e_calls * passes_per_call * world / e2e_s, "unit": UNIT,
           "h2d_bytes_per_step": PROMPT_LEN * 4, "d2h_bytes_per_step": (CYCLE + 1) * 4,
           "step": f"one gpt2_generate call: {PROMPT_LEN}-id host prompt, {PROMPT_LEN} prompt passes "
                   f"+ {CYCLE} greedy passes, {CYCLE + 1} ids back to host; value counts passes",
           "calls": e2e_calls}

    # ---- tok/s against context length (long workloads): one cycle, an event
    # every SWEEP_BUCKET positions ----
    sweep = None
    if CYCLE >= 2 * SWEEP_BUCKET:
        peaks_s, _ = measured_peaks()
        marks = []
        torch.cuda.synchronize()
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        marks.append((PROMPT_LEN, ev))
        model.decode_step(tok0, PROMPT_LEN)
        pos = PROMPT_LEN + 1
        while pos < PROMPT_LEN + CYCLE:
            n = min(SWEEP_BUCKET - (pos - PROMPT_LEN) % SWEEP_BUCKET, PROMPT_LEN + CYCLE - pos)
            model.decode_greedy(n)
            pos += n
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks.append((pos, ev))
        torch.cuda.synchronize()
        sweep = []
        for (p0, e_a), (p1, e_b) in zip(marks, marks[1:]):
            t = e_a.elapsed_time(e_b) / 1e3 / (p1 - p0)
            b = roofline.mean_bytes_per_token(cfg, args.wdtype, range(p0, p1), args.head)
            sweep.append({"positions": f"{p0}..{p1 - 1}", "us_per_token": t * 1e6, "tok_s": 1.0 / t,
                          "gbs": b / t / 1e9, "frac": b / t / 1e9 / peaks_s["hbm_gbs"]})
    model.close()

    # ---- roofline of the decode pass --------------------------------------
    positions = [PROMPT_LEN + (k % CYCLE) for k in range(CYCLE)]
    alg = roofline.mean_bytes_per_token(cfg, args.wdtype, positions, args.head)
    peaks, peak_kind = measured_peaks()
    achieved = alg / (ms / 1e3 / args.steps) / 1e9
    traffic = load_traffic().get(path, {}).get(args.wdtype if args.head == "f32" else f"{args.wdtype}+f16 head")
    kernel = {
        "cluster": "k_decode_cluster: one cooperative launch per call (one per 60-step cycle here, "
                   "a host-fed pass + 59 device-fed passes), clusters of 4 CTAs, one CTA per SM",
        "persistent": "k_decode_persistent: one cooperative launch per call (one per 60-step cycle here, "
                      "a host-fed pass + 59 device-fed passes), one CTA per SM",
    }.get(path, f"decode pass: one CUDA graph of {kps} kernels (PDL-chained)")
    roof = {"bound": "hbm", "kernel": kernel,
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_kind": f"{peak_kind} copy bandwidth",
            "traffic": traffic, "algorithmic_bytes_per_launch": alg}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if args.wdtype == "f32" else
            f"{args.wdtype} weights, f32 math", "data": "synthetic",
            "config": dict(workload_config(args.wdtype, world, args.head), path=path), "e2e": e2e,
            "gpu_launches": launches,
            "roofline": roof, "clocks": clocks}
    if sweep is not None:
        line["context_sweep"] = sweep

    # ---- CPU baseline: the oracle on this host (rank 0, N = 1) ---------------
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, el = oracle_sample(cfg, w, prompt, args.wdtype, args.cpu_seconds, head=args.head)
        line["cpu_baseline"] = {"value": n / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} greedy decode passes of the same workload (positions "
                                          f"{PROMPT_LEN}..{PROMPT_LEN + CYCLE - 1}) after an untimed "
                                          f"prefill, single-threaded C oracle, ~{args.cpu_seconds:.0f} s"}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
