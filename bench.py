#!/usr/bin/env python
"""GPT-2 124M batch-1 greedy decode throughput on GB300.

Headline workload: GPT-2 small (12 layers, n_embd 768, 12 heads, vocab
50257, 1024 positions), fp32 weights drawn from N(0, 0.02) with seed 0, a
10-token prompt (seed 1) and 60 greedy decode steps at positions 10..69.  A
bench "step" is one decode pass over one token: embedding, 12 blocks, final
LayerNorm, tied head and argmax.  The timed region runs exactly --steps
passes; they cycle through the workload's generation (each cycle re-enters
its first position with the generation's first token, the rest are
device-fed greedy passes), so any step count keeps the workload's positions.

The same run also times the two other single-sequence configurations, each
over whole cycles of its own generation, and reports them under "variants":
int4 block matrices (10-token prompt + 128 steps) and fp16 block matrices
(16-token prompt decoded to the full 1024-position cache, 1008 steps, with
tok/s and GB/s per 64 positions in "context_sweep"), and the batched
configuration: 64 independent sequences with bf16 weights on the tensor
cores, prompts of 32..512 tokens prefilled untimed, then 64 device-fed
greedy steps of all 64 sequences (aggregate tok/s = 64 x steps / time),
with an fp32 and with a bf16 KV cache.
--wdtype picks one of the other configurations as the headline instead
(then no variants): f16, int4, or bf16 for the batched one.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--wdtype f32|f16|int4|bf16] [--kv f32|bf16]
  python bench.py --impl reference ...     # the CPU oracle, same metric

Prints one JSON line on rank 0.  N > 1 runs N independent replicas (one
process per GPU, launched by torchrun); the value is the total over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
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
SWEEP_BUCKET = 64
# The batched configuration: 64 independent sequences, bf16 weights, prompts
# of uniform length in [32, 512] (seed 2), 64 greedy steps per sequence.
BATCH, BATCH_PROMPT, BATCH_STEPS = 64, (32, 512), 64
CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


def parse(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=120)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--wdtype", choices=["f32", "f16", "int4", "bf16"], default="f32",
                   help="the headline configuration; bf16 = the batched one (64 sequences, tensor cores)")
    p.add_argument("--head", choices=["f32", "f16", "int4"], default="f32",
                   help="LM head storage: the tied fp32 wte (the configurations), an fp16 copy (README -h) or int4")
    p.add_argument("--kv", choices=["f32", "bf16"], default="f32",
                   help="with --wdtype bf16: the KV cache's element type")
    p.add_argument("--no-variants", action="store_true",
                   help="time only the headline workload (not the int4 and fp16 configurations)")
    p.add_argument("--e2e-calls", type=int, default=50)
    p.add_argument("--cpu-seconds", type=float, default=8.0,
                   help="CPU time budget of each leg of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", choices=["auto", "per_kernel"], default="auto",
                   help="auto: the cluster decode kernel where the device allows it")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def workload_config(wdtype: str, world: int, head: str = "f32") -> dict:
    n_prompt, cycle = WORKLOADS[wdtype]
    return {"workload": f"GPT-2 small 124M, {wdtype} block weights, {head} LM head, batch 1, {n_prompt}-token prompt "
                        f"+ {cycle} greedy decode steps (positions {n_prompt}..{n_prompt + cycle - 1}), "
                        "cycled",
            "n_layer": 12, "n_embd": 768, "n_head": 12, "vocab": 50257, "n_positions": 1024,
            "batch": 1, "weights": "synthetic N(0,0.02), seed 0; prompt ids uniform, seed 1",
            "l2": "no flush: every step streams all weights (f32 494.6 MB, f16 324.7 MB, int4 209.3 MB) "
                  "through a 129 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def timed_positions(wdtype: str, steps: int) -> list:
    """Positions of the passes a timed region of `steps` passes runs."""
    n_prompt, cycle = WORKLOADS[wdtype]
    return [n_prompt + (k % cycle) for k in range(steps)]


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


SOURCES = {"cluster": ("cluster.cu", "cluster.h", "common.cuh"),
           "batched": ("batch.cu", "batch.h", "tc_gemm.cu", "tc_gemm.h", "common.cuh")}


def kernel_source_sha(path: str = "cluster") -> str:
    """sha256 prefix of a decode path's kernel sources: a traffic figure taken
    on other sources no longer describes the kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_decode_token_gb300", "csrc")
    for name in SOURCES[path]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(path: str, key: str, alg=None):
    """DRAM bytes per decode pass (batched: per step) from the committed ncu
    summaries (profiles/traffic.json: {path: {key: {"bytes": B, "sources":
    sha}}}), or None if there is none for the current kernel sources.  An
    entry captured on a step with other positions ("algorithmic": its
    algorithmic bytes) is scaled to `alg` by the algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f).get(path, {}).get(key)
    except OSError:
        return None
    if not isinstance(t, dict) or t.get("sources") != kernel_source_sha(path if path in SOURCES else "cluster"):
        return None
    if alg is not None and t.get("algorithmic"):
        return t["bytes"] * alg / t["algorithmic"]
    return t.get("bytes")


# ---- CPU oracle timing -------------------------------------------------------

def oracle_sample(cfg, weights, prompt, wdtype, budget_s, max_steps=None, head="f32", omp=False, kv="f32"):
    """Decode passes of the oracle after an untimed prefill, at the
    workload's positions; stops after ~budget_s seconds (or max_steps).
    bf16 (the batched configuration): one of its sequences, the given prompt
    followed by its greedy steps, with the weights and head that
    configuration stores.  Returns (passes, seconds)."""
    from oracle import oracle as orc
    if wdtype == "bf16":
        n_prompt, cycle, head = len(prompt), BATCH_STEPS, "bf16"
    else:
        n_prompt, cycle = WORKLOADS[wdtype]
    sw = orc.stored_weights(weights, wdtype, head=head)
    m = orc.OracleModel(cfg, sw, omp=omp, kv=kv)
    try:
        tok = None
        for pos, t in enumerate(prompt):
            _, tok = m.forward(int(t), pos)
        n, pos = 0, len(prompt)
        t0 = time.perf_counter()
        while True:
            if pos >= n_prompt + cycle:           # keep the workload's positions
                pos = n_prompt
            _, tok = m.forward(tok, pos)
            pos += 1
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s or (max_steps is not None and n >= max_steps):
                return n, el
    finally:
        m.close()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from transformer_decode_token_gb300 import synth
    cfg = synth.SMALL
    w = synth.make_weights(cfg, 0)
    if args.wdtype == "bf16":   # one sequence of the batched workload (the oracle runs one at a time)
        prompt = min(synth.make_batch_prompts(cfg, BATCH, *BATCH_PROMPT, seed=2), key=len)
        config = {"workload": f"GPT-2 small 124M, batched configuration ({BATCH} sequences, bf16 block weights "
                              f"and head, prompts of {BATCH_PROMPT[0]}..{BATCH_PROMPT[1]} tokens, {BATCH_STEPS} "
                              "greedy steps); the oracle decodes its shortest sequence",
                  "batch": BATCH, "weights": "synthetic N(0,0.02), seed 0"}
    else:
        prompt = synth.make_prompt(cfg, WORKLOADS[args.wdtype][0], 1)
        config = workload_config(args.wdtype, 1, args.head)
    cores = host_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    kv = args.kv if args.wdtype == "bf16" else "f32"
    oracle_sample(cfg, w, prompt, args.wdtype, 1e9, max_steps=min(args.warmup, 3), head=args.head, omp=True, kv=kv)
    n, el = oracle_sample(cfg, w, prompt, args.wdtype, 60.0, max_steps=args.steps, head=args.head, omp=True, kv=kv)
    value = n / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if args.wdtype == "f32" else f"{args.wdtype} weights, f32 math",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(os.environ["OMP_NUM_THREADS"]),
                             "kind": "oracle",
                             "sample": f"{n} of the {args.steps} requested decode passes (60 s cap), the C oracle's "
                                       "OpenMP build (each matrix product's outputs split between the threads), "
                                       "after an untimed prefill"},
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
    """Queues decode passes that cycle through a workload's generation: a
    host-fed pass at the first generated position, then device-fed greedy
    passes up to the cycle's end."""

    def __init__(self, model, first_token: int, n_prompt: int, cycle: int):
        self.m = model
        self.tok0 = first_token
        self.n_prompt = n_prompt
        self.cycle = cycle
        self.k = 0
        self.host_steps = 0

    def run(self, n: int):
        while n > 0:
            if self.k % self.cycle == 0:
                self.m.decode_step(self.tok0, self.n_prompt)
                self.host_steps += 1
                self.k += 1
                n -= 1
            else:
                c = min(n, self.cycle - self.k % self.cycle)
                self.m.decode_greedy(c)
                self.k += c
                n -= c


KERNEL_DESC = {
    "cluster": "k_decode_cluster: one cooperative launch per call (a host-fed pass, then one launch of the "
               "cycle's remaining device-fed passes), clusters of 4 CTAs, one CTA per SM",
}


def measure(torch, cfg, w, wdtype, head, path, steps, warmup, world, local, barrier, max_over_ranks,
            sweep=False, e2e_calls=0):
    """Times `steps` decode passes of one workload on a fresh model; returns
    the workload's fields of the JSON line."""
    from transformer_decode_token_gb300 import binding, roofline, synth
    n_prompt, cycle = WORKLOADS[wdtype]
    prompt = synth.make_prompt(cfg, n_prompt, 1)
    dw = binding.upload_weights(w)
    model = binding.Model(cfg, dw, wdtype, path=path, head=head)
    del dw
    torch.cuda.empty_cache()
    out = {}
    try:
        kps = model.kernels_per_step()
        path_used = model.path()
        model.prefill(prompt)
        tok0 = model.argmax()
        runner = StepRunner(model, tok0, n_prompt, cycle)
        runner.run(warmup)
        model.sync()
        runner = StepRunner(model, tok0, n_prompt, cycle)
        sampler = ClockSampler(gpu_id_for(torch, local))
        sampler.start()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t_begin = time.time()
        n0 = model.launch_count()
        e0.record(stream)
        runner.run(steps)
        e1.record(stream)
        launches = model.launch_count() - n0
        torch.cuda.synchronize()
        t_end = time.time()
        barrier()
        clocks = sampler.stop(t_begin, t_end)
        model.sync()
        ms = max_over_ranks(e0.elapsed_time(e1))
        out["value"] = job_throughput(steps, world, ms)
        out["ms_per_step"] = ms / steps
        out["steps"] = steps
        out["gpu_launches"] = launches
        out["clocks"] = clocks
        out["path"] = path_used

        if e2e_calls:
            # end to end through gpt2_generate: host prompt in, host ids out
            model.generate(prompt, cycle)
            barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(e2e_calls):
                model.generate(prompt, cycle)
            torch.cuda.synchronize()
            e2e_s = max_over_ranks(time.perf_counter() - t0)
            out["e2e"] = {"value": e2e_calls * (n_prompt + cycle) * world / e2e_s, "unit": UNIT,
                          "h2d_bytes_per_step": n_prompt * 4, "d2h_bytes_per_step": (cycle + 1) * 4,
                          "generated_tok_s": e2e_calls * (cycle + 1) * world / e2e_s,
                          "step": f"one gpt2_generate call: {n_prompt}-id host prompt in, {n_prompt} prompt passes "
                                  f"+ {cycle} greedy passes, {cycle + 1} ids back to host; value counts passes "
                                  "(prompt and greedy), generated_tok_s counts the ids returned",
                          "calls": e2e_calls}

        if sweep and cycle >= 2 * SWEEP_BUCKET:
            # tok/s against context length: one cycle, an event every SWEEP_BUCKET positions
            peaks_s, _ = measured_peaks()
            marks = []
            torch.cuda.synchronize()
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks.append((n_prompt, ev))
            model.decode_step(tok0, n_prompt)
            pos = n_prompt + 1
            while pos < n_prompt + cycle:
                n = min(SWEEP_BUCKET - (pos - n_prompt) % SWEEP_BUCKET, n_prompt + cycle - pos)
                model.decode_greedy(n)
                pos += n
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(stream)
                marks.append((pos, ev))
            torch.cuda.synchronize()
            rows = []
            for (p0, e_a), (p1, e_b) in zip(marks, marks[1:]):
                t = e_a.elapsed_time(e_b) / 1e3 / (p1 - p0)
                b = roofline.mean_bytes_per_token(cfg, wdtype, range(p0, p1), head)
                rows.append({"positions": f"{p0}..{p1 - 1}", "us_per_token": t * 1e6, "tok_s": 1.0 / t,
                             "gbs": b / t / 1e9, "frac": b / t / 1e9 / peaks_s["hbm_gbs"]})
            out["context_sweep"] = rows
    finally:
        model.close()

    # roofline of the decode pass over the positions the timed region ran
    positions = timed_positions(wdtype, steps)
    alg = roofline.mean_bytes_per_token(cfg, wdtype, positions, head)
    peaks, peak_kind = measured_peaks()
    achieved = alg / (out["ms_per_step"] / 1e3) / 1e9
    key = wdtype if head == "f32" else f"{wdtype}+{head} head"
    out["roofline"] = {
        "bound": "hbm",
        "kernel": KERNEL_DESC.get(path_used, f"decode pass: one CUDA graph of {kps} kernels (PDL-chained)"),
        "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": achieved / peaks["hbm_gbs"], "peak_kind": f"{peak_kind} copy bandwidth",
        "traffic": load_traffic(path_used, key),
        "algorithmic_bytes_per_launch": alg,
        "positions": f"{min(positions)}..{max(positions)} ({len(positions)} passes)"}
    return out


def measure_batch(torch, cfg, w, steps, warmup, world, local, barrier, max_over_ranks, e2e_calls=0,
                  exact=False, kv="f32"):
    """The batched configuration on a fresh batched model: an untimed prefill
    of the 64 ragged prompts, then 64 device-resident greedy steps timed;
    repeated (each after a fresh prefill) until `steps` steps are timed,
    rounded up to whole cycles unless `exact`.
    With e2e_calls > 0, also that many whole generations through the ABI
    with host buffers (prompts in, every generated id out), wall clock.
    kv: the cache's element type ("bf16": GPT2_BATCH_KV_BF16)."""
    from transformer_decode_token_gb300 import binding, roofline, synth
    prompts = synth.make_batch_prompts(cfg, BATCH, *BATCH_PROMPT, seed=2)
    lens = [len(q) for q in prompts]
    dw = binding.upload_weights(w)
    m = binding.BatchModel(cfg, dw, BATCH, kv=kv)
    del dw
    torch.cuda.empty_cache()
    try:
        kps, _ = m.info()
        m.prefill(prompts)
        m.decode_greedy(min(warmup, BATCH_STEPS))
        m.sync()
        # whole cycles of the generation, or exactly `steps` steps (the last
        # cycle cut short) when this is the line's own workload
        n_total = steps if exact else BATCH_STEPS * max(1, -(-steps // BATCH_STEPS))
        cycles = [min(BATCH_STEPS, n_total - i) for i in range(0, n_total, BATCH_STEPS)]
        stream = torch.cuda.current_stream()
        ms = 0.0
        launches = 0
        sampler = ClockSampler(gpu_id_for(torch, local))
        sampler.start()
        t_begin = time.time()
        for i, n_cyc in enumerate(cycles):
            m.prefill(prompts)
            m.sync()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize()
            if i == 0:   # the first cycle's steps are what `ncu --profile-from-start off` captures
                torch.cuda.profiler.start()
            n0 = m.info()[1]
            e0.record(stream)
            m.decode_greedy(n_cyc)
            e1.record(stream)
            launches += m.info()[1] - n0
            torch.cuda.synchronize()
            if i == 0:
                torch.cuda.profiler.stop()
            ms += e0.elapsed_time(e1)
        t_end = time.time()
        clocks = sampler.stop(t_begin, t_end)
        m.sync()
        e2e = None
        if e2e_calls > 0:
            p0, p1 = min(lens), max(lens) + BATCH_STEPS
            barrier()
            t0 = time.perf_counter()
            for _ in range(e2e_calls):
                m.prefill(prompts)
                m.decode_greedy(BATCH_STEPS)
                ids = m.ids(p0, p1 - p0)
            el = max_over_ranks(time.perf_counter() - t0)
            e2e = {"value": BATCH * BATCH_STEPS * e2e_calls * world / el, "unit": UNIT,
                   "h2d_bytes_per_step": (sum(lens) + BATCH) * 4 / BATCH_STEPS,
                   "d2h_bytes_per_step": ids.nbytes / BATCH_STEPS,
                   "calls": e2e_calls,
                   "what": f"gpt2_prefill_batch (host prompts) + gpt2_decode_batch_greedy({BATCH_STEPS}) + "
                           "gpt2_batch_ids (host ids) per call, wall clock, prefill included; value = generated "
                           "tokens / time"}
    finally:
        m.close()
    ms = max_over_ranks(ms)
    n_steps = sum(cycles)
    # bytes and flops of the timed steps: step t of a cycle runs every sequence at lens + t
    per_t = [roofline.batched_bytes_per_step(cfg, [L + t for L in lens], kv=kv)["total"] for t in range(BATCH_STEPS)]
    alg = sum(sum(per_t[:n]) for n in cycles) / n_steps
    flops = roofline.batched_flops_per_step(cfg, BATCH)
    peaks, peak_kind = measured_peaks()
    step_s = ms / 1e3 / n_steps
    achieved = alg / step_s / 1e9
    out = {
        "value": BATCH * world / step_s, "unit": UNIT, "ms_per_step": ms / n_steps, "steps": n_steps,
        "gpu_launches": launches, "clocks": clocks,
        "dtype": "bf16 weights" + (", bf16 KV cache" if kv == "bf16" else "") + ", f32 math (bf16 x bf16 "
                 "tensor-core products of hi/lo activation parts, fp32 sums)",
        "config": {"workload": f"GPT-2 small 124M, batched: {BATCH} sequences, bf16 block weights and head, "
                               f"{'bf16' if kv == 'bf16' else 'fp32'} KV cache, "
                               f"prompts uniform in [{BATCH_PROMPT[0]}, {BATCH_PROMPT[1]}] tokens (seed 2), "
                               f"{BATCH_STEPS} greedy decode steps per sequence (prefill untimed)",
                   "batch": BATCH, "prompt_tokens": sum(lens), "weights": "synthetic N(0,0.02), seed 0",
                   "l2": "no flush: every step streams 247 MB of bf16 weights and ~1.4 GB of KV rows through a "
                         "129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": f"one batched step: a CUDA graph of {kps} kernels (tcgen05 linears, "
                                               "ragged attention, LayerNorm/gelu/argmax), PDL-chained",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": load_traffic("batched", kv, alg), "algorithmic_bytes_per_launch": alg,
                     "tensor_tflops": flops / step_s / 1e12,
                     "tensor_frac": flops / step_s / 1e12 / peaks.get("bf16_tflops", 1900.0),
                     "note": f"bytes: weights once per step + each sequence's KV rows 0..p ({kv}), embedding and "
                             "logits rows; flops: 2 x 64 x the linears' and head's multiply-adds (the hi/lo parts "
                             "double the tensor work actually issued)"},
    }
    if e2e is not None:
        out["e2e"] = e2e
    return out


def measure_prefill(torch, cfg, w, lengths=(2, 4, 8, 10, 16, 64), reps=10):
    """gpt2_prefill of prompts of several lengths (fp32 weights), on the tensor
    cores (the default on the cluster path) and as single-token passes of the
    cluster kernel (one launch of n passes): device time per call."""
    from transformer_decode_token_gb300 import binding, synth
    out = {}
    stream = torch.cuda.current_stream()
    dw = binding.upload_weights(w)
    for name, tc in (("tensor_cores", True), ("single_token_passes", False)):
        m = binding.Model(cfg, dw, "f32", tc_prefill=tc)
        try:
            row = {}
            for n in lengths:
                prompt = synth.make_prompt(cfg, n, 1)
                m.prefill(prompt)
                m.sync()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    m.prefill(prompt)
                e1.record(stream)
                torch.cuda.synchronize()
                m.sync()
                row[str(n)] = e0.elapsed_time(e1) / reps
            out[name] = row
        finally:
            m.close()
    del dw
    torch.cuda.empty_cache()
    out["unit"] = "ms per gpt2_prefill call"
    out["note"] = ("tensor cores: the prompt's positions as the rows of one batched step (up to 64 per step); "
                   "single-token passes: one cluster-kernel launch running n passes")
    return out


def batch_main(args, torch, dist, cfg, w, rank, world, local, barrier, max_over_ranks):
    """--wdtype bf16: the batched configuration as the line's own workload
    (exactly --steps timed steps)."""
    from transformer_decode_token_gb300 import synth
    b = measure_batch(torch, cfg, w, args.steps, args.warmup, world, local, barrier, max_over_ranks,
                      e2e_calls=max(1, min(args.e2e_calls, 5)), exact=True, kv=args.kv)
    line = {"metric": METRIC, "value": b["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": b["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": b["dtype"], "data": "synthetic",
            "config": b["config"], "path": "batched (tcgen05)", "e2e": b["e2e"],
            "gpu_launches": b["gpu_launches"], "roofline": b["roofline"], "clocks": b["clocks"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        prompts = synth.make_batch_prompts(cfg, BATCH, *BATCH_PROMPT, seed=2)
        prompt = min(prompts, key=len)
        cores = host_cores()
        os.environ.setdefault("OMP_NUM_THREADS", str(cores))
        n, el = oracle_sample(cfg, w, prompt, "bf16", args.cpu_seconds, omp=True, kv=args.kv)
        line["cpu_baseline"] = {
            "value": n / el, "unit": UNIT, "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
            "sample": f"{n} greedy decode passes of the batched workload's shortest sequence ({len(prompt)}-token "
                      f"prompt, untimed prefill), bf16-stored weights and head, the C oracle's OpenMP build; "
                      f"the oracle runs one sequence at a time, ~{args.cpu_seconds:.0f} s"}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist
    from transformer_decode_token_gb300 import synth

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
    if args.wdtype == "bf16":
        return batch_main(args, torch, dist, cfg, w, rank, world, local, barrier, max_over_ranks)
    head = measure(torch, cfg, w, args.wdtype, args.head, args.path, args.steps, args.warmup, world, local,
                   barrier, max_over_ranks, sweep=True, e2e_calls=max(3, min(args.e2e_calls, 3000 // sum(
                       WORKLOADS[args.wdtype]))))
    n_prompt, cycle = WORKLOADS[args.wdtype]
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if args.wdtype == "f32" else f"{args.wdtype} weights, f32 math", "data": "synthetic",
            "config": workload_config(args.wdtype, world, args.head), "path": head["path"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "roofline": head["roofline"], "clocks": head["clocks"]}
    if "context_sweep" in head:
        line["context_sweep"] = head["context_sweep"]

    # the other single-sequence configurations, each over whole cycles of its generation
    if not args.no_variants and args.wdtype == "f32" and args.head == "f32":
        variants = {}
        for wd in ("int4", "f16"):
            cyc = WORKLOADS[wd][1]
            steps = cyc * max(1, -(-args.steps // cyc))
            v = measure(torch, cfg, w, wd, "f32", args.path, steps, args.warmup, world, local, barrier,
                        max_over_ranks, sweep=(wd == "f16"))
            v["config"] = workload_config(wd, world)
            v["dtype"] = f"{wd} weights, f32 math"
            variants[wd] = v
        # (at most 10 cycles: each cycle re-runs the untimed prefill of all 64 prompts)
        for name, kv in (("batch64_bf16", "f32"), ("batch64_bf16_kvbf16", "bf16")):
            variants[name] = measure_batch(torch, cfg, w, min(args.steps, 10 * BATCH_STEPS), args.warmup, world,
                                           local, barrier, max_over_ranks, kv=kv)
        line["variants"] = variants
        line["prefill"] = measure_prefill(torch, cfg, w)

    # ---- CPU baseline: the oracle on this host (rank 0, N = 1) ---------------
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        prompt = synth.make_prompt(cfg, n_prompt, 1)
        cores = host_cores()
        os.environ.setdefault("OMP_NUM_THREADS", str(cores))
        n1, el1 = oracle_sample(cfg, w, prompt, args.wdtype, args.cpu_seconds, head=args.head)
        nm, elm = oracle_sample(cfg, w, prompt, args.wdtype, args.cpu_seconds, head=args.head, omp=True)
        line["cpu_baseline"] = {
            "value": nm / elm, "unit": UNIT, "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
            "sample": f"{nm} greedy decode passes of the same workload (positions {n_prompt}..{n_prompt + cycle - 1}) "
                      f"after an untimed prefill, the C oracle's OpenMP build (each matrix product's outputs "
                      f"split between the threads), ~{args.cpu_seconds:.0f} s",
            "single_thread": {"value": n1 / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} passes of the same workload, single-threaded build, "
                                        f"~{args.cpu_seconds:.0f} s"}}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
