"""Phase timeline of the cluster decode kernel, from its own clock stamps.

Builds a variant of the library with -DGPT2_CTRACE (into _build_trace/), in
which thread 0 of every CTA records %globaltimer and clock64 at the phase
boundaries of two decode passes of one launch; runs GPT-2 small (synthetic
weights, 10-token prompt, then device-fed greedy passes) and prints, for the
head-cluster CTAs and the fc CTAs, the median over CTAs of each phase's
duration in a middle layer, and the LM-head phases.  Stamps cost ~100-200
cycles each, so the traced pass is somewhat slower than an untraced one.

  python -m transformer_decode_token_gb300.trace_cluster [--wdtype f32|f16|int4] [--json out.json]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os

import numpy as np

from . import build as _build

TRACE_DIR = os.path.join(_build.HERE, "_build_trace")
N_CTAS, N_PASSES, N_SLOTS = 160, 2, 208   # the stamp array of the trace build
# slots: layer l uses l * 16 + i; the LM head 200..206
HEAD_PHASES = [("wait for x (GPU-wide sum)", 0, 1), ("LN/bias parameters", 1, 2),
               ("QKV rows (LN folded)", 2, 3), ("q,k,v exchange in cluster", 3, 4),
               ("attention", 4, 5), ("out-proj tile", 5, 6), ("add into x_new", 6, 7)]
FC_PHASES = [("wait for x_new (GPU-wide sum)", 0, 1), ("LN/bias parameters", 1, 2),
             ("fc rows + gelu_new (LN folded)", 2, 3), ("mlp-proj tile", 4, 5),
             ("cluster reduce + add into x", 5, 6)]
# inside the dot-product phases (slot offsets 8..10: canonical rows, 11 and 13: tile rows)
HEAD_SUB = [("QKV: x*gamma to registers + LN stat shares", 2, 8), ("QKV: ring-stage waits", 8, 9),
            ("QKV: row groups (dot products, butterflies)", 9, 10), ("QKV: window barrier", 10, 3),
            ("out-proj: rows", 11, 13), ("out-proj: window barrier", 13, 6)]
FC_SUB = [("fc: x*gamma to registers + LN stat shares", 2, 8), ("fc: ring-stage waits", 8, 9),
          ("fc: row groups (dot products, gelu_new)", 9, 10), ("fc: window barrier", 10, 3),
          ("mlp-proj: rows", 11, 13), ("mlp-proj: window barrier", 13, 5)]
LM_PHASES = [("wait for x (GPU-wide sum)", 200, 201), ("LM-head rows + argmax keys", 201, 202),
             ("publish the tagged argmax key", 202, 203)]


def run(wdtype: str, layer: int = 5):
    lib = _build.build(force=True, extra=["-DGPT2_CTRACE"], lib=os.path.join(TRACE_DIR, "libgpt2_trace.so"),
                       objdir=TRACE_DIR)
    from . import binding, synth
    binding.load_library(lib)
    cfg = synth.SMALL
    w = synth.make_weights(cfg, 0)
    prompt = synth.make_prompt(cfg, 10, 1)
    m = binding.Model(cfg, binding.upload_weights(w), wdtype)
    if m.path() != "cluster":
        raise RuntimeError(f"the cluster kernel is not available here (path {m.path()})")
    m.prefill(prompt)
    m.argmax()
    m.decode_step(m.argmax(), 10)
    m.decode_greedy(40)      # passes 20 and 21 of this launch are stamped
    m.sync()
    L = binding.lib()
    arr = np.zeros((N_CTAS, N_PASSES, N_SLOTS, 6), np.uint64)
    rc = L.gpt2_debug_ctrace(arr.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(arr.nbytes))
    if rc != 0:
        raise RuntimeError(f"gpt2_debug_ctrace returned {rc}")
    m.close()
    a = arr.astype(np.int64)
    grid = int(np.count_nonzero(a[:, 0, 0, 0]))
    n_head = cfg.n_head * 4
    out = {"wdtype": wdtype, "layer": layer, "ctas": grid, "head_ctas": n_head}

    def med_us(rng, s0, s1, slot_base):
        t = np.array([a[c, 0, slot_base + s1, 0] - a[c, 0, slot_base + s0, 0] for c in rng], np.float64)
        return float(np.median(t)) / 1e3

    out["head_cluster_us"] = {n: med_us(range(n_head), s0, s1, layer * 16) for n, s0, s1 in HEAD_PHASES}
    out["fc_us"] = {n: med_us(range(n_head, grid), s0, s1, layer * 16) for n, s0, s1 in FC_PHASES}
    out["lm_head_us"] = {n: med_us(range(grid), s0, s1, 0) for n, s0, s1 in LM_PHASES}
    out["head_cluster_sub_us"] = {n: med_us(range(n_head), s0, s1, layer * 16) for n, s0, s1 in HEAD_SUB}
    out["fc_sub_us"] = {n: med_us(range(n_head, grid), s0, s1, layer * 16) for n, s0, s1 in FC_SUB}
    t0 = a[:grid, 0, 0, 0].min()
    out["pass_us"] = float(a[:grid, 0, 203, 0].max() - t0) / 1e3
    out["layer_us"] = float(np.median(a[:n_head, 0, (layer + 1) * 16 + 1, 0] - a[:n_head, 0, layer * 16 + 1, 0])) / 1e3
    return out


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--wdtype", choices=["f32", "f16", "int4"], default="f32")
    p.add_argument("--layer", type=int, default=5)
    p.add_argument("--json")
    a = p.parse_args()
    out = run(a.wdtype, a.layer)
    print(f"cluster kernel, GPT-2 small {out['wdtype']}, {out['ctas']} CTAs ({out['head_ctas']} in head clusters); "
          f"layer {out['layer']}: {out['layer_us']:.2f} us per layer (head-CTA x arrival to x arrival)")
    for grp in ("head_cluster_us", "fc_us", "lm_head_us", "head_cluster_sub_us", "fc_sub_us"):
        print(f"  {grp}:")
        for n, v in out[grp].items():
            print(f"    {n:46s} {v:7.2f} us")
    if a.json:
        with open(a.json, "w") as f:
            json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
