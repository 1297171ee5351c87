"""Seeded synthetic inputs: GPT-2 shaped weights and prompt ids.

This module only draws random numbers into arrays of the right names and
shapes.  It holds none of the model's arithmetic, so that the CPU oracle and
the CUDA library can both be fed from it without sharing any of the method.

Recipe (the same for every configuration):
  * matrices, wte and wpe ~ N(0, 0.02^2);
  * LayerNorm gamma = 1 + N(0, 0.01^2), beta ~ N(0, 0.01^2);
  * biases ~ N(0, 0.01^2);
  * prompt ids uniform in [0, vocab).
Weights come from one numpy PCG64 stream (seed 0 by default) drawn in a fixed
order; prompts from a separate stream (seed 1 by default).  PCG64 and numpy's
normal sampler give the same numbers on x86-64 and AArch64.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class GPT2Config:
    n_layer: int
    n_embd: int
    n_head: int
    n_positions: int
    vocab_size: int
    ln_eps: float = 1e-5

    @property
    def head_dim(self) -> int:
        return self.n_embd // self.n_head

    @property
    def n_mlp(self) -> int:
        return 4 * self.n_embd


# 2 layers, E=128, 4 heads of 32, mlp 512, vocab 512, 64 positions.
TINY = GPT2Config(n_layer=2, n_embd=128, n_head=4, n_positions=64, vocab_size=512)
# GPT-2 small (124M): 12 layers, E=768, 12 heads of 64, vocab 50257, 1024 positions.
SMALL = GPT2Config(n_layer=12, n_embd=768, n_head=12, n_positions=1024, vocab_size=50257)

LAYER_KEYS = ("ln1_w", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
              "ln2_w", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


def layer_shapes(cfg: GPT2Config) -> dict:
    """Checkpoint (HF Conv1D) shapes: matrices are [input][output]."""
    E, F = cfg.n_embd, cfg.n_mlp
    return {"ln1_w": (E,), "ln1_b": (E,), "attn_w": (E, 3 * E), "attn_b": (3 * E,),
            "proj_w": (E, E), "proj_b": (E,), "ln2_w": (E,), "ln2_b": (E,),
            "fc_w": (E, F), "fc_b": (F,), "mlp_proj_w": (F, E), "mlp_proj_b": (E,)}


def _normal(rng, shape, std, mean=0.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    if mean:
        a += np.float32(mean)
    return a


def make_weights(cfg: GPT2Config, seed: int = 0) -> dict:
    rng = np.random.Generator(np.random.PCG64(seed))
    E, V, P = cfg.n_embd, cfg.vocab_size, cfg.n_positions
    w = {"wte": _normal(rng, (V, E), 0.02), "wpe": _normal(rng, (P, E), 0.02)}
    layers = []
    for _ in range(cfg.n_layer):
        L = {}
        for k, shape in layer_shapes(cfg).items():
            if k.startswith("ln") and k.endswith("_w"):
                L[k] = _normal(rng, shape, 0.01, mean=1.0)
            elif k.endswith("_w"):
                L[k] = _normal(rng, shape, 0.02)
            else:                       # LayerNorm beta and linear biases
                L[k] = _normal(rng, shape, 0.01)
        layers.append(L)
    w["layers"] = layers
    w["ln_f_w"] = _normal(rng, (E,), 0.01, mean=1.0)
    w["ln_f_b"] = _normal(rng, (E,), 0.01)
    return w


# Stress inputs: the recipe's weights with a shifted distribution, to reach
# parts of a decode path that N(0, 0.02) weights never exercise.
#   "offset":   wpe + 30 in every dimension: the residual stream carries a
#               common offset of 30 through every block, so |mean(x)| is
#               about a thousand times std(x) at the first LayerNorm;
#   "outliers": three dimensions get +400 in every MLP output bias, so those
#               residual values grow into the thousands (one block adds 400);
#   "overflow": wpe + 1e5 in every dimension (residual values of 1e5).
STRESS_KINDS = ("offset", "outliers", "overflow")


def make_stress_weights(cfg: GPT2Config, kind: str, seed: int = 0) -> dict:
    if kind not in STRESS_KINDS:
        raise ValueError(f"unknown stress kind {kind!r}")
    w = make_weights(cfg, seed)
    if kind == "offset":
        w["wpe"] = w["wpe"] + np.float32(30.0)
    elif kind == "overflow":
        w["wpe"] = w["wpe"] + np.float32(1e5)
    else:
        dims = [1, cfg.n_embd // 2 + 3, cfg.n_embd - 5]
        for L in w["layers"]:
            b = L["mlp_proj_b"].copy()
            b[dims] += np.float32(400.0)
            L["mlp_proj_b"] = b
    return w


def make_prompt(cfg: GPT2Config, n: int, seed: int = 1) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, cfg.vocab_size, size=n, dtype=np.int64).astype(np.int32)


def make_batch_prompts(cfg: GPT2Config, n_seq: int, lo: int, hi: int, seed: int = 2):
    """Ragged prompts for the batched workload: lengths uniform in [lo, hi]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lo, hi + 1, size=n_seq)
    return [rng.integers(0, cfg.vocab_size, size=int(n), dtype=np.int64).astype(np.int32)
            for n in lens]
