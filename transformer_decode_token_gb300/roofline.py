"""Algorithmic bytes and multiply-adds of one decode pass.

"Algorithmic" means what the pass must move at least once: every stored
weight it multiplies, one row each of wte and wpe for the embedding, the
biases and LayerNorm parameters, the KV cache rows it reads and the row it
writes, and the logits it writes.  Activations (a few KB, cache-resident)
are not counted.  Pinned to the sizes the pages print by
tests/test_roofline_accounting.py.
"""
from __future__ import annotations


def block_params(cfg) -> int:
    """Weights of the 4 block matrices of all layers: 12 E^2 per layer."""
    E = cfg.n_embd
    return cfg.n_layer * (3 * E * E + E * E + 4 * E * E + 4 * E * E)


def block_matrix_bytes(cfg, wdtype: str) -> int:
    n = block_params(cfg)
    if wdtype == "f32":
        return 4 * n
    if wdtype in ("f16", "bf16"):
        return 2 * n
    if wdtype == "int4":
        return n // 2 + (n // 32) * 4 + n // 64     # codes + fp32 scales + 4-bit zero points
    raise ValueError(wdtype)


def bytes_per_token(cfg, wdtype: str, pos: int, head: str = "f32") -> dict:
    """Bytes one decode pass at position `pos` must move (head: the LM head's
    storage, the fp32 tied wte or its fp16 copy)."""
    E, V, L = cfg.n_embd, cfg.vocab_size, cfg.n_layer
    parts = {
        "block_matrices": block_matrix_bytes(cfg, wdtype),
        "head": (V * E // 2 + (V * E // 32) * 4 + V * E // 64) if head == "int4" else V * E * (2 if head == "f16" else 4),
        "biases_ln": L * 13 * E * 4 + 2 * E * 4,         # 9E bias + 4E LN per layer, ln_f
        "embedding_rows": 2 * E * 4,                     # wte[token], wpe[pos]
        "logits": V * 4,
        "kv": L * 2 * E * 4 * (pos + 2),                 # read rows 0..pos, write row pos
    }
    parts["total"] = sum(parts.values())
    return parts


def batched_bytes_per_step(cfg, positions, wdtype: str = "bf16", head: str = "bf16", kv: str = "f32") -> dict:
    """Bytes one step of the batched path must move: every stored weight once
    for the whole batch (block matrices and head), the small fp32 parameters,
    and per sequence at position p its embedding rows, its logits row and
    its KV rows (read 0..p, write p; fp32 or bf16 elements)."""
    E, V, L = cfg.n_embd, cfg.vocab_size, cfg.n_layer
    positions = list(positions)
    n = len(positions)
    head_bytes = V * E * {"f32": 4, "f16": 2, "bf16": 2}[head]
    parts = {
        "block_matrices": block_matrix_bytes(cfg, wdtype),
        "head": head_bytes,
        "biases_ln": L * 13 * E * 4 + 2 * E * 4,
        "embedding_rows": n * 2 * E * 4,
        "logits": n * V * 4,
        "kv": sum(L * 2 * E * {"f32": 4, "bf16": 2}[kv] * (p + 2) for p in positions),
    }
    parts["total"] = sum(parts.values())
    return parts


def batched_flops_per_step(cfg, n_seq: int) -> int:
    """Multiply-adds x 2 of the linears and the head for n_seq sequences."""
    return 2 * n_seq * macs_per_token(cfg)


def mean_bytes_per_token(cfg, wdtype: str, positions, head: str = "f32") -> float:
    positions = list(positions)
    return sum(bytes_per_token(cfg, wdtype, p, head)["total"] for p in positions) / len(positions)


def macs_per_token(cfg) -> int:
    """Multiply-adds of the matrix products (block linears + tied head)."""
    return block_params(cfg) + cfg.vocab_size * cfg.n_embd


def parameter_count(cfg) -> int:
    E, V, P, L = cfg.n_embd, cfg.vocab_size, cfg.n_positions, cfg.n_layer
    return V * E + P * E + block_params(cfg) + L * 13 * E + 2 * E
