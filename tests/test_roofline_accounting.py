"""The byte / multiply-add accounting behind the roofline, pinned to the
sizes the pages print for GPT-2 small."""
import json
import os

import pytest

from transformer_decode_token_gb300 import roofline, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_sizes.json")


def computed(name, cfg=synth.SMALL):
    E, L, P, V = cfg.n_embd, cfg.n_layer, cfg.n_positions, cfg.vocab_size
    if name == "kv_cache_bytes":
        return L * P * E * 2 * 4
    if name == "block_matrix_bytes_f32":
        return roofline.block_matrix_bytes(cfg, "f32")
    if name == "head_padded_bytes":
        return ((V + 63) // 64 * 64) * E * 4
    if name == "weight_bytes_f32":
        return roofline.parameter_count(cfg) * 4
    if name == "macs_per_token":
        return roofline.macs_per_token(cfg)
    raise KeyError(name)


@pytest.mark.parametrize("fig", json.load(open(GOLDEN))["figures"], ids=lambda f: f["name"])
def test_page_figure(fig):
    v = computed(fig["name"])
    if "value_mb" in fig:
        assert abs(v / 1e6 - fig["value_mb"]) <= fig["rel_tol"] * fig["value_mb"]
    else:
        assert abs(v / 1e6 - fig["value_m"]) <= fig["rel_tol"] * fig["value_m"]


def test_bytes_per_token_components():
    cfg = synth.SMALL
    b = roofline.bytes_per_token(cfg, "f32", 0)
    assert b["block_matrices"] == 339_738_624
    assert b["head"] == 154_389_504
    assert b["kv"] == 73_728 * 2
    i4 = roofline.bytes_per_token(cfg, "int4", 0)
    assert i4["block_matrices"] == 42_467_328 + 10_616_832 + 1_327_104
    f16 = roofline.bytes_per_token(cfg, "f16", 0)
    assert f16["block_matrices"] == 339_738_624 // 2
    assert roofline.bytes_per_token(cfg, "f32", 1023)["kv"] == 12 * 1025 * 2 * 768 * 4
    with pytest.raises(ValueError):
        roofline.block_matrix_bytes(cfg, "int8")


def test_stored_head_bytes():
    """The LM head's bytes with a separately stored head: fp16 is half of the
    fp32 tied head; int4 is codes (half a byte per weight) + one fp32 scale per
    32 weights + one 4-bit zero point per 32 weights, as for the block
    matrices; the rest of the pass does not change."""
    cfg = synth.SMALL
    n = cfg.vocab_size * cfg.n_embd
    f32 = roofline.bytes_per_token(cfg, "int4", 10)
    f16 = roofline.bytes_per_token(cfg, "int4", 10, head="f16")
    i4 = roofline.bytes_per_token(cfg, "int4", 10, head="int4")
    assert f16["head"] * 2 == f32["head"] == 4 * n
    assert i4["head"] == n // 2 + (n // 32) * 4 + n // 64
    for k in ("block_matrices", "biases_ln", "embedding_rows", "logits", "kv"):
        assert f32[k] == f16[k] == i4[k]
    assert roofline.mean_bytes_per_token(cfg, "f32", [10, 11], head="f16") == pytest.approx(
        (roofline.bytes_per_token(cfg, "f32", 10, "f16")["total"] + roofline.bytes_per_token(cfg, "f32", 11, "f16")["total"]) / 2)


def test_batched_step_bytes():
    """One batched step streams every stored weight once for the whole batch
    (bf16: half the fp32 block bytes the pages print, and a bf16 head of half
    the tied head), and per sequence its own embedding rows, logits row and
    KV rows; a batch of one is a single-sequence pass with those weights."""
    cfg = synth.SMALL
    one = roofline.batched_bytes_per_step(cfg, [37])
    assert one["block_matrices"] == 339_738_624 // 2
    assert one["head"] == 154_389_504 // 2
    single = roofline.bytes_per_token(cfg, "bf16", 37)
    for k in ("block_matrices", "biases_ln", "embedding_rows", "logits", "kv"):
        assert one[k] == single[k]
    pos = [40, 300, 511]
    many = roofline.batched_bytes_per_step(cfg, pos)
    assert many["block_matrices"] == one["block_matrices"] and many["head"] == one["head"]
    assert many["kv"] == sum(roofline.bytes_per_token(cfg, "f32", p)["kv"] for p in pos)
    assert many["logits"] == 3 * cfg.vocab_size * 4
    assert roofline.batched_flops_per_step(cfg, 64) == 2 * 64 * roofline.macs_per_token(cfg)
    # a bf16 cache: the pages' fp32 KV bytes (the 75.5 MB cache at 1024 rows) halved, the rest unchanged
    half = roofline.batched_bytes_per_step(cfg, pos, kv="bf16")
    assert 2 * half["kv"] == many["kv"]
    assert all(half[k] == many[k] for k in ("block_matrices", "head", "biases_ln", "embedding_rows", "logits"))
    assert roofline.batched_bytes_per_step(cfg, [1022], kv="bf16")["kv"] * 2 == 12 * 2 * 768 * 4 * 1024
