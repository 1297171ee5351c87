"""Pins for the oracle's whole decode pass.

* Against an independent float64 GPT-2 forward assembled from torch library
  routines (layer_norm, scaled_dot_product_attention with a causal mask, tanh
  gelu, matmul) on the checkpoint-layout weights.  A transposed operand, a
  swapped gamma/beta, a wrong q/k/v split or head order, a wrong attention
  scale or a missing residual all fail it.
* KV-cached decode equals whole-sequence recompute with a causal mask.
* Position handling: append-only, rewind, bad inputs.
"""
import numpy as np
import pytest
from oracle import oracle as orc
from ref64 import torch_gpt2_logits
from transformer_decode_token_gb300 import synth


# head_dim 32 (tiny) and head_dim 64 (the GPT-2 head, scale 1/8)
CFG64 = synth.GPT2Config(n_layer=3, n_embd=256, n_head=4, n_positions=48, vocab_size=700)


@pytest.mark.parametrize("cfg", [synth.TINY, CFG64], ids=["tiny", "d64"])
def test_decode_matches_library_float64_forward(cfg):
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 20, seed=1)
    ref = torch_gpt2_logits(cfg, w, toks)
    m = orc.OracleModel(cfg, w)
    for pos, t in enumerate(toks):
        logits, am = m.forward(int(t), pos)
        assert np.abs(logits - ref[pos]).max() <= 2e-5
        top2 = np.sort(ref[pos])[-2:]
        if top2[1] - top2[0] > 1e-3:
            assert am == int(np.argmax(ref[pos]))
    m.close()


def test_cached_decode_equals_full_recompute():
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=3)
    toks = synth.make_prompt(cfg, 24, seed=4)
    full = orc.forward_full(cfg, w, toks)
    m = orc.OracleModel(cfg, w)
    for pos, t in enumerate(toks):
        logits, _ = m.forward(int(t), pos)
        assert np.abs(logits - full[pos]).max() <= 1e-5
    m.close()


def test_full_recompute_matches_library():
    cfg = CFG64
    w = synth.make_weights(cfg, seed=5)
    toks = synth.make_prompt(cfg, 16, seed=6)
    assert np.abs(orc.forward_full(cfg, w, toks) - torch_gpt2_logits(cfg, w, toks)).max() <= 2e-5


def test_rewind_and_bad_positions():
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    m = orc.OracleModel(cfg, w)
    a = [m.forward(t, p)[0] for p, t in enumerate([5, 6, 7, 8])]
    # rewinding to position 2 and feeding the same token reproduces the row
    again, _ = m.forward(7, 2)
    assert np.array_equal(again, a[2])
    with pytest.raises(ValueError):
        m.forward(9, 4)          # only positions 0..3 are valid after the rewind
    with pytest.raises(ValueError):
        m.forward(cfg.vocab_size, 3)
    with pytest.raises(ValueError):
        m.forward(-1, 3)
    m.reset()
    with pytest.raises(ValueError):
        m.forward(1, 1)
    first, _ = m.forward(5, 0)
    assert np.array_equal(first, a[0])
    m.close()


def test_greedy_teacher_forcing_consistent():
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    p = synth.make_prompt(cfg, 4, seed=1)
    ids, logits = orc.greedy(cfg, w, p, 16)
    assert len(ids) == 17 and logits.shape == (20, cfg.vocab_size)
    ids2, logits2 = orc.greedy(cfg, w, p, 16, teacher=ids[:16])
    assert ids2 == ids and np.array_equal(logits, logits2)
    assert ids[0] == int(np.argmax(logits[3]))


@pytest.mark.parametrize("head", ["f16", "int4", "bf16"])
def test_separately_stored_head(head):
    """The output head as a separate stored matrix ("gpt2.s" README, Options:
    -h stores it in fp16; or grouped int4; or bf16, the batched path's
    head): passing wte itself changes
    nothing, bit for bit; a rounded head matches the library forward with
    that head, while the embedding still reads the fp32 wte."""
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 12, seed=2)
    w_same = dict(w, head=np.array(w["wte"], copy=True))
    w16 = orc.stored_weights(w, "f32", head=head)
    assert not np.array_equal(w16["head"], w["wte"])
    assert np.array_equal(w16["wte"], w["wte"])
    ref16 = torch_gpt2_logits(cfg, w16, toks)
    ref32 = torch_gpt2_logits(cfg, w, toks)
    a, b, c = orc.OracleModel(cfg, w), orc.OracleModel(cfg, w_same), orc.OracleModel(cfg, w16)
    try:
        moved = 0.0
        for pos, t in enumerate(toks):
            la, _ = a.forward(int(t), pos)
            lb, _ = b.forward(int(t), pos)
            lc, _ = c.forward(int(t), pos)
            assert np.array_equal(la, lb)
            assert np.abs(lc - ref16[pos]).max() <= 2e-5
            moved = max(moved, float(np.abs(ref16[pos] - ref32[pos]).max()))
        assert moved > 1e-5                    # the stored head is a different matrix
    finally:
        a.close(); b.close(); c.close()


def test_multicore_build_gives_the_same_bits():
    """The CPU baseline's OpenMP build splits each matrix product's outputs
    between threads; every output keeps its operations and their order, so
    the logits are bitwise those of the single-thread build."""
    import os
    cfg = synth.TINY
    w = synth.make_weights(cfg, 0)
    prompt = synth.make_prompt(cfg, 6, 1)
    rows = {}
    old = os.environ.get("OMP_NUM_THREADS")
    os.environ["OMP_NUM_THREADS"] = "3"        # an uneven split of every output range
    try:
        for omp in (False, True):
            m = orc.OracleModel(cfg, w, omp=omp)
            try:
                rows[omp] = np.stack([m.forward(int(t), p)[0] for p, t in enumerate(prompt)])
            finally:
                m.close()
    finally:
        if old is None:
            os.environ.pop("OMP_NUM_THREADS", None)
        else:
            os.environ["OMP_NUM_THREADS"] = old
    assert np.array_equal(rows[False].view(np.uint32), rows[True].view(np.uint32))


def test_export_kv_layout():
    """The oracle's cache accessor returns, for layer 0, row p of head h = the
    k and v slices of LN1(wte[t] + wpe[p]) . W_attn + b_attn (float64 torch
    routines), laid out [head][row][head_dim]."""
    import torch
    import torch.nn.functional as F
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 7, seed=3)
    m = orc.OracleModel(cfg, w)
    try:
        for p, t in enumerate(toks):
            m.forward(int(t), p)
        k, v = m.export_kv(0, len(toks))
    finally:
        m.close()
    d = lambda a: torch.from_numpy(np.asarray(a, np.float32)).double()
    E, H, D = cfg.n_embd, cfg.n_head, cfg.head_dim
    L0 = w["layers"][0]
    x = d(w["wte"])[torch.as_tensor(np.asarray(toks, np.int64))] + d(w["wpe"])[:len(toks)]
    qkv = F.layer_norm(x, (E,), d(L0["ln1_w"]), d(L0["ln1_b"]), eps=cfg.ln_eps) @ d(L0["attn_w"]) + d(L0["attn_b"])
    kr = qkv[:, E:2 * E].reshape(len(toks), H, D).transpose(0, 1).numpy()
    vr = qkv[:, 2 * E:].reshape(len(toks), H, D).transpose(0, 1).numpy()
    assert np.abs(k - kr).max() <= 1e-5 and np.abs(v - vr).max() <= 1e-5
    with pytest.raises(ValueError):
        m2 = orc.OracleModel(cfg, w)
        try:
            m2.export_kv(0, 1)                       # nothing cached yet
        finally:
            m2.close()


def test_bf16_kv_cache_holds_rounded_rows():
    """bf16 KV mode: every cached value is a bf16 number (low 16 bits zero),
    and layer 0's rows are exactly torch's bf16 rounding of the fp32 mode's
    rows (layer 0 sees the same inputs in both modes)."""
    import torch
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 9, seed=3)
    kv = {}
    for mode in ("f32", "bf16"):
        m = orc.OracleModel(cfg, w, kv=mode)
        try:
            for p, t in enumerate(toks):
                m.forward(int(t), p)
            kv[mode] = [m.export_kv(l, len(toks)) for l in range(cfg.n_layer)]
        finally:
            m.close()
    for l in range(cfg.n_layer):
        for a in kv["bf16"][l]:
            assert not np.any(a.view(np.uint32) & 0xFFFF)
    for a32, a16 in zip(kv["f32"][0], kv["bf16"][0]):
        rounded = torch.from_numpy(a32).bfloat16().float().numpy()
        assert np.array_equal(a16.view(np.uint32), rounded.view(np.uint32))


@pytest.mark.parametrize("cfg", [synth.TINY, CFG64], ids=["tiny", "d64"])
def test_bf16_kv_decode_matches_library_float64_forward(cfg):
    """The bf16 KV mode against the float64 library forward whose k and v are
    rounded to bf16: far closer to it than to the unrounded forward (the
    rounding changes the logits by ~1e-3, a pass that skipped it or rounded
    q instead would sit as far from the rounded reference)."""
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 20, seed=1)
    ref_r = torch_gpt2_logits(cfg, w, toks, kv_round="bf16")
    ref_f = torch_gpt2_logits(cfg, w, toks)
    m = orc.OracleModel(cfg, w, kv="bf16")
    try:
        got = np.stack([m.forward(int(t), p)[0] for p, t in enumerate(toks)])
    finally:
        m.close()
    d_r, d_f = np.abs(got - ref_r).max(), np.abs(got - ref_f).max()
    assert d_r <= 2e-5, d_r
    assert d_r * 10 <= d_f, (d_r, d_f)
