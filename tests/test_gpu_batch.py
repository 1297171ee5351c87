"""GPU parity of the batched decode path (tcgen05 linears, ragged attention)
against the CPU oracle, through the C ABI.

The oracle runs each sequence on its own with the weights as the batched
model stores them: the 48 block matrices rounded to bf16 and the output head
a bf16 copy of wte (the embedding still reads the fp32 wte).  Activations
enter each tensor-core product as bf16 hi + lo parts (about 16 bits), sums
are fp32, so the stored-weight tolerance applies: logits within 2e-3 abs,
ids wherever the oracle's top-2 margin exceeds 1e-3.  The oracle's chosen
ids are fed to both sides (teacher forcing).  With the bf16 KV cache
(GPT2_BATCH_KV_BF16) the oracle runs its bf16 KV mode: k and v rounded to
bf16 as the cache stores them.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from transformer_decode_token_gb300 import binding, synth

from gpu_util import max_abs, top2_margin

pytestmark = pytest.mark.gpu

ATOL = 2e-3


def bf16_round(a):
    return orc.bf16_bits_to_f32(orc.f32_to_bf16_bits(np.asarray(a, np.float32)))


# ---- the tensor-core linear on its own ----------------------------------------------

@pytest.mark.parametrize("M,n,K", [(128, 64, 64), (300, 37, 192), (2304, 64, 768), (768, 64, 3072),
                                   (50257, 9, 768), (96, 1, 128)])
def test_linear_bf16_matches_float64(M, n, K):
    """Y = X . W^T with W bf16 (exact in float64) and X fp32, against float64:
    several 128-row tiles with a ragged last one, K splits, a batch below
    64.  The hi + lo parts keep |x - hi - lo| <= 2^-17 |x| and the MMA sums
    in fp32, so the error stays below 1e-4 of sum |w x| (a transposed
    operand, a wrong tile row or a lost K chunk are off by O(1))."""
    import torch
    rng = np.random.default_rng(M + n + K)
    W = bf16_round(0.02 * rng.standard_normal((M, K)))
    X = rng.standard_normal((n, K)).astype(np.float32)
    Wt = torch.from_numpy(orc.f32_to_bf16_bits(W).view(np.int16)).cuda().view(torch.bfloat16)
    Y = binding.op_linear_bf16(Wt, torch.from_numpy(X).cuda()).cpu().numpy()
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    scale = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    err = np.abs(Y - ref)
    assert np.all(err <= 1e-4 * scale + 1e-6), f"max err {err.max():.3g}, max scale {scale.max():.3g}"


# ---- the batched model --------------------------------------------------------------

def oracle_weights(w):
    return orc.stored_weights(w, "bf16", head="bf16")


def run_batch(cfg, prompts, n_steps, check_seqs, kv="f32"):
    """Prefill the ragged prompts, then n_steps teacher-forced steps (every
    sequence fed the oracle's greedy ids); compares the logits of the
    sequences in check_seqs with the oracle at every step."""
    w = synth.make_weights(cfg, 0)
    sw = oracle_weights(w)
    B = len(prompts)
    ref = {}
    for b in check_seqs:
        ref[b] = orc.greedy(cfg, sw, prompts[b], n_steps, omp=True, kv=kv)
    m = binding.BatchModel(cfg, binding.upload_weights(w), B, kv=kv)
    try:
        m.prefill(prompts)
        first = m.argmax(B)
        for b in check_seqs:
            ids, rows = ref[b]
            if top2_margin(rows[len(prompts[b]) - 1]) > 1e-3:
                assert first[b] == ids[0], f"sequence {b}: first choice"
        lens = np.array([len(q) for q in prompts])
        toks = np.array(first, np.int32)
        for step in range(n_steps):
            for b in check_seqs:
                toks[b] = ref[b][0][step]
            m.decode(toks, lens + step)
            lg = m.logits(B)
            got = m.argmax(B)
            for b in check_seqs:
                row = ref[b][1][len(prompts[b]) + step]
                d = max_abs(lg[b], row)
                assert d <= ATOL, f"sequence {b} step {step}: max abs {d:.3g}"
                if top2_margin(row) > 1e-3:
                    assert got[b] == int(np.argmax(row)), f"sequence {b} step {step}: argmax"
            toks = np.array(got, np.int32)
        return m, ref
    except Exception:
        m.close()
        raise


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_tiny_batch_ragged(kv):
    """Tiny model, 13 sequences with prompts of 3..20 tokens, 10 steps; every
    sequence checked."""
    cfg = synth.TINY
    prompts = synth.make_batch_prompts(cfg, 13, 3, 20, seed=2)
    m, _ = run_batch(cfg, prompts, 10, list(range(13)), kv=kv)
    m.close()


def test_tiny_batch_full_and_kv_cache():
    """64 sequences (the full batch), every one checked; the cache rows of
    one sequence hold the oracle's k and v (layer 0)."""
    cfg = synth.TINY
    prompts = synth.make_batch_prompts(cfg, 64, 1, 30, seed=5)
    m, _ = run_batch(cfg, prompts, 6, list(range(64)))
    try:
        w = synth.make_weights(cfg, 0)
        b = 7
        toks = prompts[b]
        k, v = m.export_kv(0, b, len(toks))
        E = cfg.n_embd
        L0 = w["layers"][0]
        W0 = bf16_round(L0["attn_w"])
        for p, t in enumerate(toks):
            x = w["wte"][t] + w["wpe"][p]
            qkv = orc.linear(orc.layernorm(x, L0["ln1_w"], L0["ln1_b"]), W0, L0["attn_b"])
            assert max_abs(k[:, p, :].reshape(-1), qkv[E:2 * E]) <= 1e-4
            assert max_abs(v[:, p, :].reshape(-1), qkv[2 * E:]) <= 1e-4
        kps, _ = m.info()
        assert kps == 8 * cfg.n_layer + 4
    finally:
        m.close()


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_tiny_batch_of_one(kv):
    """max_batch 1: one cache slot, so prompts run a decode step per position
    (nothing to pack) and decode steps append before attending."""
    cfg = synth.TINY
    prompts = synth.make_batch_prompts(cfg, 1, 9, 9, seed=11)
    m, _ = run_batch(cfg, prompts, 6, [0], kv=kv)
    m.close()


def test_tiny_batch_prompt_steps_packing():
    """Prompts of 1, 2, 63, 64, 65 and 3 tokens: the prompt steps pack
    max_batch (here 6) (sequence, position) rows at a time, so sequences
    start and end inside a step and run across step boundaries; one-token
    prompts have no prompt step at all (only the final decode step).  Every
    sequence checked."""
    import dataclasses
    cfg = dataclasses.replace(synth.TINY, n_positions=128)
    base = synth.make_batch_prompts(cfg, 6, 63, 63, seed=9)
    lens = [1, 2, 63, 64, 65, 3]
    prompts = [[int(t) for t in np.resize(np.asarray(q), L)] for q, L in zip(base, lens)]
    m, _ = run_batch(cfg, prompts, 5, list(range(6)))
    m.close()


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_tiny_batch_long_contexts_span_attention_chunks(kv):
    """Tiny model with 256 positions: prompts of 40..230 tokens, so a
    sequence's attention covers up to four chunks of 64 positions (each
    chunk's softmax merged with the others'), 12 steps across chunk
    boundaries; every sequence checked."""
    import dataclasses
    cfg = dataclasses.replace(synth.TINY, n_positions=256)
    prompts = synth.make_batch_prompts(cfg, 9, 40, 230, seed=4)
    prompts[0] = prompts[0][:60]    # crosses the 64-position boundary during the steps
    prompts[1] = prompts[1][:128]   # starts exactly on a boundary
    m, _ = run_batch(cfg, prompts, 12, list(range(9)), kv=kv)
    m.close()


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_small_batch_of_64_ragged_prompts(kv):
    """GPT-2 small, 64 sequences with prompts of 32..512 tokens (the batched
    workload's shape), 3 teacher-forced steps; the oracle checks the three
    sequences with the shortest prompts (it runs each whole prompt)."""
    cfg = synth.SMALL
    prompts = synth.make_batch_prompts(cfg, 64, 32, 512, seed=2)
    order = np.argsort([len(q) for q in prompts])
    m, _ = run_batch(cfg, prompts, 3, [int(i) for i in order[:3]], kv=kv)
    m.close()


def test_bf16_kv_cache_rows():
    """With the bf16 cache every stored k, v is a bf16 number, within one
    bf16 rounding of the oracle's bf16 KV mode: the two round fp32 values
    computed in different orders (and from hi + lo activation parts), which
    differ by up to a few 1e-6, so values near zero may land a few bf16 steps
    apart (the 1e-5 absolute term); a row of another sequence or position
    would be off by O(0.1)."""
    cfg = synth.TINY
    prompts = synth.make_batch_prompts(cfg, 6, 5, 30, seed=7)
    m, _ = run_batch(cfg, prompts, 4, [2], kv="bf16")
    try:
        w = synth.make_weights(cfg, 0)
        om = orc.OracleModel(cfg, oracle_weights(w), kv="bf16")
        try:
            for p, t in enumerate(prompts[2]):
                om.forward(int(t), p)
            for layer in range(cfg.n_layer):
                rk, rv = om.export_kv(layer, len(prompts[2]))
                k, v = m.export_kv(layer, 2, len(prompts[2]))
                for got, ref in ((k, rk), (v, rv)):
                    assert not np.any(got.view(np.uint32) & 0xFFFF)
                    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-5)
        finally:
            om.close()
    finally:
        m.close()


def test_batch_greedy_matches_host_fed_steps():
    """Device-resident greedy steps give bitwise the host-fed steps' logits
    and ids (same kernels, same order), and inactive rows (-1) leave a
    sequence's cache and choice untouched."""
    cfg = synth.TINY
    w = synth.make_weights(cfg, 0)
    prompts = synth.make_batch_prompts(cfg, 5, 4, 9, seed=3)
    m = binding.BatchModel(cfg, binding.upload_weights(w), 5)
    try:
        m.prefill(prompts)
        m.decode_greedy(6)
        lg_dev = m.logits(5)
        ids_dev = m.argmax(5)
        m.prefill(prompts)
        toks = np.array(m.argmax(5), np.int32)
        lens = np.array([len(q) for q in prompts])
        for step in range(6):
            m.decode(toks, lens + step)
            toks = np.array(m.argmax(5), np.int32)
        assert np.array_equal(m.logits(5), lg_dev)
        assert list(toks) == ids_dev
        # sequence 2 sits one step out: its choice and cache stay as they were
        k_before, _ = m.export_kv(0, 2, lens[2] + 6)
        pos = lens + 6
        pos[2] = -1
        m.decode(toks, pos)
        assert m.argmax(5)[2] == toks[2]
        k_after, _ = m.export_kv(0, 2, lens[2] + 6)
        assert np.array_equal(k_before, k_after)
    finally:
        m.close()


def test_batch_rejects_bad_arguments():
    cfg = synth.TINY
    w = synth.make_weights(cfg, 0)
    dw = binding.upload_weights(w)
    with pytest.raises(binding.GPT2Error):
        binding.BatchModel(cfg, dw, 65)                 # more rows than one tile
    with pytest.raises(binding.GPT2Error):
        binding.BatchModel(cfg, dw, 4, wdtype="f32")    # bf16 weights only
    m = binding.BatchModel(cfg, dw, 4)
    try:
        with pytest.raises(binding.GPT2Error) as e:
            m.decode([1, 2], [0, 1])                    # position past the cached length
        assert e.value.name == "POSITION_RANGE"
        with pytest.raises(binding.GPT2Error) as e:
            m.decode([cfg.vocab_size], [0])
        assert e.value.name == "TOKEN_RANGE"
        with pytest.raises(binding.GPT2Error) as e:
            m.decode_greedy(1)
        assert e.value.name == "NOT_READY"
    finally:
        m.close()
