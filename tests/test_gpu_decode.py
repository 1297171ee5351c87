"""GPU parity: the CUDA decode path (through the C ABI) against the CPU oracle
on the same seeded weights and prompts.

Tolerances: fp32 logits max abs 1e-3 and relative L2 1e-4; fp16 and int4
logits max abs 2e-3 against the oracle run on the same stored weights; int4
codes / scales / zero points, fp16 bits and dequantised weights bit-exact;
argmax ids bit-exact wherever the oracle's top-2 margin exceeds 1e-3.  The
oracle's own chosen ids are fed to both sides (teacher forcing), so a legal
flip at a near tie cannot derail later steps.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from transformer_decode_token_gb300 import binding, synth

from gpu_util import check_rows, max_abs, rel_l2, teacher_forced, top2_margin

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-3, 1e-4), "f16": (2e-3, None), "int4": (2e-3, None)}
PATHS = ["cluster", "per_kernel"]
_BINDING_PATH = {"cluster": "auto", "per_kernel": "per_kernel"}
_cache = {}
_oracle_cache = {}


def model(cfg, dw, wdtype, path):
    m = binding.Model(cfg, dw, wdtype, path=_BINDING_PATH[path])
    assert m.path() == path
    return m


def weights(cfg, seed=0):
    key = (cfg, seed)
    if key not in _cache:
        _cache.clear()
        w = synth.make_weights(cfg, seed)
        _cache[key] = (w, binding.upload_weights(w))
    return _cache[key]


def run_parity(cfg, wdtype, n_prompt, n_steps, path, seed=0, prompt_seed=1):
    w, dw = weights(cfg, seed)
    prompt = synth.make_prompt(cfg, n_prompt, prompt_seed)
    key = (cfg, wdtype, n_prompt, n_steps, seed, prompt_seed)
    if key not in _oracle_cache:
        sw = orc.stored_weights(w, wdtype)
        _oracle_cache[key] = orc.greedy(cfg, sw, prompt, n_steps)
    ref_ids, ref_rows = _oracle_cache[key]
    tokens = list(prompt) + ref_ids[:n_steps]
    m = model(cfg, dw, wdtype, path)
    try:
        rows, ids = teacher_forced(m, tokens)
    finally:
        m.close()
    atol, rl2 = TOL[wdtype]
    check_rows(rows, ref_rows, ids, atol, rl2)
    return ref_ids, ref_rows, ids


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wdtype", ["f32", "f16", "int4"])
def test_tiny_teacher_forced(wdtype, path):
    run_parity(synth.TINY, wdtype, 4, 16, path)


@pytest.mark.parametrize("path", PATHS)
def test_small_fp32_config(path):
    """GPT-2 small fp32: 10-token prompt, 60 greedy steps, every step checked."""
    run_parity(synth.SMALL, "f32", 10, 60, path)


@pytest.mark.parametrize("path", PATHS)
def test_small_int4_config(path):
    """GPT-2 small with int4 block linears: 10-token prompt, 128 steps."""
    run_parity(synth.SMALL, "int4", 10, 128, path)


@pytest.mark.parametrize("path", PATHS)
def test_small_fp16_full_context(path):
    """GPT-2 small with fp16 block linears: 16-token prompt, decode until the
    1024-position cache is full (positions 0..1023)."""
    run_parity(synth.SMALL, "f16", 16, 1008, path)


@pytest.mark.parametrize("wdtype", ["f32", "int4"])
def test_paths_agree(wdtype):
    """The two paths compute the same pass: the same row dot products up to
    summation order (the cluster kernel adds the residual stream as
    fixed-point integers, the others in fp32)."""
    cfg = synth.SMALL
    _, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 10, 1)
    out = {}
    for path in PATHS:
        m = model(cfg, dw, wdtype, path)
        ids = m.generate(prompt, 30)
        out[path] = (ids, m.logits())
        m.close()
    for path in PATHS[:-1]:
        assert max_abs(out[path][1], out["per_kernel"][1]) <= 1e-4, path
        assert out[path][0] == out["per_kernel"][0], path


# ---- stored weights -----------------------------------------------------------

@pytest.mark.parametrize("cfg", [synth.TINY, synth.SMALL], ids=["tiny", "small"])
@pytest.mark.parametrize("wdtype", ["f32", "f16", "int4"])
def test_stored_weights_bit_exact(cfg, wdtype):
    w, dw = weights(cfg)
    m = binding.Model(cfg, dw, wdtype)
    try:
        layers = range(cfg.n_layer) if cfg is synth.TINY else [0, cfg.n_layer - 1]
        for l in layers:
            for which, key in enumerate(binding.MATRIX_KEYS):
                W = w["layers"][l][key]                       # HF [in][out]
                main, sc, z = m.export_matrix(l, which)
                if wdtype == "f32":
                    assert np.array_equal(main.view(np.float32).reshape(W.shape[::-1]), W.T)
                    ref_deq = np.ascontiguousarray(W.T)
                elif wdtype == "f16":
                    bits = orc.f32_to_f16_bits(np.ascontiguousarray(W.T))
                    assert np.array_equal(main.view(np.uint16).reshape(bits.shape), bits)
                    ref_deq = orc.f16_bits_to_f32(bits)
                else:
                    codes, scales, zeros = orc.quant_int4(W)
                    assert np.array_equal(main.reshape(codes.shape), codes)
                    assert np.array_equal(sc.view(np.float32).reshape(scales.shape).view(np.uint32),
                                          scales.view(np.uint32))
                    assert np.array_equal(z.reshape(zeros.shape), zeros)
                    ref_deq = orc.dequant_int4(codes, scales, zeros)
                deq = m.export_dequant(l, which)
                assert np.array_equal(deq.view(np.uint32), ref_deq.view(np.uint32))
    finally:
        m.close()


# ---- decoding semantics ----------------------------------------------------

@pytest.mark.parametrize("path", PATHS)
def test_generate_matches_oracle_and_host_loop(path):
    cfg = synth.TINY
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 4, 1)
    ref_ids, ref_rows = orc.greedy(cfg, w, prompt, 16)
    m = model(cfg, dw, "f32", path)
    try:
        ids = m.generate(prompt, 16)
        for i, (a, b) in enumerate(zip(ids, ref_ids)):
            if top2_margin(ref_rows[len(prompt) - 1 + i]) > 1e-3:
                assert a == b
            else:
                break                    # a legal near-tie flip: the runs may diverge
        last = m.logits()
        # the same passes driven from the host one token at a time
        m.prefill(prompt)
        for pos, t in enumerate(ids[:16]):
            m.decode_step(t, len(prompt) + pos)
        assert np.array_equal(m.logits(), last)      # bitwise: same kernels, same order
    finally:
        m.close()


@pytest.mark.parametrize("path", PATHS)
def test_runs_are_bitwise_reproducible(path):
    cfg = synth.TINY
    _, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 5, 3)
    outs = []
    for _ in range(2):
        m = model(cfg, dw, "int4", path)
        ids = m.generate(prompt, 20)
        outs.append((ids, m.logits()))
        m.close()
    assert outs[0][0] == outs[1][0]
    assert np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("path", PATHS)
def test_rewind_and_errors(path):
    cfg = synth.TINY
    _, dw = weights(cfg)
    m = model(cfg, dw, "f32", path)
    try:
        with pytest.raises(binding.GPT2Error) as e:
            m.argmax()
        assert e.value.name == "NOT_READY"
        rows = []
        for pos, t in enumerate([5, 6, 7, 8]):
            m.decode_step(t, pos)
            rows.append(m.logits())
        m.decode_step(7, 2)                              # rewind to position 2
        assert np.array_equal(m.logits(), rows[2])
        with pytest.raises(binding.GPT2Error) as e:
            m.decode_step(1, 4)                          # past the cached length (3)
        assert e.value.name == "POSITION_RANGE"
        with pytest.raises(binding.GPT2Error) as e:
            m.decode_step(cfg.vocab_size, 3)
        assert e.value.name == "TOKEN_RANGE"
        with pytest.raises(binding.GPT2Error) as e:
            m.decode_step(-1, 3)
        assert e.value.name == "TOKEN_RANGE"
        with pytest.raises(binding.GPT2Error):
            m.generate([1, 2], cfg.n_positions - 1)      # 2 + 63 > 64 positions
        with pytest.raises(binding.GPT2Error):
            m.prefill(np.zeros(cfg.n_positions + 1, np.int32))
        m.sync()
    finally:
        m.close()


@pytest.mark.parametrize("path", PATHS)
def test_full_context_edge(path):
    """Prefill the whole context, and generate up to the last position."""
    cfg = synth.TINY
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, cfg.n_positions, 4)
    full = orc.forward_full(cfg, w, prompt)
    m = model(cfg, dw, "f32", path)
    try:
        m.prefill(prompt)
        assert max_abs(m.logits(), full[-1]) <= 1e-3
        p2 = prompt[:8]
        ids = m.generate(p2, cfg.n_positions - 8)
        assert len(ids) == cfg.n_positions - 7
        ref_ids, _ = orc.greedy(cfg, w, p2, cfg.n_positions - 8)
        assert ids[0] == ref_ids[0]
        with pytest.raises(binding.GPT2Error) as e:
            m.decode_greedy(1)                           # the cache is full
        assert e.value.name == "POSITION_RANGE"
    finally:
        m.close()


@pytest.mark.parametrize("path", PATHS)
def test_kv_cache_contents(path):
    """The cache holds each position's k and v (stored by head)."""
    cfg = synth.TINY
    w, dw = weights(cfg)
    toks = synth.make_prompt(cfg, 6, 5)
    m = model(cfg, dw, "f32", path)
    try:
        m.prefill(toks)
        m.sync()
        k, v = m.export_kv(0, len(toks))
        # layer 0's k, v at position p come from LN1(wte[t] + wpe[p]) . W_attn + b
        E, H, D = cfg.n_embd, cfg.n_head, cfg.head_dim
        L0 = w["layers"][0]
        for p, t in enumerate(toks):
            x = w["wte"][t] + w["wpe"][p]
            qkv = orc.linear(orc.layernorm(x, L0["ln1_w"], L0["ln1_b"]), L0["attn_w"], L0["attn_b"])
            assert max_abs(k[:, p, :].reshape(-1), qkv[E:2 * E]) <= 1e-4
            assert max_abs(v[:, p, :].reshape(-1), qkv[2 * E:]) <= 1e-4
        assert m.kernels_per_step() == (5 * cfg.n_layer + 1 if path == "per_kernel" else 1)
    finally:
        m.close()


# ---- the launch configuration bench.py times -----------------------------------

@pytest.mark.parametrize("wdtype", ["f32", "int4"])
def test_bench_launch_configuration(wdtype):
    """GPT-2 small, default path, in the calls bench.py times: after a 10-token
    prefill, one host-fed pass (decode_step at position 10) and 59 device-fed
    greedy passes in one launch (decode_greedy).  The free-running greedy ids
    of gpt2_generate must equal the oracle's while the oracle's top-2 margin
    exceeds 1e-3; the bench's sequence of calls must end with bitwise the same
    logits as gpt2_generate (same kernels, same order), and those must match
    the oracle's last pass within the tolerance when no near tie intervened."""
    cfg = synth.SMALL
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 10, 1)
    ref_ids, ref_rows = orc.greedy(cfg, orc.stored_weights(w, wdtype), prompt, 60)
    m = binding.Model(cfg, dw, wdtype)
    try:
        ids = m.generate(prompt, 60)
        gen_last = m.logits()
        clean = True
        for i, (a, b) in enumerate(zip(ids, ref_ids)):
            if top2_margin(ref_rows[len(prompt) - 1 + i]) <= 1e-3:
                clean = False            # a legal near-tie flip: the runs may diverge from here
                break
            assert a == b, f"{wdtype}: greedy id {i} differs"
        # the bench's calls: prefill, argmax, decode_step, decode_greedy(59)
        m.prefill(prompt)
        tok0 = m.argmax()
        assert tok0 == ids[0]
        m.decode_step(tok0, len(prompt))
        m.decode_greedy(59)
        assert m.argmax() == ids[60]
        bench_last = m.logits()
        assert np.array_equal(bench_last, gen_last)
        if clean:
            atol, rl2 = TOL[wdtype]
            check_rows(bench_last[None, :], ref_rows[-1][None, :], [ids[60]], atol, rl2)
    finally:
        m.close()


# ---- temperature sampling ---------------------------------------------------------

@pytest.mark.parametrize("cfg_name,n_prompt,n_steps", [("tiny", 4, 16), ("small", 10, 40)])
def test_sampling_matches_oracle(cfg_name, n_prompt, n_steps):
    """Temperature sampling (T = 0.8) on the default path, fed the oracle's own
    draws (teacher forcing): every drawn id equals the oracle's wherever the
    top-2 margin of the oracle's perturbed scores exceeds 1e-3, and the logits
    meet the fp32 tolerance."""
    cfg = synth.TINY if cfg_name == "tiny" else synth.SMALL
    T, seed = 0.8, 20241
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, n_prompt, 1)
    ref_ids, ref_rows = orc.greedy(cfg, w, prompt, n_steps, temperature=T, seed=seed)
    tokens = list(prompt) + ref_ids[:n_steps]
    m = binding.Model(cfg, dw, "f32")
    try:
        assert m.path() == "cluster"
        m.set_sampling(T, seed)
        rows, ids = teacher_forced(m, tokens)
    finally:
        m.close()
    atol, _ = TOL["f32"]
    checked = 0
    for pos in range(len(tokens)):
        assert max_abs(rows[pos], ref_rows[pos]) <= atol, f"step {pos}"
        sc = orc.sample_scores(ref_rows[pos], T, seed, pos)
        if top2_margin(sc) > 1e-3:
            assert ids[pos] == int(np.argmax(sc)), f"step {pos}: drawn id differs"
            checked += 1
    assert checked >= len(tokens) // 2
    # a draw, not the greedy choice: at T = 0.8 some tokens differ from the argmax
    assert any(ids[p] != int(np.argmax(ref_rows[p])) for p in range(len(tokens)))


def test_sampling_controls():
    cfg = synth.TINY
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 4, 1)
    ref_ids, _ = orc.greedy(cfg, w, prompt, 8)
    m = binding.Model(cfg, dw, "f32")
    try:
        for bad in (-0.5, float("nan"), float("inf")):
            with pytest.raises(binding.GPT2Error):
                m.set_sampling(bad, 1)
        m.set_sampling(0.9, 5)
        a = m.generate(prompt, 8)
        b = m.generate(prompt, 8)
        assert a == b                                    # same seed and prompt: same draws
        m.set_sampling(0.0, 5)
        assert m.generate(prompt, 8) == ref_ids          # temperature 0 is greedy again
    finally:
        m.close()
    m = binding.Model(cfg, dw, "f32", path="per_kernel")
    try:
        with pytest.raises(binding.GPT2Error):
            m.set_sampling(0.8, 1)                       # drawn only by the cluster kernel
        m.set_sampling(0.0, 1)
    finally:
        m.close()


# ---- the fp16 output head (the README's -h mode) ----------------------------------

@pytest.mark.parametrize("cfg_name,wdtype,head,n_prompt,n_steps",
                         [("tiny", "f16", "f16", 4, 16), ("tiny", "f32", "f16", 4, 16),
                          ("small", "f16", "f16", 10, 60), ("small", "int4", "f16", 10, 30),
                          ("tiny", "int4", "int4", 4, 16), ("small", "int4", "int4", 10, 30)])
def test_stored_head_matches_oracle(cfg_name, wdtype, head, n_prompt, n_steps):
    """GPT2_FLAG_HEAD_F16 / _INT4: the LM head reads an fp16 or int4 copy of
    wte (the embedding still reads the fp32 wte); against the oracle run on
    the same stored weights (block matrices and head as stored),
    teacher-forced: logits within 2e-3, ids wherever the oracle's top-2 margin
    exceeds 1e-3."""
    cfg = synth.TINY if cfg_name == "tiny" else synth.SMALL
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, n_prompt, 1)
    ref_ids, ref_rows = orc.greedy(cfg, orc.stored_weights(w, wdtype, head=head), prompt, n_steps)
    tokens = list(prompt) + ref_ids[:n_steps]
    m = binding.Model(cfg, dw, wdtype, head=head)
    try:
        assert m.path() == "cluster"
        rows, ids = teacher_forced(m, tokens)
    finally:
        m.close()
    check_rows(rows, ref_rows, ids, 2e-3)


def test_stored_head_needs_the_cluster_kernel():
    cfg = synth.TINY
    _, dw = weights(cfg)
    for head in ("f16", "int4"):
        with pytest.raises(binding.GPT2Error):
            binding.Model(cfg, dw, "f32", path="per_kernel", head=head)


# ---- inputs that reach the numerically fragile parts -------------------------------

def _stress_parity(cfg, kind, wdtype, n_prompt, n_steps, path):
    """Teacher-forced parity on a stress input, measured against exact
    (float64) arithmetic.  With a common offset of 30 the residual stream is
    ill-conditioned for fp32: LayerNorm divides rounding errors of size
    ulp(30) ~ 2e-6 by std(x) ~ 0.03, so any fp32 evaluation, the oracle's
    included, is off from exact arithmetic by ~2e-4 (tiny) to ~3e-3 (GPT-2
    small) in the logits; the standard tolerance against the oracle then
    measures the conditioning, not the kernel.  The bar: per step, the CUDA
    path's distance from the exact logits is at most max(standard tolerance,
    3 x the oracle's own), element-wise and in relative L2, and its token is
    the exact argmax wherever the exact top-2 margin exceeds twice that.  A
    LayerNorm fold that cancels (W.(gamma*x) - mean*W.gamma at |mean| >> std)
    puts an error of ~3e-4 on every folded row of unit scale (a numpy model of
    the fold in fp32: ~3e-7 when centred on x[0]), a thousand times the
    centred fold's."""
    from ref64 import torch_gpt2_logits
    w = synth.make_stress_weights(cfg, kind)
    sw = orc.stored_weights(w, wdtype)
    dw = binding.upload_weights(w)
    prompt = synth.make_prompt(cfg, n_prompt, 1)
    ref_ids, ref_rows = orc.greedy(cfg, sw, prompt, n_steps)
    tokens = list(prompt) + ref_ids[:n_steps]
    m = model(cfg, dw, wdtype, path)
    try:
        rows, ids = teacher_forced(m, tokens)
    finally:
        m.close()
    atol, rl2 = TOL[wdtype]
    exact = torch_gpt2_logits(cfg, sw, tokens)
    for i in range(len(tokens)):
        tol = max(atol, 3 * max_abs(ref_rows[i], exact[i]))
        assert max_abs(rows[i], exact[i]) <= tol, f"step {i}"
        if rl2 is not None:
            assert rel_l2(rows[i], exact[i]) <= max(rl2, 3 * rel_l2(ref_rows[i], exact[i])), f"step {i}"
        if top2_margin(exact[i]) > 2 * tol:
            assert ids[i] == int(np.argmax(exact[i])), f"step {i}: argmax differs"


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("kind", ["offset", "outliers"])
@pytest.mark.parametrize("cfg_name,n_prompt,n_steps", [("tiny", 4, 16), ("small", 10, 20)])
def test_large_offset_and_outlier_residuals(cfg_name, n_prompt, n_steps, kind, path):
    """Residual streams with a common offset of 30 (|mean| ~ 1000 std at the
    first LayerNorm) or with three dimensions in the thousands: the cluster
    kernel folds each LayerNorm into the rows that follow it, a difference of
    two sums that cancels when |mean| >> std, and adds the residual stream in
    fixed point; fp32 tolerance against the oracle, teacher-forced."""
    cfg = synth.TINY if cfg_name == "tiny" else synth.SMALL
    _stress_parity(cfg, kind, "f32", n_prompt, n_steps, path)


@pytest.mark.parametrize("wdtype", ["f16", "int4"])
def test_large_offset_stored_weights(wdtype):
    _stress_parity(synth.TINY, "offset", wdtype, 4, 16, "cluster")


def test_fixed_point_range_is_reported():
    """A residual value beyond the fixed-point sums' range (|x| ~ 1e5 > 65000)
    is reported as GPT2_ERR_RANGE by the next synchronising call, not summed
    as a clamped value with status OK; the model stays usable afterwards."""
    cfg = synth.TINY
    dw = binding.upload_weights(synth.make_stress_weights(cfg, "overflow"))
    m = model(cfg, dw, "f32", "cluster")
    try:
        m.decode_step(5, 0)
        with pytest.raises(binding.GPT2Error) as e:
            m.sync()
        assert e.value.name == "RANGE"
        m.sync()                                         # reported once, then cleared
    finally:
        m.close()
    # the same weights within range (no offset) run clean on a fresh model
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 4, 1)
    ref_ids, _ = orc.greedy(cfg, w, prompt, 8)
    m = model(cfg, dw, "f32", "cluster")
    try:
        assert m.generate(prompt, 8) == ref_ids
    finally:
        m.close()


# ---- bounded device waits ------------------------------------------------------------

def test_wait_limit_runs_out_and_the_model_recovers():
    """Every wait of the cluster kernel is bounded.  With a limit of 0 ns the
    first wait that does not succeed at once gives up: the kernel records
    GPT2_ERR_TIMEOUT, every CTA skips its remaining work (the abort word, the
    producer's drain, the final cluster barrier) and returns, and the next
    synchronising call reports it within a second.  With the default limit
    restored, the same model and a fresh one match the oracle again."""
    import time
    cfg = synth.TINY
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 4, 1)
    ref_ids, ref_rows = orc.greedy(cfg, w, prompt, 12)
    m = model(cfg, dw, "f32", "cluster")
    try:
        m.set_wait_limit(0)
        t0 = time.perf_counter()
        status = "OK"
        try:
            m.generate(prompt, 12)
        except binding.GPT2Error as e:
            status = e.name
        assert status in ("TIMEOUT", "OK")
        assert time.perf_counter() - t0 < 1.0
        assert status == "TIMEOUT"                       # the weights cannot all be resident at once
        m.sync()                                         # the error was reported once and cleared
        m.set_wait_limit(2_000_000_000)
        assert m.generate(prompt, 12) == ref_ids
        assert max_abs(m.logits(), ref_rows[-1]) <= 1e-3
    finally:
        m.close()
    m = model(cfg, dw, "f32", "cluster")
    try:
        assert m.generate(prompt, 12) == ref_ids
    finally:
        m.close()
    m = model(cfg, dw, "f32", "per_kernel")
    try:
        with pytest.raises(binding.GPT2Error):
            m.set_wait_limit(0)                          # no cross-CTA waits on that path
    finally:
        m.close()


# ---- prompts on the tensor cores ----------------------------------------------------

@pytest.mark.parametrize("wdtype", ["f32", "f16", "int4"])
@pytest.mark.parametrize("cfg_name,n", [("tiny", 5), ("tiny", 13), ("tiny", 64), ("small", 10), ("small", 100)])
def test_tc_prefill_matches_oracle(cfg_name, n, wdtype):
    """gpt2_prefill on the cluster path runs the prompt's positions as the
    rows of one batched tensor-core step (two for more than 64): every
    position's K and V in every layer, and the last position's logits and
    choice, against the oracle on the same stored weights; then greedy
    passes continue from the state it leaves (the cluster kernel's first
    pass reads the choice as its token)."""
    cfg = synth.TINY if cfg_name == "tiny" else synth.SMALL
    if n > cfg.n_positions:
        pytest.skip("prompt longer than the context")
    w, dw = weights(cfg)
    sw = orc.stored_weights(w, wdtype)
    prompt = synth.make_prompt(cfg, n, 7)
    om = orc.OracleModel(cfg, sw, omp=True)
    try:
        for p, t in enumerate(prompt):
            ref_last, ref_tok = om.forward(int(t), p)
        ref_kv = [om.export_kv(l, n) for l in range(cfg.n_layer)]
    finally:
        om.close()
    atol = TOL[wdtype][0]
    m = model(cfg, dw, wdtype, "cluster")
    try:
        m.prefill(prompt)
        assert max_abs(m.logits(), ref_last) <= atol
        if top2_margin(ref_last) > 1e-3:
            assert m.argmax() == ref_tok
        for l in range(cfg.n_layer):
            k, v = m.export_kv(l, n)
            assert max_abs(k, ref_kv[l][0]) <= atol, f"layer {l} K"
            assert max_abs(v, ref_kv[l][1]) <= atol, f"layer {l} V"
        # greedy passes continue from the state the prefill leaves
        if n + 3 <= cfg.n_positions:
            m.decode_greedy(3)
            m.sync()
            ref_ids, ref_rows = orc.greedy(cfg, sw, prompt, 3, omp=True)
            if all(top2_margin(ref_rows[n - 1 + i]) > 1e-3 for i in range(4)):
                assert m.argmax() == ref_ids[3]
    finally:
        m.close()


def test_tc_prefill_agrees_with_single_token_passes():
    """The two prefill paths leave the same cache and logits (within the fp32
    tolerance) and the same greedy continuation."""
    cfg = synth.SMALL
    w, dw = weights(cfg)
    prompt = synth.make_prompt(cfg, 20, 9)
    out = {}
    for name, flags in (("tc", "auto"), ("passes", "no_tc")):
        m = binding.Model(cfg, dw, "f32", path="auto", tc_prefill=(flags == "auto"))
        try:
            ids = m.generate(prompt, 8)
            k, v = m.export_kv(cfg.n_layer - 1, 28)
            out[name] = (ids, m.logits(), k, v)
        finally:
            m.close()
    assert max_abs(out["tc"][1], out["passes"][1]) <= 1e-3
    assert max_abs(out["tc"][2], out["passes"][2]) <= 1e-3
    assert max_abs(out["tc"][3], out["passes"][3]) <= 1e-3
    ref_ids, ref_rows = orc.greedy(cfg, w, prompt, 8, omp=True)
    for i, (a, b) in enumerate(zip(out["tc"][0], ref_ids)):
        if top2_margin(ref_rows[len(prompt) - 1 + i]) <= 1e-3:
            break
        assert a == b
