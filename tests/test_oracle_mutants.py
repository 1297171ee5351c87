"""The pins reject a wrong oracle: each case plants one plausible mistake in a
copy of the oracle's C source (built on the CPU into a temporary library) and
checks that the pin guarding that part fails on it, while the unmodified
source passes the same check.  The mistakes: a dropped or changed term
(the exp polynomial's last coefficient, gelu_new's cubic coefficient), a wrong
divisor (unbiased variance), a wrong or missing scale (attention), a wrong
index (the attention skipping the current position), a missing term (the MLP
residual), swapped operands (LayerNorm's gamma and beta)."""
import math
import os

import numpy as np
import pytest

from oracle import oracle as orc
from ref64 import torch_gpt2_logits
from transformer_decode_token_gb300 import synth

MUTANTS = {
    "exp_degree5": ("    float p = 1.0f / 720.0f;\n    p = p * r + 1.0f / 120.0f;",
                    "    float p = 1.0f / 120.0f;"),
    "gelu_coefficient": ("0.044715f * x3", "0.04715f * x3"),
    "unbiased_variance": ("    float var = ss / (float)n;", "    float var = ss / (float)(n - 1);"),
    "gamma_beta_swapped": ("y[i] = (x[i] - mean) * rstd * gamma[i] + beta[i];",
                           "y[i] = (x[i] - mean) * rstd * beta[i] + gamma[i];"),
    "attention_unscaled": ("            s[j] = dot * scale;", "            s[j] = dot;"),
    "attention_skips_current": ("            s[j] = dot * scale;",
                                "            s[j] = (j == pos && pos > 0) ? -INFINITY : dot * scale;"),
    "mlp_residual_dropped": ("        orc_linear(m->act, L->mlp_proj_w, L->mlp_proj_b, F, E, m->mix);\n"
                             "        for (int32_t e = 0; e < E; ++e) m->x[e] = m->x[e] + m->mix[e];",
                             "        orc_linear(m->act, L->mlp_proj_w, L->mlp_proj_b, F, E, m->mix);\n"
                             "        for (int32_t e = 0; e < E; ++e) m->x[e] = m->mix[e];"),
}


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_mutants")
    src = orc.source()
    out = {"original": orc.load(orc.build_variant(src, os.path.join(str(d), "original.so")))}
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"{name}: the text to change is not in the oracle source once"
        out[name] = orc.load(orc.build_variant(src.replace(old, new), os.path.join(str(d), name + ".so")))
    return out


def whole_pass_error(L):
    """The whole-pass pin: max |oracle - float64 library forward| over a
    20-token sequence (tolerance 2e-5 in test_oracle_model)."""
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    toks = synth.make_prompt(cfg, 20, seed=1)
    ref = torch_gpt2_logits(cfg, w, toks)
    m = orc.OracleModel(cfg, w, library=L)
    try:
        got = np.stack([m.forward(int(t), p)[0] for p, t in enumerate(toks)])
    finally:
        m.close()
    return float(np.abs(got - ref).max())


def exp_error(L):
    """The exp pin: max relative error against double exp over [-87, 88]
    (bound 3e-7 in test_oracle_math)."""
    xs = np.linspace(-87.0, 88.0, 20001, dtype=np.float32)
    return max(abs(L.orc_expf(float(x)) / math.exp(float(x)) - 1.0) for x in xs)


def gelu_error(L):
    """The gelu_new pin: max |oracle - the graph file's sigmoid form in
    double| (bound 1e-6 in test_oracle_math)."""
    xs = np.linspace(-6.0, 6.0, 2001, dtype=np.float32)
    c = 2.0 * math.sqrt(2.0 / math.pi)
    return max(abs(L.orc_gelu_new(float(x)) - float(x) / (1.0 + math.exp(-c * (float(x) + 0.044715 * float(x) ** 3))))
               for x in xs)


def test_the_original_passes_the_pins(libs):
    L = libs["original"]
    assert whole_pass_error(L) <= 2e-5
    assert exp_error(L) <= 3e-7
    assert gelu_error(L) <= 1e-6


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_a_planted_mistake_fails_its_pin(libs, name):
    """The exp polynomial's dropped term moves the logits by ~6e-7 only, so
    its own pin (the relative error bound) is the one that catches it; every
    other mistake fails the whole-pass pin."""
    L = libs[name]
    if name == "exp_degree5":
        assert exp_error(L) > 3e-7
        return
    if name == "gelu_coefficient":
        assert gelu_error(L) > 1e-6
    assert whole_pass_error(L) > 2e-5
