"""Pins for the oracle's scalar and vector functions.

Each check ties the oracle to something other than itself: double-precision
libm / numpy / torch library routines, closed forms and invariants that the
pages state, and brute force on tiny shapes.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc


# ---- exp ("Let's make GPT-2 in assembly", Step 5) -----------------------

def test_expf_error_bound_and_claim():
    x = np.linspace(-87.0, 88.0, 2_000_001, dtype=np.float32)
    y = orc.expf_vec(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    # degree-6 Taylor remainder at |r| = ln2/2 is ~1.7e-7 relative, plus fp32
    # rounding of the polynomial and of 2^k * p.
    assert rel.max() <= 3e-7
    # Step 5: the error stays below one part in ten million "in most places"
    assert (rel < 1e-7).mean() >= 0.9


def test_expf_special_values():
    assert orc.expf(0.0) == 1.0
    for k in range(-120, 120, 7):
        xk = np.float32(k * np.log(2.0))          # close to k ln2: result close to 2^k
        assert orc.expf(float(xk)) == pytest.approx(np.exp(np.float64(xk)), rel=3e-7)
        assert orc.expf(float(xk)) == pytest.approx(2.0 ** k, rel=1e-5)
    assert orc.expf(100.0) == float("inf")
    assert orc.expf(-100.0) == 0.0
    assert orc.expf(88.7) == pytest.approx(np.exp(np.float64(np.float32(88.7))), rel=3e-7)


def test_expf_range_reduction():
    # Step 5: x = k ln2 + r with r always between -0.35 and 0.35
    for x in np.linspace(-87, 88, 4001, dtype=np.float32):
        k, r = orc.expf_reduce(float(x))
        assert abs(r) <= 0.35
        assert abs(k * np.log(2.0) + r - float(x)) <= 1e-5 * max(1.0, abs(float(x)))


# ---- tanh and gelu_new ------------------------------------------------------

def test_tanh_via_exp():
    z = np.linspace(-12, 12, 24001).astype(np.float32)
    t = np.array([orc.tanhf(float(v)) for v in z])
    assert np.abs(t - np.tanh(z.astype(np.float64))).max() <= 3e-7
    assert orc.tanhf(0.0) == 0.0
    assert orc.tanhf(50.0) == 1.0 and orc.tanhf(-50.0) == -1.0


def test_gelu_new_matches_graph_file_sigmoid_form():
    # model.fir, comment above g2.gelu_new: x * sigmoid(2 sqrt(2/pi) (x + 0.044715 x^3))
    x = np.linspace(-10, 10, 40001).astype(np.float32)
    g = orc.gelu_new_vec(x).astype(np.float64)
    xd = x.astype(np.float64)
    u = 2.0 * np.sqrt(2.0 / np.pi) * (xd + 0.044715 * xd ** 3)
    ref = xd / (1.0 + np.exp(-u))
    assert np.abs(g - ref).max() <= 1e-6


def test_gelu_new_matches_library_tanh_gelu():
    x = torch.linspace(-8, 8, 10001, dtype=torch.float64)
    ref = F.gelu(x, approximate="tanh").numpy()
    g = orc.gelu_new_vec(x.numpy().astype(np.float32)).astype(np.float64)
    assert np.abs(g - ref).max() <= 1e-6


def test_gelu_new_identities():
    assert orc.gelu_new(0.0) == 0.0
    # gelu(x) - gelu(-x) = x for any function of the form x * (1 + odd(x)) / 2
    for x in np.linspace(-6, 6, 121, dtype=np.float32):
        assert orc.gelu_new(float(x)) - orc.gelu_new(float(-x)) == pytest.approx(float(x), abs=2e-6)
    assert orc.gelu_new(20.0) == pytest.approx(20.0, abs=1e-6)
    assert orc.gelu_new(-20.0) == pytest.approx(0.0, abs=1e-6)


# ---- LayerNorm (model.fir kernel g2.layernorm) ------------------------------

def test_layernorm_normalises_with_biased_variance():
    rng = np.random.default_rng(5)
    for n in (8, 128, 768):
        x = rng.standard_normal(n).astype(np.float32) * 3 + 1.5
        y = orc.layernorm(x, np.ones(n), np.zeros(n), eps=1e-5).astype(np.float64)
        var = np.var(x.astype(np.float64))
        assert abs(y.mean()) <= 1e-6
        # biased variance of the output is var / (var + eps); an unbiased
        # (n-1) variance would leave (n-1)/n here
        assert abs(y.var() * (var + 1e-5) / var - 1.0) <= 1e-5


def test_layernorm_gamma_beta_roles_and_constant_input():
    n = 64
    x = np.full(n, 3.25, np.float32)
    y = orc.layernorm(x, np.ones(n), np.zeros(n))
    assert np.all(y == 0.0)
    rng = np.random.default_rng(6)
    x = rng.standard_normal(n).astype(np.float32)
    y = orc.layernorm(x, np.full(n, 2.0), np.full(n, 3.0)).astype(np.float64)
    assert y.mean() == pytest.approx(3.0, abs=1e-5)
    assert y.var() == pytest.approx(4.0 * np.var(x) / (np.var(x) + 1e-5), rel=1e-5)


def test_layernorm_matches_library():
    rng = np.random.default_rng(7)
    n = 768
    x = rng.standard_normal(n).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
    b = (0.1 * rng.standard_normal(n)).astype(np.float32)
    ref = F.layer_norm(torch.from_numpy(x).double(), (n,), torch.from_numpy(g).double(),
                       torch.from_numpy(b).double(), eps=1e-5).numpy()
    assert np.abs(orc.layernorm(x, g, b) - ref).max() <= 2e-6


# ---- softmax ------------------------------------------------------------------

def test_softmax_sums_to_one_and_shift_invariance():
    rng = np.random.default_rng(8)
    for n in (1, 2, 17, 1024):
        # scores on a 2^-10 grid, so that adding 32 is exact in fp32
        s = (np.round(rng.standard_normal(n) * 4 * 1024) / 1024).astype(np.float32)
        p = orc.softmax(s)
        assert abs(p.astype(np.float64).sum() - 1.0) <= 1e-6
        assert np.all(p >= 0)
        # subtracting the maximum makes the result independent of a shift
        p2 = orc.softmax(s + np.float32(32.0))
        assert np.array_equal(p2, p)
    assert orc.softmax(np.array([5.0]))[0] == 1.0


def test_softmax_two_element_closed_form():
    for d in (-3.0, -0.5, 0.0, 0.25, 2.0):
        p = orc.softmax(np.array([0.0, d], np.float32))
        assert p[1] == pytest.approx(1.0 / (1.0 + np.exp(-d)), abs=3e-7)


# ---- linear (GEMV) -------------------------------------------------------------

@pytest.mark.parametrize("shape", [(3, 5), (7, 33), (64, 96), (128, 384)])
def test_linear_brute_force_double(shape):
    rng = np.random.default_rng(9)
    inn, out = shape
    x = rng.standard_normal(inn).astype(np.float32)
    W = rng.standard_normal((inn, out)).astype(np.float32)
    b = rng.standard_normal(out).astype(np.float32)
    y = orc.linear(x, W, b).astype(np.float64)
    ref = x.astype(np.float64) @ W.astype(np.float64) + b
    scale = np.abs(x).astype(np.float64) @ np.abs(W).astype(np.float64) + np.abs(b)
    assert np.all(np.abs(y - ref) <= 1e-6 * scale + 1e-7)


def test_linear_vs_transposed_layout_is_bitwise_equal():
    rng = np.random.default_rng(10)
    x = rng.standard_normal(96).astype(np.float32)
    W = rng.standard_normal((96, 40)).astype(np.float32)
    a = orc.linear(x, W, None)
    b = orc.linear_t(x, np.ascontiguousarray(W.T))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_linear_picks_input_rows():
    # a one-hot input returns that input's row of the [in][out] matrix plus bias
    W = np.arange(12, dtype=np.float32).reshape(3, 4)
    b = np.array([0.5, 0.0, -1.0, 2.0], np.float32)
    y = orc.linear(np.array([0, 1, 0], np.float32), W, b)
    assert np.array_equal(y, W[1] + b)


def test_argmax_ties_take_lowest_index():
    assert orc.argmax(np.array([1, 3, 3, 2], np.float32)) == 1
    assert orc.argmax(np.array([-1, -1], np.float32)) == 0
    assert orc.argmax(np.array([0, 0, 0, 7], np.float32)) == 3


# ---- attention ("Let's make GPT-2 in assembly" Step 6; model.fir g2.attn_decode) ----

def _attn_case(H=3, D=16, P=8, seed=11):
    rng = np.random.default_rng(seed)
    kc = np.zeros((H, P, D), np.float32)
    vc = np.zeros((H, P, D), np.float32)
    return rng, kc, vc


def test_attention_position_zero_returns_v():
    H, D = 3, 16
    rng, kc, vc = _attn_case(H, D)
    qkv = rng.standard_normal(3 * H * D).astype(np.float32)
    out = orc.attn_decode(qkv, 0, H, kc, vc)
    assert np.array_equal(out, qkv[2 * H * D:])
    assert np.array_equal(kc[:, 0, :].reshape(-1), qkv[H * D:2 * H * D])
    assert np.array_equal(vc[:, 0, :].reshape(-1), qkv[2 * H * D:])


def test_attention_equal_keys_give_mean_of_values():
    H, D, P = 2, 8, 6
    rng, kc, vc = _attn_case(H, D, P)
    kvec = rng.standard_normal((H, D)).astype(np.float32)
    for p in range(4):
        vc[:, p, :] = rng.standard_normal((H, D))
        kc[:, p, :] = kvec
    qkv = rng.standard_normal(3 * H * D).astype(np.float32)
    qkv[H * D:2 * H * D] = kvec.reshape(-1)
    out = orc.attn_decode(qkv, 4, H, kc, vc).reshape(H, D)
    vals = np.concatenate([vc[:, :4, :], qkv[2 * H * D:].reshape(H, 1, D)], axis=1)
    assert np.abs(out - vals.mean(axis=1)).max() <= 1e-6


def test_attention_matches_library_sdpa():
    H, D, P, pos = 4, 64, 32, 20
    rng, kc, vc = _attn_case(H, D, P)
    kc[:, :pos, :] = rng.standard_normal((H, pos, D))
    vc[:, :pos, :] = rng.standard_normal((H, pos, D))
    qkv = rng.standard_normal(3 * H * D).astype(np.float32)
    k_all = np.concatenate([kc[:, :pos], qkv[H * D:2 * H * D].reshape(H, 1, D)], axis=1)
    v_all = np.concatenate([vc[:, :pos], qkv[2 * H * D:].reshape(H, 1, D)], axis=1)
    q = torch.from_numpy(qkv[:H * D].reshape(H, 1, D)).double()
    ref = F.scaled_dot_product_attention(q, torch.from_numpy(k_all).double(),
                                         torch.from_numpy(v_all).double()).reshape(-1).numpy()
    out = orc.attn_decode(qkv, pos, H, kc, vc)
    assert np.abs(out - ref).max() <= 2e-6
    # Step 6 divides by 8 for a head of 64: the scale is 1/sqrt(head_dim)
    s = (qkv[:D].astype(np.float64) @ k_all[0].T.astype(np.float64)) / 8.0
    p = np.exp(s - s.max()); p /= p.sum()
    assert np.abs(out[:D] - p @ v_all[0]).max() <= 2e-6
