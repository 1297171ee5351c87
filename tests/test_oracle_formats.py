"""Pins for the oracle's stored-weight formats: fp16 and bf16 rounding, and
the grouped asymmetric int4 quantiser and nibble packing."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bit_sample(n=2_000_000, seed=12):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    edge = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e-8,
                     2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 * 0.999,
                     6.1035156e-05, 5.9604645e-08, 3.0 * 2.0 ** -26, 1.0 + 2.0 ** -11,
                     1.0 + 3 * 2.0 ** -11, 3.4e38, -3.4e38, np.inf, -np.inf], np.float32)
    # values on fp16 rounding ties: odd multiples of half an fp16 ulp
    ties = (np.arange(1, 4001, 2, dtype=np.float64) * 2.0 ** -11 + 1.0).astype(np.float32)
    return np.concatenate([f, edge, ties, -ties])


def test_fp16_rounding_matches_ieee_library_conversion():
    x = _bit_sample()
    ours = orc.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):                # values past 65520 become inf
        ref = x.astype(np.float16).view(np.uint16)  # IEEE round-to-nearest-even
    assert np.array_equal(ours, ref)


def test_fp16_widening_is_exact_for_every_half():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_rounding_matches_library():
    x = _bit_sample(seed=13)
    ours = orc.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = orc.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


# ---- int4 ----------------------------------------------------------------------

def test_nibble_pack_unpack_roundtrip_all_bytes():
    allbytes = np.arange(256, dtype=np.uint8)
    vals = orc.unpack_nibbles(allbytes, 512)
    assert np.array_equal(vals[0::2], allbytes & 0xF)      # low nibble first
    assert np.array_equal(vals[1::2], allbytes >> 4)
    assert np.array_equal(orc.pack_nibbles(vals), allbytes)
    rng = np.random.default_rng(14)
    v = rng.integers(0, 16, size=1001).astype(np.uint8)
    assert np.array_equal(orc.unpack_nibbles(orc.pack_nibbles(v), 1001), v)


def test_int4_golden_grid():
    """A group whose weights lie on a grid of 1/8 quantises exactly."""
    with open(os.path.join(GOLDEN, "int4_grid.json")) as f:
        g = json.load(f)
    W = np.array(g["W_in_out"], np.float32)                 # [64][2]
    codes, scales, zeros = orc.quant_int4(W)
    assert scales.tolist() == g["scales"]
    assert [[(b & 0xF), b >> 4] for b in zeros[:, 0]] == g["zeros"]
    unpacked = [orc.unpack_nibbles(codes[o], 64).tolist() for o in range(2)]
    assert unpacked == g["codes"]
    assert np.array_equal(orc.dequant_int4(codes, scales, zeros), W.T)


def test_int4_layout_one_hot():
    """A single nonzero weight lands in the nibble of its (output, input)."""
    inn, out = 128, 8
    for (i, o) in [(0, 0), (1, 0), (37, 5), (127, 7), (64, 3)]:
        W = np.zeros((inn, out), np.float32)
        W[i, o] = 0.75
        codes, scales, zeros = orc.quant_int4(W)
        deq = orc.dequant_int4(codes, scales, zeros)       # [out][in]
        assert deq[o, i] == np.float32(0.75)
        deq[o, i] = 0
        assert np.all(deq == 0)
        g = i // 32
        assert scales[o, g] == np.float32(0.75 / 15)
        assert np.all(np.delete(scales.reshape(-1), o * (inn // 32) + g) == 1.0)
        nib = (codes[o, i // 2] >> (4 * (i & 1))) & 0xF
        assert nib == 15


def test_int4_error_bound_and_zero_group():
    rng = np.random.default_rng(15)
    inn, out = 256, 40
    W = (rng.standard_normal((inn, out)) * 0.02).astype(np.float32)
    W[:32, 3] = 0.0                                         # an all-zero group
    W[32:64, 4] = np.abs(W[32:64, 4])                       # a group with min > 0
    W[64:96, 5] = -np.abs(W[64:96, 5])                      # a group with max < 0
    codes, scales, zeros = orc.quant_int4(W)
    deq = orc.dequant_int4(codes, scales, zeros)            # [out][in]
    s_full = np.repeat(scales, 32, axis=1)
    err = np.abs(deq - W.T)
    assert np.all(err <= s_full * (0.5 + 1e-5))
    assert np.all(deq[3, :32] == 0.0) and scales[3, 0] == 1.0
    q = np.stack([orc.unpack_nibbles(codes[o], inn) for o in range(out)])
    assert (zeros[4, 0] >> 4) == 0        # row 4, group 1 (high nibble): min 0 -> zero point 0
    assert (zeros[5, 1] & 0xF) == 15      # row 5, group 2 (low nibble): max 0 -> zero point 15
    assert q.min() == 0 and q.max() == 15
    # every group reaches its end of the range: min -> code 0 or max -> code 15
    for o in range(out):
        for gi in range(inn // 32):
            grp = q[o, 32 * gi:32 * gi + 32]
            if scales[o, gi] != 1.0:
                assert grp.min() == 0 or grp.max() == 15


def test_stored_weights_modes():
    from transformer_decode_token_gb300 import synth
    cfg = synth.TINY
    w = synth.make_weights(cfg, seed=0)
    for mode in ("f16", "int4", "bf16"):
        sw = orc.stored_weights(w, mode)
        assert sw["wte"] is w["wte"]                          # head / embeddings stay fp32
        for L, L2 in zip(w["layers"], sw["layers"]):
            for k in orc.MATRIX_KEYS:
                assert L2[k].shape == L[k].shape
                d = np.abs(L2[k] - L[k]).max()
                assert 0 < d < (0.02 if mode == "int4" else 1e-3)
            assert L2["attn_b"] is L["attn_b"]
    with pytest.raises(ValueError):
        orc.stored_weights(w, "int8")
