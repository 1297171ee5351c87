"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, it exports every function include/gpt2.h declares, and calls with bad
arguments are rejected before any device work."""
import ctypes
import os
import re

import pytest

from transformer_decode_token_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gpt2.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gpt2_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gpt2_create", "gpt2_prefill", "gpt2_decode_step", "gpt2_argmax", "gpt2_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = binding.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"libgpt2.so does not export {n}"
    assert set(binding.EXPORTED) <= set(declared_functions())


def test_strerror_names_every_status():
    L = binding.lib()
    for code in binding.STATUS:
        assert L.gpt2_strerror(code)
    assert L.gpt2_strerror(0) == b"ok"
    assert b"unknown" in L.gpt2_strerror(12345)


def test_invalid_arguments_are_rejected_on_the_host():
    L = binding.lib()
    out = ctypes.c_void_p()
    # NULL config / NULL out / NULL model pointers
    assert L.gpt2_create(None, None, 0, None, ctypes.byref(out)) == -1
    assert L.gpt2_create(None, None, 0, None, None) == -1
    bad = [binding.Config(2, 128, 3, 64, 512, 1e-5),    # n_embd % n_head
           binding.Config(2, 120, 4, 64, 512, 1e-5),    # n_embd % 32
           binding.Config(2, 128, 8, 64, 512, 1e-5),    # head_dim 16
           binding.Config(0, 128, 4, 64, 512, 1e-5),    # no layers
           binding.Config(2, 128, 4, 64, 512, 0.0),     # eps
           binding.Config(2, 128, 4, 0, 512, 1e-5)]     # no positions
    w = binding.Weights()
    for c in bad:
        assert L.gpt2_create(ctypes.byref(c), ctypes.byref(w), 0, None, ctypes.byref(out)) == -1
    good = binding.Config(2, 128, 4, 64, 512, 1e-5)
    assert L.gpt2_create(ctypes.byref(good), ctypes.byref(w), 7, None, ctypes.byref(out)) == -1  # dtype
    int4_bad = binding.Config(2, 96, 3, 64, 512, 1e-5)   # int4 needs n_embd % 128
    assert L.gpt2_create(ctypes.byref(int4_bad), ctypes.byref(w), 2, None, ctypes.byref(out)) == -1
    for fn in ("gpt2_reset", "gpt2_sync"):
        assert getattr(L, fn)(None) == -1
    assert L.gpt2_decode_step(None, 0, 0, None) == -1
    assert L.gpt2_argmax(None, None) == -1
    assert L.gpt2_decode_greedy(None, 1) == -1
    assert L.gpt2_prefill(None, None, 1) == -1
    L.gpt2_destroy(None)
    assert L.gpt2_op_layernorm(None, None, None, 1, 4, 1e-5, None, None) == -1
    assert L.gpt2_op_head_argmax_workspace(50257, 768) >= 16 + 8 * 152


def test_new_options_are_rejected_on_the_host():
    """gpt2_set_sampling and the head flags validate their arguments before
    any device work: a NULL model, a negative or non-finite temperature,
    unknown or conflicting create flags."""
    L = binding.lib()
    out = ctypes.c_void_p()
    assert L.gpt2_set_sampling(None, 0.8, 1) == -1
    assert L.gpt2_set_sampling(None, 0.0, 1) == -1
    good = binding.Config(2, 128, 4, 64, 512, 1e-5)
    w = binding.Weights()
    # unknown flag bit; both head flags at once
    assert L.gpt2_create_ex(ctypes.byref(good), ctypes.byref(w), 0, 64, None, ctypes.byref(out)) == -1
    assert L.gpt2_create_ex(ctypes.byref(good), ctypes.byref(w), 0, 4 | 8, None, ctypes.byref(out)) == -1
    assert L.gpt2_path(None, None) == -1
    assert L.gpt2_launch_count(None, None) == -1

    assert L.gpt2_set_wait_limit(None, 0) == -1
    # the flag that once selected a third path is no longer accepted
    assert L.gpt2_create_ex(ctypes.byref(good), ctypes.byref(w), 0, 2, None, ctypes.byref(out)) == -1
    # batched models: unknown option bits, NULL arguments
    assert L.gpt2_create_batch_ex(ctypes.byref(good), ctypes.byref(w), 3, 4, 2, None, ctypes.byref(out)) == -1
    assert L.gpt2_create_batch_ex(None, None, 3, 4, 1, None, ctypes.byref(out)) == -1
    assert L.gpt2_create_batch_ex(ctypes.byref(good), ctypes.byref(w), 3, 4, 1, None, None) == -1
