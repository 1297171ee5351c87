"""The no-allocation head + argmax entry point.

Some callers cannot allocate device memory: hosts that own every byte of it
through their own pools and hand the library only fixed input and output
buffers, or decode loops that must never enter the CUDA allocator.  For them
gpt2_op_head_argmax_noalloc keeps its small scratch inside the library.  This
test calls it through the C ABI and checks that, on two calls in a row (the
second one finds the first call's leftovers in the shared scratch), its
logits and token match gpt2_op_head_argmax, the entry point that takes a
caller-allocated workspace.  It lives in a file of its own that pytest
collects last, and it does not depend on any other test having run.
"""
import ctypes

import numpy as np
import pytest

from transformer_decode_token_gb300 import binding

pytestmark = pytest.mark.gpu


def _inputs(V, E, seed):
    import torch
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(E).astype(np.float32)
    g = (1 + 0.01 * rng.standard_normal(E)).astype(np.float32)
    b = (0.01 * rng.standard_normal(E)).astype(np.float32)
    wte = (0.02 * rng.standard_normal((V, E))).astype(np.float32)
    return [torch.from_numpy(a).cuda() for a in (x, g, b, wte)]


@pytest.mark.parametrize("V,E", [(50257, 768), (512, 128), (131072, 64)])
def test_noalloc_matches_workspace_entry_point(V, E):
    import torch
    L = binding.lib()
    for seed in (1, 2):                       # two calls in a row, different data
        x, g, b, wte = _inputs(V, E, seed + V)
        ref_logits = torch.empty(V, dtype=torch.float32, device="cuda")
        ref_tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        ws = torch.empty(binding.op_head_argmax_workspace(V, E), dtype=torch.uint8, device="cuda")
        binding.op_head_argmax(x, g, b, 1e-5, wte, ref_logits, ref_tok, ws)
        logits = torch.full((V,), float("nan"), dtype=torch.float32, device="cuda")
        tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = L.gpt2_op_head_argmax_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                                           ctypes.c_void_p(b.data_ptr()), 1e-5, ctypes.c_void_p(wte.data_ptr()),
                                           V, E, ctypes.c_void_p(logits.data_ptr()),
                                           ctypes.c_void_p(tok.data_ptr()), stream)
        assert rc == 0, L.gpt2_strerror(rc)
        torch.cuda.synchronize()
        a, r = logits.cpu().numpy(), ref_logits.cpu().numpy()
        assert np.abs(a - r).max() <= 1e-4
        assert int(tok.item()) == int(ref_tok.item()) == int(np.argmax(r))


def test_noalloc_rejects_vocab_beyond_its_scratch():
    import torch
    L = binding.lib()
    E = 4
    V = 131072 + 1                            # one row more than the scratch covers
    x = torch.zeros(E, device="cuda")
    wte = torch.zeros((V, E), device="cuda")
    logits = torch.empty(V, device="cuda")
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = L.gpt2_op_head_argmax_noalloc(p(x), p(x), p(x), 1e-5, p(wte), V, E, p(logits), p(tok), None)
    assert rc == -1                            # GPT2_ERR_INVALID_ARG
