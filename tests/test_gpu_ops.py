"""GPU parity of the stand-alone operations against the oracle's functions."""
import numpy as np
import pytest

from oracle import oracle as orc
from transformer_decode_token_gb300 import binding

from gpu_util import max_abs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,n", [(1, 768), (37, 768), (5, 128), (3, 100), (64, 3072)])
def test_layernorm_rows(rows, n):
    import torch
    rng = np.random.default_rng(rows * 1000 + n)
    x = (rng.standard_normal((rows, n)) * 2 + 0.3).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
    b = (0.1 * rng.standard_normal(n)).astype(np.float32)
    y = binding.op_layernorm(torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda(),
                             torch.from_numpy(b).cuda(), 1e-5).cpu().numpy()
    torch.cuda.synchronize()
    for r in range(rows):
        assert max_abs(y[r], orc.layernorm(x[r], g, b, 1e-5)) <= 2e-5


@pytest.mark.parametrize("V,E", [(512, 128), (50257, 768), (1001, 64), (7, 4)])
def test_head_argmax(V, E):
    import torch
    rng = np.random.default_rng(V + E)
    x = rng.standard_normal(E).astype(np.float32)
    g = (1 + 0.01 * rng.standard_normal(E)).astype(np.float32)
    b = (0.01 * rng.standard_normal(E)).astype(np.float32)
    wte = (0.02 * rng.standard_normal((V, E))).astype(np.float32)
    ref = orc.linear_t(orc.layernorm(x, g, b, 1e-5), wte)
    dev = lambda a: torch.from_numpy(a).cuda()
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.op_head_argmax_workspace(V, E), dtype=torch.uint8, device="cuda")
    for _ in range(2):                      # the workspace is reused across calls
        binding.op_head_argmax(dev(x), dev(g), dev(b), 1e-5, dev(wte), logits, tok, ws)
        out = logits.cpu().numpy()
        assert max_abs(out, ref) <= 1e-4
        # the kernel's argmax is exactly the argmax of the logits it wrote
        assert int(tok.item()) == int(np.argmax(out))
        s = np.sort(ref)
        if V > 1 and s[-1] - s[-2] > 1e-3:
            assert int(tok.item()) == int(np.argmax(ref))


def test_head_argmax_ties_take_lowest_index():
    import torch
    V, E = 4096, 64
    x = np.ones(E, np.float32)
    x[::2] = -1.0                                 # LN(x) = +-1 exactly
    g = np.ones(E, np.float32)
    b = np.zeros(E, np.float32)
    wte = np.zeros((V, E), np.float32)
    for r in (17, 1000, 3333):                    # three equal maxima
        wte[r, 1] = 0.5
    dev = lambda a: torch.from_numpy(a).cuda()
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.op_head_argmax_workspace(V, E), dtype=torch.uint8, device="cuda")
    binding.op_head_argmax(dev(x), dev(g), dev(b), 1e-5, dev(wte), logits, tok, ws)
    assert int(tok.item()) == 17
