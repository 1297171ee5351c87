"""Helpers shared by the GPU parity tests."""
import numpy as np


def max_abs(a, b) -> float:
    return float(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).max())


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def top2_margin(v) -> float:
    s = np.sort(np.asarray(v, np.float64))
    return float(s[-1] - s[-2])


def teacher_forced(model, tokens):
    """Runs the GPU model on tokens[i] at position i; returns (logits rows,
    argmax ids)."""
    rows, ids = [], []
    for pos, t in enumerate(tokens):
        model.decode_step(int(t), pos)
        rows.append(model.logits())
        ids.append(model.argmax())
    return np.stack(rows), ids


def check_rows(gpu_rows, ref_rows, gpu_ids, atol, rl2=None, margin=1e-3):
    """Element-wise parity of every step's logits, and bit-exact argmax ids
    wherever the oracle's top-2 margin exceeds `margin`."""
    assert gpu_rows.shape == ref_rows.shape
    for i in range(ref_rows.shape[0]):
        d = max_abs(gpu_rows[i], ref_rows[i])
        assert d <= atol, f"step {i}: max abs {d:.3g} > {atol}"
        if rl2 is not None:
            r = rel_l2(gpu_rows[i], ref_rows[i])
            assert r <= rl2, f"step {i}: relative L2 {r:.3g} > {rl2}"
        if top2_margin(ref_rows[i]) > margin:
            assert gpu_ids[i] == int(np.argmax(ref_rows[i])), f"step {i}: argmax differs"
