"""Thin ctypes binding over libgpt2.so (C ABI: include/gpt2.h).

Argument marshalling only: every step of the decode pass runs in the CUDA
library.  PyTorch provides device memory and streams.  If the library cannot
be built or loaded, every call raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

GPT2_F32, GPT2_F16, GPT2_INT4, GPT2_BF16 = 0, 1, 2, 3
WDTYPES = {"f32": GPT2_F32, "f16": GPT2_F16, "int4": GPT2_INT4, "bf16": GPT2_BF16}
MAT_ATTN, MAT_PROJ, MAT_FC, MAT_MLP_PROJ = 0, 1, 2, 3
MATRIX_KEYS = ("attn_w", "proj_w", "fc_w", "mlp_proj_w")   # index = MAT_*

STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED_DEVICE", -3: "TOKEN_RANGE",
          -4: "POSITION_RANGE", -5: "NOT_READY", -6: "CUDA", -7: "TIMEOUT",
          -8: "DEVICE_STATE", -9: "OUT_OF_MEMORY", -10: "RANGE"}

EXPORTED = ("gpt2_create", "gpt2_create_ex", "gpt2_path", "gpt2_launch_count", "gpt2_destroy", "gpt2_reset", "gpt2_decode_step", "gpt2_prefill",
            "gpt2_argmax", "gpt2_decode_greedy", "gpt2_generate", "gpt2_copy_logits", "gpt2_sync",
            "gpt2_matrix_bytes", "gpt2_export_matrix", "gpt2_export_dequant", "gpt2_export_kv",
            "gpt2_kernels_per_step", "gpt2_op_layernorm", "gpt2_op_head_argmax_workspace",
            "gpt2_op_head_argmax", "gpt2_op_head_argmax_noalloc", "gpt2_set_sampling", "gpt2_set_wait_limit",
            "gpt2_create_batch", "gpt2_create_batch_ex", "gpt2_destroy_batch", "gpt2_decode_batch", "gpt2_prefill_batch",
            "gpt2_decode_batch_greedy", "gpt2_argmax_batch", "gpt2_batch_ids", "gpt2_copy_logits_batch",
            "gpt2_export_kv_batch", "gpt2_batch_info", "gpt2_sync_batch", "gpt2_op_linear_bf16_workspace",
            "gpt2_op_linear_bf16", "gpt2_strerror")


class GPT2Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        msg = lib().gpt2_strerror(status).decode() if _lib is not None else self.name
        super().__init__(f"{what}: GPT2_ERR_{self.name} ({msg})" if what else msg)


class Config(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int32), ("n_embd", ctypes.c_int32), ("n_head", ctypes.c_int32),
                ("n_positions", ctypes.c_int32), ("vocab_size", ctypes.c_int32), ("ln_eps", ctypes.c_float)]


_LAYER_KEYS = ("ln1_w", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
               "ln2_w", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


class LayerWeights(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in _LAYER_KEYS]


class Weights(ctypes.Structure):
    _fields_ = [("wte", ctypes.c_void_p), ("wpe", ctypes.c_void_p), ("ln_f_w", ctypes.c_void_p),
                ("ln_f_b", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights))]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load_library(path: str):
    """Loads a specific build of the library (for example the phase-trace build
    that trace_cluster.py makes) in place of libgpt2.so.  Must come before any
    other call into the library."""
    global _lib
    if _lib is not None:
        raise RuntimeError("the library is already loaded")
    return lib(path=path)


def lib(build_if_stale: bool = True, path: str = None):
    """Loads libgpt2.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if path is None:
                path = _build.build() if build_if_stale else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libgpt2.so not found at {path}")
            L = ctypes.CDLL(path)
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            pi32 = ctypes.POINTER(ctypes.c_int32)
            L.gpt2_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, vp,
                                      ctypes.POINTER(vp)]
            L.gpt2_create_ex.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, i32, vp,
                                         ctypes.POINTER(vp)]
            L.gpt2_path.argtypes = [vp, pi32]
            L.gpt2_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
            L.gpt2_destroy.argtypes = [vp]
            L.gpt2_destroy.restype = None
            L.gpt2_reset.argtypes = [vp]
            L.gpt2_decode_step.argtypes = [vp, i32, i32, ctypes.POINTER(vp)]
            L.gpt2_prefill.argtypes = [vp, pi32, i32]
            L.gpt2_argmax.argtypes = [vp, pi32]
            L.gpt2_decode_greedy.argtypes = [vp, i32]
            L.gpt2_generate.argtypes = [vp, pi32, i32, i32, pi32]
            L.gpt2_copy_logits.argtypes = [vp, vp]
            L.gpt2_sync.argtypes = [vp]
            L.gpt2_matrix_bytes.argtypes = [vp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                            ctypes.POINTER(sz)]
            L.gpt2_export_matrix.argtypes = [vp, i32, i32, vp, vp, vp]
            L.gpt2_export_dequant.argtypes = [vp, i32, i32, vp]
            L.gpt2_export_kv.argtypes = [vp, i32, i32, vp, vp]
            L.gpt2_kernels_per_step.argtypes = [vp, pi32]
            L.gpt2_op_layernorm.argtypes = [vp, vp, vp, i32, i32, f32, vp, vp]
            L.gpt2_op_head_argmax_workspace.argtypes = [i32, i32]
            L.gpt2_op_head_argmax_workspace.restype = sz
            L.gpt2_op_head_argmax.argtypes = [vp, vp, vp, f32, vp, i32, i32, vp, vp, vp, sz, vp]
            L.gpt2_op_head_argmax_noalloc.argtypes = [vp, vp, vp, f32, vp, i32, i32, vp, vp, vp]
            L.gpt2_set_sampling.argtypes = [vp, f32, ctypes.c_uint64]
            L.gpt2_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
            L.gpt2_create_batch.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, i32, vp,
                                            ctypes.POINTER(vp)]
            L.gpt2_create_batch_ex.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, i32,
                                               ctypes.c_uint32, vp, ctypes.POINTER(vp)]
            L.gpt2_destroy_batch.argtypes = [vp]
            L.gpt2_destroy_batch.restype = None
            L.gpt2_decode_batch.argtypes = [vp, pi32, pi32, i32, ctypes.POINTER(vp)]
            L.gpt2_prefill_batch.argtypes = [vp, pi32, pi32, i32]
            L.gpt2_decode_batch_greedy.argtypes = [vp, i32]
            L.gpt2_argmax_batch.argtypes = [vp, pi32, i32]
            L.gpt2_batch_ids.argtypes = [vp, i32, i32, pi32]
            L.gpt2_copy_logits_batch.argtypes = [vp, i32, vp]
            L.gpt2_export_kv_batch.argtypes = [vp, i32, i32, i32, vp, vp]
            L.gpt2_batch_info.argtypes = [vp, pi32, ctypes.POINTER(ctypes.c_uint64)]
            L.gpt2_sync_batch.argtypes = [vp]
            L.gpt2_op_linear_bf16_workspace.argtypes = [i32, i32, i32]
            L.gpt2_op_linear_bf16_workspace.restype = sz
            L.gpt2_op_linear_bf16.argtypes = [vp, vp, i32, i32, i32, vp, vp, sz, vp]
            L.gpt2_strerror.argtypes = [ctypes.c_int]
            L.gpt2_strerror.restype = ctypes.c_char_p
            for n in EXPORTED:
                if n not in ("gpt2_destroy", "gpt2_destroy_batch", "gpt2_op_head_argmax_workspace",
                             "gpt2_op_linear_bf16_workspace", "gpt2_strerror"):
                    getattr(L, n).restype = ctypes.c_int
            _lib = L
    return _lib


def check(status: int, what: str = ""):
    if status != 0:
        raise GPT2Error(status, what)


def _ptr(t) -> ctypes.c_void_p:
    """Device (or host) address of a torch tensor / numpy array, or None."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def upload_weights(weights: dict, device="cuda"):
    """numpy weights (checkpoint layout) -> dict of contiguous fp32 CUDA tensors."""
    import torch

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    out = {k: t(weights[k]) for k in ("wte", "wpe", "ln_f_w", "ln_f_b")}
    out["layers"] = [{k: t(L[k]) for k in _LAYER_KEYS} for L in weights["layers"]]
    return out


class Model:
    """One GPT-2 decode model on the current CUDA device."""

    def __init__(self, cfg, dev_weights: dict, wdtype: str = "f32", stream=None, path: str = "auto",
                 head: str = "f32", tc_prefill: bool = True):
        """path: "auto" (the cluster kernel where possible, else the per-kernel
        graph) or "per_kernel".  head: "f32" (the tied wte), "f16" or "int4" (a
        copy for the LM head, GPT2_FLAG_HEAD_F16 / _INT4; cluster kernel only).
        tc_prefill=False: prompts as single-token passes (GPT2_FLAG_NO_TC_PREFILL)."""
        L = lib()
        self.cfg = cfg
        self.wdtype = wdtype
        self._stream_obj = stream
        c = Config(cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_positions, cfg.vocab_size, cfg.ln_eps)
        layers = (LayerWeights * cfg.n_layer)()
        for i, Lw in enumerate(dev_weights["layers"]):
            for k in _LAYER_KEYS:
                setattr(layers[i], k, Lw[k].data_ptr())
        w = Weights(dev_weights["wte"].data_ptr(), dev_weights["wpe"].data_ptr(),
                    dev_weights["ln_f_w"].data_ptr(), dev_weights["ln_f_b"].data_ptr(),
                    ctypes.cast(layers, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        flags = {"auto": 0, "per_kernel": 1}[path] | {"f32": 0, "f16": 4, "int4": 8}[head] | (0 if tc_prefill else 16)
        check(L.gpt2_create_ex(ctypes.byref(c), ctypes.byref(w), WDTYPES[wdtype], flags,
                               _stream_handle(stream), ctypes.byref(h)), "gpt2_create_ex")
        self._h = h

    # ---- decoding ----
    def reset(self):
        check(lib().gpt2_reset(self._h), "gpt2_reset")

    def decode_step(self, token: int, position: int) -> int:
        """Queues one pass; returns the device address of the logits."""
        p = ctypes.c_void_p()
        check(lib().gpt2_decode_step(self._h, int(token), int(position), ctypes.byref(p)),
              "gpt2_decode_step")
        return p.value

    def prefill(self, ids):
        a = np.ascontiguousarray(ids, np.int32)
        check(lib().gpt2_prefill(self._h, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), a.size),
              "gpt2_prefill")

    def argmax(self) -> int:
        t = ctypes.c_int32()
        check(lib().gpt2_argmax(self._h, ctypes.byref(t)), "gpt2_argmax")
        return int(t.value)

    def decode_greedy(self, n_steps: int):
        check(lib().gpt2_decode_greedy(self._h, int(n_steps)), "gpt2_decode_greedy")

    def set_sampling(self, temperature: float, seed: int = 0):
        check(lib().gpt2_set_sampling(self._h, float(temperature), int(seed) & (2**64 - 1)), "gpt2_set_sampling")

    def set_wait_limit(self, ns: int):
        check(lib().gpt2_set_wait_limit(self._h, int(ns)), "gpt2_set_wait_limit")

    def generate(self, prompt, n_steps: int) -> list:
        p = np.ascontiguousarray(prompt, np.int32)
        out = np.zeros(n_steps + 1, np.int32)
        i32p = ctypes.POINTER(ctypes.c_int32)
        check(lib().gpt2_generate(self._h, p.ctypes.data_as(i32p), p.size, int(n_steps),
                                  out.ctypes.data_as(i32p)), "gpt2_generate")
        return out.tolist()

    def logits(self) -> np.ndarray:
        out = np.empty(self.cfg.vocab_size, np.float32)
        check(lib().gpt2_copy_logits(self._h, _ptr(out)), "gpt2_copy_logits")
        return out

    def copy_logits_to(self, dst):
        check(lib().gpt2_copy_logits(self._h, _ptr(dst)), "gpt2_copy_logits")

    def sync(self):
        check(lib().gpt2_sync(self._h), "gpt2_sync")

    # ---- inspection ----
    def matrix_bytes(self, which: int):
        a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
        check(lib().gpt2_matrix_bytes(self._h, which, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
              "gpt2_matrix_bytes")
        return a.value, b.value, c.value

    def export_matrix(self, layer: int, which: int):
        """Raw stored bytes: (main, scales, zeros) as numpy uint8 arrays."""
        mb, sb, zb = self.matrix_bytes(which)
        main = np.empty(mb, np.uint8)
        sc = np.empty(sb, np.uint8) if sb else None
        z = np.empty(zb, np.uint8) if zb else None
        check(lib().gpt2_export_matrix(self._h, layer, which, _ptr(main), _ptr(sc), _ptr(z)),
              "gpt2_export_matrix")
        return main, sc, z

    def export_dequant(self, layer: int, which: int) -> np.ndarray:
        import torch
        E = self.cfg.n_embd
        shape = {MAT_ATTN: (3 * E, E), MAT_PROJ: (E, E), MAT_FC: (4 * E, E), MAT_MLP_PROJ: (E, 4 * E)}[which]
        t = torch.empty(shape, dtype=torch.float32, device="cuda")
        check(lib().gpt2_export_dequant(self._h, layer, which, _ptr(t)), "gpt2_export_dequant")
        return t.cpu().numpy()

    def export_kv(self, layer: int, n_rows: int):
        H, D = self.cfg.n_head, self.cfg.n_embd // self.cfg.n_head
        k = np.empty((H, n_rows, D), np.float32)
        v = np.empty((H, n_rows, D), np.float32)
        check(lib().gpt2_export_kv(self._h, layer, n_rows, _ptr(k), _ptr(v)), "gpt2_export_kv")
        return k, v

    def path(self) -> str:
        p = ctypes.c_int32()
        check(lib().gpt2_path(self._h, ctypes.byref(p)), "gpt2_path")
        return {0: "per_kernel", 2: "cluster"}[p.value]

    def launch_count(self) -> int:
        n = ctypes.c_uint64()
        check(lib().gpt2_launch_count(self._h, ctypes.byref(n)), "gpt2_launch_count")
        return int(n.value)

    def kernels_per_step(self) -> int:
        n = ctypes.c_int32()
        check(lib().gpt2_kernels_per_step(self._h, ctypes.byref(n)), "gpt2_kernels_per_step")
        return int(n.value)

    def close(self):
        if getattr(self, "_h", None):
            lib().gpt2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- stand-alone operations ------------------------------------------------

def op_layernorm(x, gamma, beta, eps: float, y=None, stream=None):
    """Warp-per-row LayerNorm of a [rows, n] fp32 CUDA tensor."""
    import torch
    rows, n = x.shape
    if y is None:
        y = torch.empty_like(x)
    check(lib().gpt2_op_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), rows, n, float(eps), _ptr(y),
                                  _stream_handle(stream)), "gpt2_op_layernorm")
    return y


def op_head_argmax_workspace(vocab: int, n_embd: int) -> int:
    return int(lib().gpt2_op_head_argmax_workspace(vocab, n_embd))


def op_head_argmax(x, ln_w, ln_b, eps: float, wte, logits, token, workspace, stream=None):
    """Final LayerNorm + tied head + argmax on CUDA tensors; token is int32[1]."""
    V, E = wte.shape
    check(lib().gpt2_op_head_argmax(_ptr(x), _ptr(ln_w), _ptr(ln_b), float(eps), _ptr(wte), V, E,
                                    _ptr(logits), _ptr(token), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream)), "gpt2_op_head_argmax")


def op_head_argmax_noalloc(x, ln_w, ln_b, eps: float, wte, logits, token, stream=None):
    """gpt2_op_head_argmax without a workspace, for callers that cannot
    allocate device memory; scratch lives inside the library (see gpt2.h)."""
    V, E = wte.shape
    check(lib().gpt2_op_head_argmax_noalloc(_ptr(x), _ptr(ln_w), _ptr(ln_b), float(eps), _ptr(wte), V, E,
                                            _ptr(logits), _ptr(token), _stream_handle(stream)),
          "gpt2_op_head_argmax_noalloc")


# ---- batched decoding ----------------------------------------------------------

def _i32(a):
    a = np.ascontiguousarray(a, np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


BATCH_KV_BF16 = 1


class BatchModel:
    """Up to max_batch independent sequences decoded together (bf16 weights,
    tensor-core linears); see gpt2_create_batch in include/gpt2.h.  kv:
    the cache's element type, "f32" or "bf16" (GPT2_BATCH_KV_BF16)."""

    def __init__(self, cfg, dev_weights: dict, max_batch: int, wdtype: str = "bf16", stream=None,
                 kv: str = "f32"):
        if kv not in ("f32", "bf16"):
            raise ValueError(f"unknown KV cache type {kv!r}")
        L = lib()
        self.cfg = cfg
        self.max_batch = max_batch
        c = Config(cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_positions, cfg.vocab_size, cfg.ln_eps)
        layers = (LayerWeights * cfg.n_layer)()
        for i, Lw in enumerate(dev_weights["layers"]):
            for k in _LAYER_KEYS:
                setattr(layers[i], k, Lw[k].data_ptr())
        w = Weights(dev_weights["wte"].data_ptr(), dev_weights["wpe"].data_ptr(),
                    dev_weights["ln_f_w"].data_ptr(), dev_weights["ln_f_b"].data_ptr(),
                    ctypes.cast(layers, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        check(L.gpt2_create_batch_ex(ctypes.byref(c), ctypes.byref(w), WDTYPES[wdtype], int(max_batch),
                                     BATCH_KV_BF16 if kv == "bf16" else 0, _stream_handle(stream), ctypes.byref(h)),
              "gpt2_create_batch_ex")
        self.kv = kv
        self._h = h

    def decode(self, tokens, positions) -> int:
        t, tp = _i32(tokens)
        p, pp = _i32(positions)
        assert t.size == p.size
        d = ctypes.c_void_p()
        check(lib().gpt2_decode_batch(self._h, tp, pp, t.size, ctypes.byref(d)), "gpt2_decode_batch")
        return d.value

    def prefill(self, prompts):
        lens, lp = _i32([len(q) for q in prompts])
        ids, ip = _i32(np.concatenate([np.asarray(q, np.int32) for q in prompts]))
        check(lib().gpt2_prefill_batch(self._h, ip, lp, lens.size), "gpt2_prefill_batch")

    def decode_greedy(self, n_steps: int):
        check(lib().gpt2_decode_batch_greedy(self._h, int(n_steps)), "gpt2_decode_batch_greedy")

    def argmax(self, n: int) -> list:
        out = np.zeros(n, np.int32)
        check(lib().gpt2_argmax_batch(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n),
              "gpt2_argmax_batch")
        return out.tolist()

    def ids(self, first_pos: int, n_pos: int) -> np.ndarray:
        out = np.zeros((n_pos, self.max_batch), np.int32)
        check(lib().gpt2_batch_ids(self._h, first_pos, n_pos, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
              "gpt2_batch_ids")
        return out

    def logits(self, n: int) -> np.ndarray:
        out = np.empty((n, self.cfg.vocab_size), np.float32)
        check(lib().gpt2_copy_logits_batch(self._h, n, _ptr(out)), "gpt2_copy_logits_batch")
        return out

    def export_kv(self, layer: int, seq: int, n_rows: int):
        H, D = self.cfg.n_head, self.cfg.n_embd // self.cfg.n_head
        k = np.empty((H, n_rows, D), np.float32)
        v = np.empty((H, n_rows, D), np.float32)
        check(lib().gpt2_export_kv_batch(self._h, layer, seq, n_rows, _ptr(k), _ptr(v)), "gpt2_export_kv_batch")
        return k, v

    def info(self):
        k, n = ctypes.c_int32(), ctypes.c_uint64()
        check(lib().gpt2_batch_info(self._h, ctypes.byref(k), ctypes.byref(n)), "gpt2_batch_info")
        return int(k.value), int(n.value)

    def sync(self):
        check(lib().gpt2_sync_batch(self._h), "gpt2_sync_batch")

    def close(self):
        if getattr(self, "_h", None):
            lib().gpt2_destroy_batch(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def op_linear_bf16(W_bf16, X, stream=None):
    """Y = X . W^T on the tensor cores: W a CUDA bf16 [M][K] tensor, X a CUDA
    fp32 [n][K] tensor (n <= 64); returns a new CUDA fp32 [n][M] tensor."""
    import torch
    M, K = W_bf16.shape
    n = X.shape[0]
    Y = torch.empty((n, M), dtype=torch.float32, device=X.device)
    ws_bytes = int(lib().gpt2_op_linear_bf16_workspace(M, n, K))
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=X.device)
    check(lib().gpt2_op_linear_bf16(_ptr(W_bf16), _ptr(X), M, n, K, _ptr(Y), _ptr(ws), ws_bytes,
                                    _stream_handle(stream)), "gpt2_op_linear_bf16")
    return Y
