"""ctypes wrapper around the C oracle (gpt2_oracle.c).  TEST INFRASTRUCTURE.

Only tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline and
reference legs may import this module.  It never imports the CUDA library,
and the CUDA library never imports it.

Weights are passed as dicts of float32 numpy arrays in the checkpoint's
(HF Conv1D) layout; see ``transformer_decode_token_gb300.synth`` for the
names and shapes.  Sources are cited in gpt2_oracle.h.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gpt2_oracle.c")
_HDR = os.path.join(_HERE, "gpt2_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None

# -ffp-contract=off: every product and sum rounds separately (GCC contracts
# a*b+c into an FMA by default on AArch64); no -ffast-math.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall"]


def build(force: bool = False, omp: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc); omp=True builds the
    multi-core variant liboracle_omp.so (-fopenmp: each matrix product's
    outputs split between threads, the same bits as the single-thread build)."""
    path = _LIB_OMP if omp else _LIB
    stale = (not os.path.exists(path) or
             os.path.getmtime(path) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = path + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, *(["-fopenmp"] if omp else []), "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


class _Cfg(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int32), ("n_embd", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_positions", ctypes.c_int32),
                ("vocab_size", ctypes.c_int32), ("ln_eps", ctypes.c_float)]


_FP = ctypes.POINTER(ctypes.c_float)
_LAYER_KEYS = ("ln1_w", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
               "ln2_w", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


class _Layer(ctypes.Structure):
    _fields_ = [(k, _FP) for k in _LAYER_KEYS]


class _Weights(ctypes.Structure):
    _fields_ = [("wte", _FP), ("wpe", _FP), ("lnf_w", _FP), ("lnf_b", _FP),
                ("layers", ctypes.POINTER(_Layer)), ("head", _FP)]


def build_variant(src_text: str, out_path: str) -> str:
    """Compile another oracle source (e.g. one with a planted mistake, for the
    tests that check the pins reject it) into out_path, same flags."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", *CFLAGS, "-I", _HERE, "-o", out_path, src, "-lm"])
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def load(path: str):
    """A ctypes handle on an oracle library at path, its calls typed."""
    L = ctypes.CDLL(path)
    _type_calls(L)
    return L


def lib(omp: bool = False):
    """The oracle library; omp=True: its multi-core build (OMP_NUM_THREADS,
    default all host cores)."""
    global _lib, _lib_omp
    with _lock:
        if (_lib_omp if omp else _lib) is None:
            L = load(build(omp=omp))
            if omp:
                _lib_omp = L
            else:
                _lib = L
    return _lib_omp if omp else _lib


def _type_calls(L):
    """Argument and result types of the oracle's C calls."""
    c_sz, c_i32, c_f = ctypes.c_size_t, ctypes.c_int32, ctypes.c_float
    vp = ctypes.c_void_p
    L.orc_expf.restype = c_f; L.orc_expf.argtypes = [c_f]
    L.orc_tanhf.restype = c_f; L.orc_tanhf.argtypes = [c_f]
    L.orc_gelu_new.restype = c_f; L.orc_gelu_new.argtypes = [c_f]
    L.orc_expf_reduce.argtypes = [c_f, ctypes.POINTER(c_i32), ctypes.POINTER(c_f)]
    L.orc_gelu_new_vec.argtypes = [vp, vp, c_sz]
    L.orc_expf_vec.argtypes = [vp, vp, c_sz]
    L.orc_layernorm.argtypes = [vp, vp, vp, c_i32, c_f, vp]
    L.orc_softmax.argtypes = [vp, c_i32]
    L.orc_linear.argtypes = [vp, vp, vp, c_i32, c_i32, vp]
    L.orc_linear_t.argtypes = [vp, vp, c_i32, c_i32, vp]
    L.orc_attn_decode.argtypes = [vp, c_i32, c_i32, c_i32, c_i32, vp, vp, vp]
    L.orc_argmax.restype = c_i32; L.orc_argmax.argtypes = [vp, c_i32]
    c_u64 = ctypes.c_uint64
    L.orc_splitmix64.restype = c_u64; L.orc_splitmix64.argtypes = [c_u64, c_u64]
    L.orc_uniform.restype = c_f; L.orc_uniform.argtypes = [c_u64, c_u64]
    L.orc_uniform_bits.restype = c_f; L.orc_uniform_bits.argtypes = [c_u64]
    L.orc_sample_scores.argtypes = [vp, c_i32, c_f, c_u64, c_i32, vp]
    L.orc_sample.restype = c_i32; L.orc_sample.argtypes = [vp, c_i32, c_f, c_u64, c_i32]
    L.orc_create.restype = vp
    L.orc_create.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Weights)]
    L.orc_destroy.argtypes = [vp]
    L.orc_reset.argtypes = [vp]
    L.orc_set_kv_bf16.restype = None
    L.orc_set_kv_bf16.argtypes = [vp, c_i32]
    L.orc_forward.restype = c_i32
    L.orc_forward.argtypes = [vp, c_i32, c_i32, vp]
    L.orc_export_kv.restype = c_i32
    L.orc_export_kv.argtypes = [vp, c_i32, c_i32, vp, vp]
    L.orc_forward_full.restype = c_i32
    L.orc_forward_full.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Weights),
                                   vp, c_i32, vp]
    for n in ("orc_f32_to_f16", "orc_f16_to_f32", "orc_f32_to_bf16", "orc_bf16_to_f32"):
        getattr(L, n).argtypes = [vp, vp, c_sz]
    L.orc_quant_int4.argtypes = [vp, c_i32, c_i32, vp, vp, vp]
    L.orc_dequant_int4.argtypes = [vp, vp, vp, c_i32, c_i32, vp]
    L.orc_pack_nibbles.argtypes = [vp, c_sz, vp]
    L.orc_unpack_nibbles.argtypes = [vp, c_sz, vp]


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


# ---- scalar / vector functions --------------------------------------------

def expf(x: float) -> float:
    return float(lib().orc_expf(float(x)))


def tanhf(z: float) -> float:
    return float(lib().orc_tanhf(float(z)))


def gelu_new(x: float) -> float:
    return float(lib().orc_gelu_new(float(x)))


def expf_reduce(x: float):
    k = ctypes.c_int32()
    r = ctypes.c_float()
    lib().orc_expf_reduce(float(x), ctypes.byref(k), ctypes.byref(r))
    return int(k.value), float(r.value)


def expf_vec(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().orc_expf_vec(_p(x), _p(y), x.size)
    return y


def gelu_new_vec(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().orc_gelu_new_vec(_p(x), _p(y), x.size)
    return y


def layernorm(x, gamma, beta, eps: float = 1e-5) -> np.ndarray:
    x, g, b = _f32(x), _f32(gamma), _f32(beta)
    y = np.empty_like(x)
    lib().orc_layernorm(_p(x), _p(g), _p(b), x.size, eps, _p(y))
    return y


def softmax(s) -> np.ndarray:
    s = _f32(s).copy()
    lib().orc_softmax(_p(s), s.size)
    return s


def linear(x, W, b=None) -> np.ndarray:
    """HF Conv1D linear: W is [in][out]."""
    x, W = _f32(x), _f32(W)
    inn, out = W.shape
    y = np.empty(out, np.float32)
    bb = _f32(b) if b is not None else None
    lib().orc_linear(_p(x), _p(W), _p(bb) if bb is not None else None, inn, out, _p(y))
    return y


def linear_t(x, W) -> np.ndarray:
    """y = W @ x for W stored [out][in]."""
    x, W = _f32(x), _f32(W)
    out, inn = W.shape
    y = np.empty(out, np.float32)
    lib().orc_linear_t(_p(x), _p(W), inn, out, _p(y))
    return y


def attn_decode(qkv, pos: int, n_head: int, k_cache: np.ndarray, v_cache: np.ndarray):
    """One layer; caches are [H][P][D] float32 arrays updated in place."""
    qkv = _f32(qkv)
    H, P, D = k_cache.shape
    assert H == n_head and k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.shape == k_cache.shape and v_cache.dtype == np.float32
    out = np.empty(H * D, np.float32)
    lib().orc_attn_decode(_p(qkv), pos, H, D, P, _p(k_cache), _p(v_cache), _p(out))
    return out


def argmax(v) -> int:
    v = _f32(v)
    return int(lib().orc_argmax(_p(v), v.size))


# ---- stored-weight formats -------------------------------------------------

def splitmix64(seed: int, k: int) -> int:
    return int(lib().orc_splitmix64(seed, k))


def uniform(seed: int, k: int) -> float:
    return float(lib().orc_uniform(seed, k))


def uniform_bits(z: int) -> float:
    """The uniform number that 64 random bits z map to."""
    return float(lib().orc_uniform_bits(z & (2**64 - 1)))


def sample_scores(logits, temperature: float, seed: int, pos: int) -> np.ndarray:
    """Gumbel-max scores of a temperature draw (their argmax is the draw)."""
    s = _f32(logits)
    out = np.empty_like(s)
    lib().orc_sample_scores(_p(s), s.size, temperature, seed, pos, _p(out))
    return out


def sample(logits, temperature: float, seed: int, pos: int) -> int:
    """The token chosen from these logits by the pass at position `pos`:
    greedy when temperature is 0, else a draw from softmax(logits / T)."""
    s = _f32(logits)
    return int(lib().orc_sample(_p(s), s.size, temperature, seed, pos))


def f32_to_f16_bits(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16(_p(x), _p(out), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_f16_to_f32(_p(h), _p(out), h.size)
    return out


def f32_to_bf16_bits(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16(_p(x), _p(out), x.size)
    return out


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_bf16_to_f32(_p(h), _p(out), h.size)
    return out


def quant_int4(W):
    """W is HF [in][out]; returns (codes [out][in/2] u8, scales [out][in/32]
    f32, zeros [out][in/64] u8)."""
    W = _f32(W)
    inn, out = W.shape
    assert inn % 64 == 0
    codes = np.empty((out, inn // 2), np.uint8)
    scales = np.empty((out, inn // 32), np.float32)
    zeros = np.empty((out, inn // 64), np.uint8)
    lib().orc_quant_int4(_p(W), inn, out, _p(codes), _p(scales), _p(zeros))
    return codes, scales, zeros


def dequant_int4(codes, scales, zeros) -> np.ndarray:
    """Returns the dequantised matrix as [out][in]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = _f32(scales)
    zeros = np.ascontiguousarray(zeros, np.uint8)
    out, half = codes.shape
    inn = half * 2
    W = np.empty((out, inn), np.float32)
    lib().orc_dequant_int4(_p(codes), _p(scales), _p(zeros), inn, out, _p(W))
    return W


def pack_nibbles(vals) -> np.ndarray:
    vals = np.ascontiguousarray(vals, np.uint8)
    out = np.empty((vals.size + 1) // 2, np.uint8)
    lib().orc_pack_nibbles(_p(vals), vals.size, _p(out))
    return out


def unpack_nibbles(packed, n: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    out = np.empty(n, np.uint8)
    lib().orc_unpack_nibbles(_p(packed), n, _p(out))
    return out


MATRIX_KEYS = ("attn_w", "proj_w", "fc_w", "mlp_proj_w")


def stored_weights(weights: dict, wdtype: str, head: str = "f32") -> dict:
    """The weights as a given storage mode holds them, widened back to fp32
    in the checkpoint layout: the 48 block matrices are rounded to fp16 or
    quantised to grouped int4; embeddings, biases, LayerNorm and the tied head
    stay fp32.  'f32' returns the weights unchanged.  head='f16' adds the
    output head stored as fp16 ("gpt2.s" README, Options: -h), head='int4'
    as grouped int4 (the same scheme as the block matrices, groups of 32
    along n_embd), a separate matrix: the embedding lookup still reads the
    fp32 wte."""
    if head == "f16":
        out = dict(stored_weights(weights, wdtype))
        out["head"] = f16_bits_to_f32(f32_to_f16_bits(_f32(weights["wte"])))
        return out
    if head == "bf16":   # the batched path's head: a bf16 copy of wte (round to nearest even)
        out = dict(stored_weights(weights, wdtype))
        out["head"] = bf16_bits_to_f32(f32_to_bf16_bits(_f32(weights["wte"])))
        return out
    if head == "int4":   # wte is already [out][in]; quant_int4 takes the HF [in][out] layout
        out = dict(stored_weights(weights, wdtype))
        out["head"] = np.ascontiguousarray(dequant_int4(*quant_int4(np.ascontiguousarray(_f32(weights["wte"]).T))))
        return out
    if head != "f32":
        raise ValueError(f"unknown head dtype {head!r}")
    if wdtype == "f32":
        return weights
    out = dict(weights)
    out["layers"] = []
    for L in weights["layers"]:
        L2 = dict(L)
        for k in MATRIX_KEYS:
            W = _f32(L[k])
            if wdtype == "f16":
                L2[k] = f16_bits_to_f32(f32_to_f16_bits(W))
            elif wdtype == "bf16":
                L2[k] = bf16_bits_to_f32(f32_to_bf16_bits(W))
            elif wdtype == "int4":
                L2[k] = np.ascontiguousarray(dequant_int4(*quant_int4(W)).T)
            else:
                raise ValueError(f"unknown weight dtype {wdtype!r}")
        out["layers"].append(L2)
    return out


# ---- the model -----------------------------------------------------------

def _cfg_struct(cfg) -> _Cfg:
    return _Cfg(cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_positions,
                cfg.vocab_size, cfg.ln_eps)


class _WeightsHolder:
    """Keeps the numpy arrays alive while C holds pointers to them."""

    def __init__(self, cfg, weights: dict):
        self.arrays = []

        def fp(a):
            a = _f32(a)
            self.arrays.append(a)
            return a.ctypes.data_as(_FP)

        n = cfg.n_layer
        assert len(weights["layers"]) == n
        self.layers = (_Layer * n)()
        for i, L in enumerate(weights["layers"]):
            for k in _LAYER_KEYS:
                setattr(self.layers[i], k, fp(L[k]))
        head = weights.get("head")
        self.w = _Weights(fp(weights["wte"]), fp(weights["wpe"]),
                          fp(weights["ln_f_w"]), fp(weights["ln_f_b"]),
                          ctypes.cast(self.layers, ctypes.POINTER(_Layer)),
                          fp(head) if head is not None else None)


class OracleModel:
    """Stateful single-sequence decode with a KV cache (omp=True: the
    multi-core build, for the CPU baseline's timing; kv="bf16": the cache
    holds k and v rounded to bf16, the batched configuration's KV variant)."""

    def __init__(self, cfg, weights: dict, omp: bool = False, kv: str = "f32", library=None):
        if kv not in ("f32", "bf16"):
            raise ValueError(f"unknown KV cache type {kv!r}")
        self.cfg = cfg
        self._lib = library if library is not None else lib(omp)
        self._c = _cfg_struct(cfg)
        self._h = _WeightsHolder(cfg, weights)
        self._m = self._lib.orc_create(ctypes.byref(self._c), ctypes.byref(self._h.w))
        if not self._m:
            raise ValueError("oracle: invalid config")
        self._lib.orc_set_kv_bf16(self._m, 1 if kv == "bf16" else 0)

    def forward(self, token: int, pos: int):
        logits = np.empty(self.cfg.vocab_size, np.float32)
        r = self._lib.orc_forward(self._m, int(token), int(pos), _p(logits))
        if r < 0:
            raise ValueError(f"oracle: bad token {token} or position {pos}")
        return logits, int(r)

    def export_kv(self, layer: int, n_rows: int):
        """The cached K and V rows 0..n_rows-1 of one layer, [H][n_rows][D] each."""
        H, D = self.cfg.n_head, self.cfg.n_embd // self.cfg.n_head
        k = np.empty((H, n_rows, D), np.float32)
        v = np.empty((H, n_rows, D), np.float32)
        if self._lib.orc_export_kv(self._m, layer, n_rows, _p(k), _p(v)) != 0:
            raise ValueError("oracle: bad layer or row count")
        return k, v

    def reset(self):
        self._lib.orc_reset(self._m)

    def close(self):
        if self._m:
            self._lib.orc_destroy(self._m)
            self._m = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward_full(cfg, weights: dict, tokens) -> np.ndarray:
    tokens = np.ascontiguousarray(tokens, np.int32)
    c = _cfg_struct(cfg)
    h = _WeightsHolder(cfg, weights)
    out = np.empty((tokens.size, cfg.vocab_size), np.float32)
    r = lib().orc_forward_full(ctypes.byref(c), ctypes.byref(h.w), _p(tokens), tokens.size, _p(out))
    if r < 0:
        raise ValueError("oracle: bad input to forward_full")
    return out


def greedy(cfg, weights: dict, prompt, n_steps: int, teacher=None, temperature: float = 0.0, seed: int = 0,
           omp: bool = False, kv: str = "f32"):
    """Prefill the prompt one token at a time (positions 0..n-1), then run
    ``n_steps`` decode passes.  Returns (ids, logits): ids[i] is the token
    chosen after pass n-1+i (so ids has n_steps + 1 entries): the greedy
    argmax, or with temperature > 0 the draw of sample(); logits has one row
    per pass (n + n_steps rows).  Decode pass i consumes ids[i], or
    teacher[i] when ``teacher`` is given (teacher forcing).  kv: the cache's
    element type (OracleModel)."""
    m = OracleModel(cfg, weights, omp=omp, kv=kv)
    try:
        prompt = [int(t) for t in prompt]
        rows = []
        last = None
        for pos, t in enumerate(prompt):
            logits, last = m.forward(t, pos)
            rows.append(logits)
        if temperature > 0:
            last = sample(rows[-1], temperature, seed, len(prompt) - 1)
        ids = [last]
        pos = len(prompt)
        for i in range(n_steps):
            feed = ids[-1] if teacher is None else int(teacher[i])
            logits, last = m.forward(feed, pos)
            if temperature > 0:
                last = sample(logits, temperature, seed, pos)
            rows.append(logits)
            ids.append(last)
            pos += 1
        return ids, np.stack(rows)
    finally:
        m.close()
