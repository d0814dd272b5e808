"""Python handle on the CPU oracle -- TEST INFRASTRUCTURE ONLY.

The oracle (``fq_oracle.cpp``) is a plain f64 C++ restatement of the Qwen3 decode step as
the fucina pages define it.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never does.
This file compiles the library in place and marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fq_oracle.cpp")
_HDR = os.path.join(_HERE, "fq_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q8_0, Q4_K, F32 = 0, 1, 2
WTYPES = {"q8_0": Q8_0, "q4_k": Q4_K}
KV_TYPES = {"f32": 0, "bf16": 1, "q8_0": 2}
OK, INVALID_CONFIG, INVALID_SEQUENCE_LENGTH, KV_CACHE_OVERFLOW, MISMATCHED_KV_CACHES, INVALID_ARGUMENT = range(6)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("vocab", "hidden", "ffn", "layers", "n_q", "n_kv", "head_dim")] + \
               [("eps", ctypes.c_double), ("theta", ctypes.c_double)] + \
               [(n, ctypes.c_int) for n in ("n_exp", "n_used", "moe_ffn", "norm_topk", "wtype", "kv_type")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, f64, u16, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_uint16, ctypes.c_size_t
            sig = {
                "or_set_threads": ([i32], i32),
                "or_fp16_to_f64": ([u16], f64), "or_f64_to_fp16": ([f64], u16),
                "or_bf16_to_f64": ([u16], f64), "or_f64_to_bf16": ([f64], u16),
                "or_f64_to_f32": ([f64], ctypes.c_float),
                "or_dequant_q8_0": ([vp, sz, vp], None), "or_quant_q8_0": ([vp, sz, vp], None),
                "or_q4k_scale_min": ([vp, i32, vp, vp], None), "or_q4k_pack_scale_min": ([vp, vp, vp], None),
                "or_dequant_q4_k": ([vp, sz, vp], None), "or_quant_q4_k": ([vp, sz, vp], None),
                "or_rmsnorm": ([vp, i32, vp, f64, vp], None), "or_rope": ([vp, i32, i32, f64], None),
                "or_attention": ([vp, vp, vp, i32, i32, sz, vp], None), "or_silu": ([f64], f64),
                "or_attention_q8": ([vp, vp, vp, i32, i32, sz, vp], None),
                "or_kv_round_row": ([i32, vp, i32, vp], None),
                "or_router": ([vp, i32, i32, i32, vp, vp], None), "or_gemv": ([i32, vp, i32, i32, vp, vp], None),
                "or_validate": ([vp], i32), "or_model_new": ([vp], vp), "or_model_free": ([vp], None),
                "or_model_set_global": ([vp, vp, vp, vp], None),
                "or_model_set_layer": ([vp, i32] + [vp] * 15, None),
                "or_cache_new": ([vp, i32], vp), "or_cache_free": ([vp], None), "or_cache_len": ([vp], i32),
                "or_cache_write": ([vp, i32, i32, i32, vp, vp], i32), "or_cache_set_len": ([vp, i32], i32),
                "or_cache_keep_current": ([vp, i32], i32),
                "or_cache_read": ([vp, i32, i32, i32, vp, vp], i32),
                "or_layer_step": ([vp, i32, vp, i32, vp, vp, vp], i32),
                "or_qkv_project": ([vp, i32, vp, i32, vp, vp, vp], i32),
                "or_layer_step_route": ([vp, i32, vp, i32, vp, vp, vp, vp], i32),
                "or_decode_step": ([vp, vp, i32, i32, vp, vp, vp, vp], i32),
                "or_decode_step_batch": ([vp, vp, i32, vp, vp], i32),
                "or_forward_last_logits": ([vp, vp, i32, vp], i32),
                "or_argmax": ([vp, i32], i32),
                "or_sample": ([vp, i32, vp, vp, i32, f64], i32),
                "or_uniform24": ([ctypes.c_uint64, ctypes.c_uint64], f64),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous numpy arrays"
    return a.ctypes.data


def set_threads(n: int = 0) -> int:
    return lib().or_set_threads(int(n))


# ---------------------------------------------------------------- codecs and blocks

def fp16_to_f64(h: int) -> float:
    return lib().or_fp16_to_f64(h)


def f64_to_fp16(v: float) -> int:
    return lib().or_f64_to_fp16(v)


def bf16_to_f64(h: int) -> float:
    return lib().or_bf16_to_f64(h)


def f64_to_bf16(v: float) -> int:
    return lib().or_f64_to_bf16(v)


def dequant(wtype: str, packed: np.ndarray, n: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(n, dtype=np.float32)
    if wtype == "q8_0":
        lib().or_dequant_q8_0(_p(packed), n, _p(out))
    elif wtype == "q4_k":
        lib().or_dequant_q4_k(_p(packed), n, _p(out))
    else:
        raise ValueError(wtype)
    return out


def quant(wtype: str, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    if wtype == "q8_0":
        out = np.empty(x.size // 32 * 34, dtype=np.uint8)
        lib().or_quant_q8_0(_p(x), x.size, _p(out))
    elif wtype == "q4_k":
        out = np.empty(x.size // 256 * 144, dtype=np.uint8)
        lib().or_quant_q4_k(_p(x), x.size, _p(out))
    else:
        raise ValueError(wtype)
    return out


def q4k_scale_min(s12: np.ndarray, j: int):
    s12 = np.ascontiguousarray(s12, dtype=np.uint8)
    sc, mn = ctypes.c_int(), ctypes.c_int()
    lib().or_q4k_scale_min(_p(s12), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def q4k_pack_scale_min(sc, mn) -> np.ndarray:
    sc = np.ascontiguousarray(sc, dtype=np.int32)
    mn = np.ascontiguousarray(mn, dtype=np.int32)
    out = np.zeros(12, dtype=np.uint8)
    lib().or_q4k_pack_scale_min(_p(sc), _p(mn), _p(out))
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    lib().or_rmsnorm(_p(x), x.size, _p(g), eps, _p(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    lib().or_rope(_p(v), v.size, pos, theta)
    return v


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One head: q [D] f64, K/V [T, D] f32 -> o [D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    T, D = K.shape
    o = np.empty(D, dtype=np.float64)
    lib().or_attention(_p(q), _p(K), _p(V), T, D, D, _p(o))
    return o


def attention_q8(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One head over a q8_0 cache: q [D] f64 (quantised inside), K/V [T, D] dequantised rows."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    T, D = K.shape
    o = np.empty(D, dtype=np.float64)
    lib().or_attention_q8(_p(q), _p(K), _p(V), T, D, D, _p(o))
    return o


def kv_round_row(kv_dtype: str, x: np.ndarray) -> np.ndarray:
    """The values a cache of ``kv_dtype`` holds for one row ``x``."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.size, dtype=np.float32)
    lib().or_kv_round_row(KV_TYPES[kv_dtype], _p(x), x.size, _p(out))
    return out


def silu(z: float) -> float:
    return lib().or_silu(z)


def router(logits: np.ndarray, k: int, norm: bool = True):
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    lib().or_router(_p(logits), logits.size, k, int(norm), _p(idx), _p(w))
    return idx, w


def gemv(wtype: str, W: np.ndarray, rows: int, cols: int, x: np.ndarray) -> np.ndarray:
    t = {"q8_0": Q8_0, "q4_k": Q4_K, "f32": F32}[wtype]
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().or_gemv(t, _p(W), rows, cols, _p(x), _p(y))
    return y


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, dtype=np.float64)
    return lib().or_argmax(_p(v), v.size)


class _Sampling(ctypes.Structure):
    _fields_ = [("temp", ctypes.c_double), ("top_k", ctypes.c_int), ("top_p", ctypes.c_double),
                ("min_p", ctypes.c_double), ("repeat_penalty", ctypes.c_double)]


def sample(z: np.ndarray, u: float, temp: float = 1.0, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0,
           repeat_penalty: float = 1.0, history=()) -> int:
    """The next token from one row of logits (or_sample gives the order of the steps)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    h = np.ascontiguousarray(history, dtype=np.int32)
    s = _Sampling(temp, top_k, top_p, min_p, repeat_penalty)
    return lib().or_sample(_p(z), z.size, ctypes.byref(s), _p(h) if h.size else None, h.size, float(u))


def uniform24(seed: int, counter: int) -> float:
    """Counter-based uniform in [0, 1) on a 2^-24 grid (SplitMix64 of seed + (counter + 1) * golden)."""
    return lib().or_uniform24(seed, counter)


# ---------------------------------------------------------------- model

def make_dims(dims, wtype: str, kv_dtype: str) -> _Dims:
    return _Dims(vocab=dims.vocab_size, hidden=dims.hidden_size, ffn=dims.intermediate_size,
                 layers=dims.num_layers, n_q=dims.num_attention_heads, n_kv=dims.num_key_value_heads,
                 head_dim=dims.head_dim, eps=dims.rms_norm_eps, theta=dims.rope_theta,
                 n_exp=dims.num_experts, n_used=dims.num_experts_used, moe_ffn=dims.moe_intermediate_size,
                 norm_topk=int(dims.norm_topk_prob), wtype=WTYPES[wtype], kv_type=KV_TYPES[kv_dtype])


def validate(dims, wtype: str = "q8_0", kv_dtype: str = "bf16") -> int:
    d = make_dims(dims, wtype, kv_dtype)
    return lib().or_validate(ctypes.byref(d))


class Model:
    """Oracle model over host tensors laid out as ``synth.workloads.make_weights`` returns."""

    def __init__(self, dims, weights: dict, wtype: str, kv_dtype: str):
        self.dims, self.wtype, self.kv_dtype = dims, wtype, kv_dtype
        self._d = make_dims(dims, wtype, kv_dtype)
        self._keep = weights
        self._h = lib().or_model_new(ctypes.byref(self._d))
        if not self._h:
            raise OracleError(INVALID_CONFIG, "or_model_new")
        lib().or_model_set_global(self._h, _p(weights.get("tok_embd")), _p(weights.get("output_norm")),
                                  _p(weights.get("output")))
        for L, lw in enumerate(weights["layers"]):
            g = lambda k: _p(lw.get(k))  # noqa: E731
            lib().or_model_set_layer(self._h, L, g("attn_norm"), g("wq"), g("wk"), g("wv"), g("q_norm"),
                                     g("k_norm"), g("wo"), g("ffn_norm"), g("w_gate"), g("w_up"), g("w_down"),
                                     g("router"), g("gate_exps"), g("up_exps"), g("down_exps"))

    def __del__(self):
        if getattr(self, "_h", None):
            lib().or_model_free(self._h)
            self._h = None

    def new_cache(self, capacity: int) -> "Cache":
        return Cache(self, capacity)

    def layer_step(self, layer: int, cache: "Cache", pos: int, x: np.ndarray, router_logits: bool = False):
        """(x after the layer, expert ids, expert weights[, router logits when asked])."""
        x = np.array(x, dtype=np.float64, copy=True)
        n_used = max(self.dims.num_experts_used, 1)
        idx = np.zeros(n_used, dtype=np.int32)
        w = np.zeros(n_used, dtype=np.float64)
        rl = np.zeros(max(self.dims.num_experts, 1), dtype=np.float64) if router_logits else None
        rc = lib().or_layer_step_route(self._h, layer, cache._h, pos, _p(x), _p(idx), _p(w), _p(rl))
        if rc:
            raise OracleError(rc, "or_layer_step")
        return (x, idx, w, rl) if router_logits else (x, idx, w)

    def qkv_project(self, layer: int, xn: np.ndarray, pos: int):
        """q, k, v of one token from the normalised input xn (q, k after QK-norm and RoPE)."""
        d = self.dims
        xn = np.ascontiguousarray(xn, dtype=np.float64)
        q = np.empty((d.num_attention_heads, d.head_dim), dtype=np.float64)
        k = np.empty((d.num_key_value_heads, d.head_dim), dtype=np.float64)
        v = np.empty_like(k)
        rc = lib().or_qkv_project(self._h, layer, _p(xn), pos, _p(q), _p(k), _p(v))
        if rc:
            raise OracleError(rc, "or_qkv_project")
        return q, k, v

    def decode_step(self, cache: "Cache", token: int, pos0: int, logits: bool = True, trace: bool = False):
        d = self.dims
        lg = np.empty(d.vocab_size, dtype=np.float64) if logits else None
        lo = np.empty((d.num_layers, d.hidden_size), dtype=np.float64) if trace else None
        n_used = max(d.num_experts_used, 1)
        ri = np.zeros((d.num_layers, n_used), dtype=np.int32) if trace else None
        rw = np.zeros((d.num_layers, n_used), dtype=np.float64) if trace else None
        rc = lib().or_decode_step(self._h, cache._h, int(token), int(pos0), _p(lg), _p(lo), _p(ri), _p(rw))
        if rc:
            raise OracleError(rc, "or_decode_step")
        if trace:
            return lg, lo, ri, rw
        return lg

    def decode_step_batch(self, caches, tokens) -> np.ndarray:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        arr = (ctypes.c_void_p * len(caches))(*[c._h for c in caches])
        lg = np.empty((len(caches), self.dims.vocab_size), dtype=np.float64)
        rc = lib().or_decode_step_batch(self._h, arr, len(caches), _p(tokens), _p(lg))
        if rc:
            raise OracleError(rc, "or_decode_step_batch")
        return lg

    def forward_last_logits(self, tokens) -> np.ndarray:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        lg = np.empty(self.dims.vocab_size, dtype=np.float64)
        rc = lib().or_forward_last_logits(self._h, _p(tokens), tokens.size, _p(lg))
        if rc:
            raise OracleError(rc, "or_forward_last_logits")
        return lg


class Cache:
    def __init__(self, model: Model, capacity: int):
        self.model = model
        self._h = lib().or_cache_new(model._h, capacity)
        if not self._h:
            raise OracleError(INVALID_ARGUMENT, "or_cache_new")
        self.capacity = capacity

    def __del__(self):
        if getattr(self, "_h", None):
            lib().or_cache_free(self._h)
            self._h = None

    @property
    def len(self) -> int:
        return lib().or_cache_len(self._h)

    def set_len(self, n: int) -> None:
        rc = lib().or_cache_set_len(self._h, n)
        if rc:
            raise OracleError(rc, "or_cache_set_len")

    def keep_current(self, keep: bool) -> None:
        """While set, steps attend over the rows already written at their position (see
        `write`) instead of storing the rows they compute."""
        rc = lib().or_cache_keep_current(self._h, int(bool(keep)))
        if rc:
            raise OracleError(rc, "or_cache_keep_current")

    def write(self, layer: int, pos0: int, k: np.ndarray, v: np.ndarray) -> None:
        """k, v: [n, Hkv, D] float32 values, uint16 bf16 bit patterns, or uint8 ggml Q8_0
        blocks [n, Hkv, D / 32 * 34] (dequantised here)."""
        if k.dtype == np.uint8:
            D = self.model.dims.head_dim
            k = dequant("q8_0", k, k.size // 34 * 32).reshape(k.shape[0], k.shape[1], D)
            v = dequant("q8_0", v, v.size // 34 * 32).reshape(v.shape[0], v.shape[1], D)
        k, v = _as_f32(k), _as_f32(v)
        rc = lib().or_cache_write(self._h, layer, pos0, k.shape[0], _p(k), _p(v))
        if rc:
            raise OracleError(rc, "or_cache_write")

    def read(self, layer: int, pos0: int, n: int):
        d = self.model.dims
        k = np.empty((n, d.num_key_value_heads, d.head_dim), dtype=np.float32)
        v = np.empty_like(k)
        rc = lib().or_cache_read(self._h, layer, pos0, n, _p(k), _p(v))
        if rc:
            raise OracleError(rc, "or_cache_read")
        return k, v


def _as_f32(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return np.ascontiguousarray((a.astype(np.uint32) << 16).view(np.float32))
    return np.ascontiguousarray(a, dtype=np.float32)
