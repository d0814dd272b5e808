"""ctypes binding of the fq C ABI (``include/fq.h``): the same entry points, argument
marshalling only.  Device buffers are passed as integer addresses (``tensor.data_ptr()``)
and streams as ``torch.cuda.current_stream().cuda_stream``; every computation happens in
the CUDA library.  Loading fails loudly when ``libfq.so`` has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfq.so")
_lock = threading.Lock()
_lib = None

# fq_status
OK, INVALID_CONFIG, INVALID_SEQUENCE_LENGTH, KV_CACHE_OVERFLOW, MISMATCHED_KV_CACHES, INVALID_ARGUMENT, \
    OUT_OF_MEMORY, CUDA_ERROR, DEVICE_TIMEOUT, UNSUPPORTED = range(10)
# fq_dtype
F32, BF16, Q8_0, Q4_K = 0, 1, 8, 12
DTYPES = {"f32": F32, "bf16": BF16, "q8_0": Q8_0, "q4_k": Q4_K}
# fq_weight_id
W_TOK_EMBD, W_OUTPUT, W_Q, W_K, W_V, W_O, W_GATE, W_UP, W_DOWN, W_GATE_EXPS, W_UP_EXPS, W_DOWN_EXPS = range(12)


class FqError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status}: {message}")
        self.status = status


class fq_desc_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in ("vocab_size", "hidden_size", "intermediate_size", "num_layers",
                                               "num_attention_heads", "num_key_value_heads", "head_dim")] + \
               [("rms_norm_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
               [(n, ctypes.c_uint32) for n in ("num_experts", "num_experts_used", "moe_intermediate_size")] + \
               [("norm_topk_prob", ctypes.c_int32), ("moe_expert_top_p", ctypes.c_float),
                ("max_positions", ctypes.c_uint32)]


class fq_desc(ctypes.Structure):
    _fields_ = [("p", fq_desc_params), ("magic", ctypes.c_uint32)]


class fq_tensor(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("rows", ctypes.c_uint64), ("cols", ctypes.c_uint64),
                ("data", ctypes.c_void_p)]


_LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate", "w_up", "w_down",
                 "router", "gate_exps", "up_exps", "down_exps")


class fq_layer_src(ctypes.Structure):
    _fields_ = [(n, fq_tensor) for n in _LAYER_FIELDS]


class fq_weight_src(ctypes.Structure):
    _fields_ = [("tok_embd", fq_tensor), ("output_norm", fq_tensor), ("output", fq_tensor),
                ("layers", ctypes.POINTER(fq_layer_src))]


def lib():
    """The loaded ``libfq.so``; raises if it is missing (no fallback path exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"fq CUDA library not built ({LIB_PATH}); run quantized_decoder_decode_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            vp, u32, u64, i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32
            sig = {
                "fq_desc_init": [vp, vp],
                "fq_load_weights": [vp, vp, vp, vp],
                "fq_kv_init": [vp, u32, ctypes.c_int, vp],
                "fq_kv_append": [vp, u32, u32, u32, vp, vp, vp],
                "fq_kv_commit": [vp, u32],
                "fq_kv_rewind": [vp, u32],
                "fq_kv_read": [vp, u32, u32, u32, vp, vp, vp],
                "fq_layer_step": [vp, u32, vp, u32, vp, vp],
                "fq_decode_step": [vp, vp, i32, u32, vp, vp],
                "fq_decode_step_batch": [vp, vp, u32, vp, vp, vp],
                "fq_decode_step_all_logits": [vp, vp, vp, u32, u32, vp, vp],
                "fq_forward_step": [vp, vp, vp, u32, u32, vp, vp],
                "fq_decode_greedy": [vp, vp, u32, vp, u32, vp, vp, vp],
                "fq_decode_step_trace": [vp, vp, u32, vp, vp, vp, vp, vp, vp, vp],
                "fq_dequant_rows": [vp, u32, ctypes.c_int, u64, u64, vp, vp],
                "fq_quantize_q8_0": [vp, u64, vp, vp],
                "fq_layer_step_trace": [vp, u32, vp, u32, vp, vp, vp, vp, vp],
                "fq_gemv": [vp, u32, ctypes.c_int, u32, vp, vp, vp],
                "fq_check_device": [vp, vp],
                "fq_debug_wait_timeout": [vp, vp],
                "fq_set_option": [vp, ctypes.c_int, ctypes.c_int],
                "fq_step_path": [vp, u32, ctypes.c_int, ctypes.POINTER(ctypes.c_int)],
                "fq_step_kernels": [vp, vp, ctypes.POINTER(ctypes.c_uint32)],
                "fq_layer_step_noalloc": [vp, u32, vp, u32, vp, vp],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.fq_model_free.argtypes = [vp]
            L.fq_model_free.restype = None
            L.fq_kv_free.argtypes = [vp]
            L.fq_kv_free.restype = None
            L.fq_kv_len.argtypes = [vp]
            L.fq_kv_len.restype = u32
            L.fq_kv_capacity.argtypes = [vp]
            L.fq_kv_capacity.restype = u32
            L.fq_last_error.argtypes = []
            L.fq_last_error.restype = ctypes.c_char_p
            L.fq_status_str.argtypes = [ctypes.c_int]
            L.fq_status_str.restype = ctypes.c_char_p
            _lib = L
    return _lib


EXPORTED = ("fq_desc_init", "fq_load_weights", "fq_model_free", "fq_kv_init", "fq_kv_free", "fq_kv_len",
            "fq_kv_capacity", "fq_kv_append", "fq_kv_commit", "fq_kv_rewind", "fq_kv_read", "fq_layer_step", "fq_decode_step",
            "fq_decode_step_batch", "fq_decode_step_all_logits", "fq_forward_step", "fq_decode_greedy", "fq_decode_step_trace", "fq_dequant_rows", "fq_quantize_q8_0", "fq_layer_step_trace",
            "fq_gemv", "fq_step_kernels", "fq_check_device", "fq_debug_wait_timeout", "fq_set_option", "fq_step_path", "fq_layer_step_noalloc", "fq_last_error",
            "fq_status_str")


def _check(status: int, where: str) -> None:
    if status != OK:
        raise FqError(status, where, lib().fq_last_error().decode(errors="replace"))


# ---------------------------------------------------------------- entry points

def fq_desc_init(**params) -> fq_desc:
    """Validate a Config (keyword fields of ``fq_desc_params``) into a descriptor."""
    p = fq_desc_params(rms_norm_eps=1e-6, rope_theta=1e6, norm_topk_prob=1, moe_expert_top_p=1.0)
    for k, v in params.items():
        setattr(p, k, v)
    d = fq_desc()
    _check(lib().fq_desc_init(ctypes.byref(d), ctypes.byref(p)), "fq_desc_init")
    return d


def _tensor(arr, dtype: int, rows: int, cols: int) -> fq_tensor:
    if arr is None:
        return fq_tensor(dtype, 0, 0, None)
    assert isinstance(arr, np.ndarray) and arr.flags["C_CONTIGUOUS"]
    return fq_tensor(dtype, rows, cols, arr.ctypes.data)


def weight_src(desc: fq_desc, weights: dict, wdtype: str):
    """Build ``fq_weight_src`` over host numpy tensors laid out like the GGUF tensors
    (the dict shape ``synth.workloads.make_weights`` returns).  Returns (src, keepalive)."""
    p = desc.p
    q = DTYPES[wdtype]
    H, D, Hq, Hkv = p.hidden_size, p.head_dim, p.num_attention_heads, p.num_key_value_heads
    layers = (fq_layer_src * p.num_layers)()
    for L, lw in enumerate(weights["layers"]):
        t = layers[L]
        t.attn_norm = _tensor(lw["attn_norm"], F32, 1, H)
        t.ffn_norm = _tensor(lw["ffn_norm"], F32, 1, H)
        t.q_norm = _tensor(lw["q_norm"], F32, 1, D)
        t.k_norm = _tensor(lw["k_norm"], F32, 1, D)
        t.wq = _tensor(lw["wq"], q, Hq * D, H)
        t.wk = _tensor(lw["wk"], q, Hkv * D, H)
        t.wv = _tensor(lw["wv"], q, Hkv * D, H)
        t.wo = _tensor(lw["wo"], q, H, Hq * D)
        if p.num_experts:
            E, Fe = p.num_experts, p.moe_intermediate_size
            t.router = _tensor(lw["router"], F32, E, H)
            t.gate_exps = _tensor(lw["gate_exps"], q, E * Fe, H)
            t.up_exps = _tensor(lw["up_exps"], q, E * Fe, H)
            t.down_exps = _tensor(lw["down_exps"], q, E * H, Fe)
        else:
            F = p.intermediate_size
            t.w_gate = _tensor(lw["w_gate"], q, F, H)
            t.w_up = _tensor(lw["w_up"], q, F, H)
            t.w_down = _tensor(lw["w_down"], q, H, F)
    src = fq_weight_src()
    src.tok_embd = _tensor(weights.get("tok_embd"), q, p.vocab_size, H)
    src.output_norm = _tensor(weights.get("output_norm"), F32, 1, H)
    src.output = _tensor(weights.get("output"), q, p.vocab_size, H)
    src.layers = layers
    return src, (weights, layers)


def fq_load_weights(desc: fq_desc, src: fq_weight_src, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(lib().fq_load_weights(ctypes.byref(desc), ctypes.byref(src), stream, ctypes.byref(out)), "fq_load_weights")
    return out.value


def fq_model_free(model: int) -> None:
    lib().fq_model_free(model)


def fq_kv_init(model: int, capacity: int, kv_dtype: str = "bf16") -> int:
    out = ctypes.c_void_p()
    _check(lib().fq_kv_init(model, capacity, DTYPES[kv_dtype], ctypes.byref(out)), "fq_kv_init")
    return out.value


def fq_kv_free(kv: int) -> None:
    lib().fq_kv_free(kv)


def fq_kv_len(kv: int) -> int:
    return lib().fq_kv_len(kv)


def fq_kv_capacity(kv: int) -> int:
    return lib().fq_kv_capacity(kv)


def fq_kv_append(kv: int, layer: int, pos: int, n_pos: int, k_ptr: int, v_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_kv_append(kv, layer, pos, n_pos, k_ptr, v_ptr, stream), "fq_kv_append")


def fq_kv_commit(kv: int, length: int) -> None:
    _check(lib().fq_kv_commit(kv, length), "fq_kv_commit")


def fq_kv_rewind(kv: int, length: int) -> None:
    _check(lib().fq_kv_rewind(kv, length), "fq_kv_rewind")


def fq_kv_read(kv: int, layer: int, pos: int, n_pos: int, k_ptr: int, v_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_kv_read(kv, layer, pos, n_pos, k_ptr, v_ptr, stream), "fq_kv_read")


def fq_layer_step(model: int, layer: int, kv: int, pos: int, x_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_layer_step(model, layer, kv, pos, x_ptr, stream), "fq_layer_step")


def fq_decode_step(model: int, kv: int, token: int, pos0: int, logits_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_decode_step(model, kv, token, pos0, logits_ptr, stream), "fq_decode_step")


def _caches(kvs):
    return (ctypes.c_void_p * len(kvs))(*kvs)


def _i32(v):
    a = np.ascontiguousarray(v, dtype=np.int32)
    return a, a.ctypes.data


def fq_decode_step_batch(model: int, kvs, tokens, logits_ptr: int, stream: int = 0) -> None:
    toks, tp = _i32(tokens)
    _check(lib().fq_decode_step_batch(model, _caches(kvs), len(kvs), tp, logits_ptr, stream), "fq_decode_step_batch")


def fq_forward_step(model: int, kv: int, tokens, pos0: int, logits_ptr: int = 0, stream: int = 0) -> None:
    """forwardStep over len(tokens) tokens of one sequence at pos0..: the last row's logits
    ([vocab], device) or, with logits_ptr 0, only the K/V appends (a prefill at pos0 = 0)."""
    toks, tp = _i32(tokens)
    _check(lib().fq_forward_step(model, kv, tp, len(toks), pos0, logits_ptr or None, stream), "fq_forward_step")


def fq_decode_step_all_logits(model: int, kv: int, tokens, pos0: int, logits_ptr: int, stream: int = 0) -> None:
    """All rows' logits ([len][vocab], device) for len tokens of one sequence at pos0.."""
    toks, tp = _i32(tokens)
    _check(lib().fq_decode_step_all_logits(model, kv, tp, len(toks), pos0, logits_ptr, stream),
           "fq_decode_step_all_logits")


def fq_decode_greedy(model: int, kvs, first_tokens, n_steps: int, tokens_out_ptr: int, logits_ptr: int = 0,
                     stream: int = 0) -> None:
    toks, tp = _i32(first_tokens)
    _check(lib().fq_decode_greedy(model, _caches(kvs), len(kvs), tp, n_steps, tokens_out_ptr, logits_ptr or None,
                                  stream), "fq_decode_greedy")


def fq_decode_step_trace(model: int, kvs, tokens, logits_ptr: int, layer_out_ptr: int = 0, route_idx_ptr: int = 0,
                         route_w_ptr: int = 0, stream: int = 0, route_logits_ptr: int = 0) -> None:
    toks, tp = _i32(tokens)
    _check(lib().fq_decode_step_trace(model, _caches(kvs), len(kvs), tp, logits_ptr or None, layer_out_ptr or None,
                                      route_idx_ptr or None, route_w_ptr or None, route_logits_ptr or None, stream),
           "fq_decode_step_trace")


def fq_dequant_rows(model: int, layer: int, which: int, row0: int, n_rows: int, out_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_dequant_rows(model, layer, which, row0, n_rows, out_ptr, stream), "fq_dequant_rows")


def fq_quantize_q8_0(x_ptr: int, n: int, blocks_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_quantize_q8_0(x_ptr, n, blocks_ptr, stream), "fq_quantize_q8_0")


def fq_layer_step_trace(model: int, layer: int, kv: int, pos: int, x_ptr: int, qkv_ptr: int = 0, attn_ptr: int = 0,
                        ffn_ptr: int = 0, stream: int = 0) -> None:
    _check(lib().fq_layer_step_trace(model, layer, kv, pos, x_ptr, qkv_ptr or None, attn_ptr or None, ffn_ptr or None,
                                     stream), "fq_layer_step_trace")


def fq_gemv(model: int, layer: int, which: int, n: int, x_ptr: int, y_ptr: int, stream: int = 0) -> None:
    _check(lib().fq_gemv(model, layer, which, n, x_ptr, y_ptr, stream), "fq_gemv")


def fq_step_kernels(model: int, stream: int = 0) -> int:
    """Kernels per step of the CUDA graph last replayed on `stream` (0 if none)."""
    out = ctypes.c_uint32(0)
    _check(lib().fq_step_kernels(model, stream, ctypes.byref(out)), "fq_step_kernels")
    return int(out.value)


def fq_check_device(model: int, stream: int = 0) -> None:
    _check(lib().fq_check_device(model, stream), "fq_check_device")


OPT_STEP_PATH, OPT_DEPENDENT_LAUNCH, OPT_GRAPHS, OPT_TENSOR_CORES = range(4)
PATH_AUTO, PATH_KERNELS = 0, 1


def fq_set_option(model: int, opt: int, value: int) -> None:
    _check(lib().fq_set_option(model, opt, int(value)), "fq_set_option")


def fq_step_path(model: int, n: int, kv_dtype: str) -> bool:
    """True when a step of n sequences with a kv_dtype cache runs as the streamed kernel."""
    out = ctypes.c_int(0)
    _check(lib().fq_step_path(model, n, DTYPES[kv_dtype], ctypes.byref(out)), "fq_step_path")
    return bool(out.value)


def fq_debug_wait_timeout(model: int, stream: int = 0) -> None:
    """Test hook: make every bounded wait of one LM-head GEMV launch run out."""
    _check(lib().fq_debug_wait_timeout(model, stream), "fq_debug_wait_timeout")


def fq_layer_step_noalloc(model: int, layer: int, kv: int, pos: int, x_ptr: int, stream: int = 0) -> None:
    """fq_layer_step without any device allocation (scratch lives in a built-in array)."""
    _check(lib().fq_layer_step_noalloc(model, layer, kv, pos, x_ptr, stream), "fq_layer_step_noalloc")
