"""Seeded synthetic inputs shared by the oracle harness and the GPU harness.

The C++ generator in ``synth.cpp`` draws every value from a counter-based stream
(SplitMix64 + Box-Muller), so element ``i`` of tensor ``tid`` under ``seed`` is a pure
function of the three.  This module only builds and loads that library and wraps its
calls in numpy; it holds none of the decode step's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cpp")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` in place (plain g++, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            L.synth_set_threads.argtypes = [ctypes.c_int]
            L.synth_normal_f32.argtypes = [u64, u64, u64, u64, f64, f64, vp]
            L.synth_normal_bf16.argtypes = [u64, u64, u64, u64, f64, f64, vp]
            L.synth_uniform_i32.argtypes = [u64, u64, u64, i64, i64, vp]
            L.synth_q8_0.argtypes = [u64, u64, u64, u64, f64, vp]
            L.synth_q4_k.argtypes = [u64, u64, u64, u64, f64, vp]
            L.synth_pack_q8_0.argtypes = [vp, u64, vp]
            L.synth_pack_q4_k.argtypes = [vp, u64, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def set_threads(n: int) -> None:
    lib().synth_set_threads(int(n))


def normal_f32(seed: int, tid: int, n: int, mean: float = 0.0, std: float = 1.0,
               offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(seed, tid, offset, n, mean, std, _ptr(out))
    return out


def normal_bf16(seed: int, tid: int, n: int, mean: float = 0.0, std: float = 1.0,
                offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of the values ``normal_f32`` gives for the same stream."""
    out = np.empty(n, dtype=np.uint16)
    lib().synth_normal_bf16(seed, tid, offset, n, mean, std, _ptr(out))
    return out


def uniform_i32(seed: int, tid: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().synth_uniform_i32(seed, tid, n, lo, hi, _ptr(out))
    return out


Q8_0_BLOCK, Q8_0_BYTES = 32, 34
Q4_K_BLOCK, Q4_K_BYTES = 256, 144


def q8_0(seed: int, tid: int, rows: int, cols: int, std: float) -> np.ndarray:
    """``rows x cols`` N(0, std^2) weights as ggml Q8_0 rows: uint8 ``[rows, cols/32*34]``."""
    assert cols % Q8_0_BLOCK == 0
    out = np.empty((rows, cols // Q8_0_BLOCK * Q8_0_BYTES), dtype=np.uint8)
    lib().synth_q8_0(seed, tid, rows, cols, std, _ptr(out))
    return out


def q4_k(seed: int, tid: int, rows: int, cols: int, std: float) -> np.ndarray:
    """``rows x cols`` N(0, std^2) weights as ggml Q4_K rows: uint8 ``[rows, cols/256*144]``."""
    assert cols % Q4_K_BLOCK == 0
    out = np.empty((rows, cols // Q4_K_BLOCK * Q4_K_BYTES), dtype=np.uint8)
    lib().synth_q4_k(seed, tid, rows, cols, std, _ptr(out))
    return out


def pack_q8_0(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size % Q8_0_BLOCK == 0
    out = np.empty(x.size // Q8_0_BLOCK * Q8_0_BYTES, dtype=np.uint8)
    lib().synth_pack_q8_0(_ptr(x), x.size, _ptr(out))
    return out


def pack_q4_k(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size % Q4_K_BLOCK == 0
    out = np.empty(x.size // Q4_K_BLOCK * Q4_K_BYTES, dtype=np.uint8)
    lib().synth_pack_q4_k(_ptr(x), x.size, _ptr(out))
    return out
