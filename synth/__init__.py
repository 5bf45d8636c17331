"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This package holds none of the method's arithmetic: it turns (seed, element
index) into numbers (``synth.c``) and assembles the input buffers of each
workload (``workloads.py``).  Both the CPU oracle and the CUDA path receive
the very same bytes from here.

bf16 arrays are carried as numpy ``uint16`` (raw bits).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            lib.synth_h.argtypes = [u64, u64]
            lib.synth_h.restype = u64
            lib.synth_u64.argtypes = [u64, i64, p]
            lib.synth_uniform_f32.argtypes = [u64, i64, ctypes.c_double, ctypes.c_double, p]
            lib.synth_uniform_f64.argtypes = [u64, i64, p]
            lib.synth_normal_bf16.argtypes = [u64, i64, p]
            lib.synth_normal_f32.argtypes = [u64, i64, p]
            lib.synth_int_below.argtypes = [u64, i64, u64, i64, p]
            lib.synth_bernoulli_u8.argtypes = [u64, i64, ctypes.c_double, p]
            lib.synth_permutation_prefix.argtypes = [u64, i64, i64, p, p]
            for f in (lib.synth_u64, lib.synth_uniform_f32, lib.synth_uniform_f64, lib.synth_normal_bf16,
                      lib.synth_normal_f32, lib.synth_int_below, lib.synth_bernoulli_u8,
                      lib.synth_permutation_prefix):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def stream_seed(seed: int, tag: int) -> int:
    """Seed of an independent sub-stream ``tag`` of ``seed``."""
    return int(_load().synth_h(seed & 0xFFFFFFFFFFFFFFFF, tag & 0xFFFFFFFFFFFFFFFF))


def h(seed: int, i: int) -> int:
    return int(_load().synth_h(seed, i))


def u64(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_u64(seed, n, _ptr(out))
    return out


def uniform_f32(seed: int, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_uniform_f32(seed, out.size, lo, hi, _ptr(out))
    return out


def uniform_f64(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_uniform_f64(seed, n, _ptr(out))
    return out


def normal_bf16(seed: int, shape) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    _load().synth_normal_bf16(seed, out.size, _ptr(out))
    return out


def normal_f32(seed: int, shape) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_normal_f32(seed, out.size, _ptr(out))
    return out


def int_below(seed: int, n: int, n_range: int, lo: int = 0) -> np.ndarray:
    if not (1 <= n_range <= 1 << 32):
        raise ValueError("n_range must be in [1, 2^32]")
    out = np.empty(n, np.int64)
    _load().synth_int_below(seed, n, n_range, lo, _ptr(out))
    return out


def bernoulli_u8(seed: int, shape, p: float) -> np.ndarray:
    out = np.empty(shape, np.uint8)
    _load().synth_bernoulli_u8(seed, out.size, p, _ptr(out))
    return out


def permutation_prefix(seed: int, n_total: int, n_out: int) -> np.ndarray:
    if not (0 <= n_out <= n_total < 1 << 31):
        raise ValueError("need 0 <= n_out <= n_total < 2^31")
    work = np.empty(max(n_total, 1), np.int32)
    out = np.empty(n_out, np.int32)
    _load().synth_permutation_prefix(seed, n_total, n_out, _ptr(work), _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
