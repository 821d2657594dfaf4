"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

The arrays come from a counter-based generator in ``synth.c`` (SplitMix64 ->
uniform -> Box-Muller; Student-t as Z / sqrt(chi^2_d / d)).  The module draws
numbers only; it holds none of the quantization or GEMM arithmetic, so the
CPU oracle and the CUDA library can both be fed from it without sharing code.

Inputs are returned as numpy arrays: float32, or uint16 holding bf16 bit
patterns (round to nearest even from the float32 value).
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

F32 = "f32"
BF16 = "bf16"


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
             "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_fill.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_int]
            lib.synth_fill.restype = ctypes.c_int
            lib.synth_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_void_p]
            lib.synth_uniform.restype = None
            _lib = lib
    return _lib


def _fill(seed, dist, p0, p1, shape, dtype, start=0):
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = int(np.prod(shape)) if shape else 1
    if dtype == F32:
        out = np.empty(shape, dtype=np.float32)
        kind = 0
    elif dtype == BF16:
        out = np.empty(shape, dtype=np.uint16)
        kind = 1
    else:
        raise ValueError(f"dtype must be 'f32' or 'bf16', got {dtype!r}")
    rc = _load().synth_fill(int(seed) & (2**64 - 1), dist, float(p0), float(p1), int(start), n,
                            out.ctypes.data, kind)
    if rc != 0:
        raise ValueError("synth_fill rejected its arguments")
    return out


def normal(seed: int, shape, mean: float = 0.0, std: float = 1.0, dtype: str = F32,
           start: int = 0) -> np.ndarray:
    """N(mean, std^2) draws (std is the standard deviation)."""
    return _fill(seed, 0, mean, std, shape, dtype, start)


def student_t(seed: int, shape, df: int = 3, scale: float = 1.0, dtype: str = F32,
              start: int = 0) -> np.ndarray:
    """scale * Student-t(df) draws, df an integer in [1, 64]."""
    return _fill(seed, 1, df, scale, shape, dtype, start)


def uniform(seed: int, n: int, start: int = 0) -> np.ndarray:
    """The raw (0, 1) uniform stream behind every draw (for checking the generator)."""
    out = np.empty(int(n), dtype=np.float64)
    _load().synth_uniform(int(seed) & (2**64 - 1), int(start), int(n), out.ctypes.data)
    return out


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: the bits move up 16 places)."""
    return (u16.astype(np.uint32) << 16).view(np.float32)
