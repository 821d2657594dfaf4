"""CPU oracle (test infrastructure only).

A plain, slow, obviously correct CPU implementation of the quantize and GEMM
steps, in C++ (``oracle.cpp``), driven from numpy through ctypes.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the CUDA library never does, and the two share no code.

Functions follow the pages on the subject (AstrAI ``ops/fp8.py``: the CPU
kernels of ``custom::fp8_quantize`` and ``custom::fp8_gemm``; the POPCORNBENCH
``Kimi-K2.6 l2_p13`` trace: INT8 absmax/127 quantization with round-half-even;
the scmp_kernels README: per-row and per-head granularity).  Every function is
pinned by ``tests/test_oracle_*.py`` against values that the pages print,
closed forms, library routines and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3, E5M2 = 0, 1
NT, NN, TN = 0, 1, 2
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source: -O2, OpenMP, no FMA contraction."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
             "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            L.or_fp8_decode.argtypes = [ctypes.c_uint8, i32]
            L.or_fp8_decode.restype = ctypes.c_double
            L.or_fp8_encode_array.argtypes = [vp, i64, i32, vp]
            L.or_fp8_encode_array.restype = i32
            L.or_fp8_code_is_nan.argtypes = [ctypes.c_uint8, i32]
            L.or_fp8_code_is_nan.restype = i32
            L.or_round_half_even.argtypes = [f32]
            L.or_round_half_even.restype = ctypes.c_int32
            L.or_bf16_round.argtypes = [f32]
            L.or_bf16_round.restype = ctypes.c_uint16
            L.or_quantize_rowwise_i8.argtypes = [vp, i32, i64, i64, i64, vp, vp]
            L.or_quantize_rowwise_i8.restype = i32
            L.or_quantize_fp8.argtypes = [vp, i64, f32, i32, vp, vp]
            L.or_quantize_fp8.restype = i32
            L.or_quantize_fp8_ring.argtypes = [vp, i64, i32, vp, vp, vp, i64, i64, i32]
            L.or_quantize_fp8_ring.restype = i32
            L.or_gemm_i8.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64, vp, vp]
            L.or_gemm_i8.restype = i32
            L.or_gemm_fp8.argtypes = [vp, vp, i32, i32, i64, i64, i64, f32, f32, vp, i64, vp, vp]
            L.or_gemm_fp8.restype = i32
            L.or_gemm_fp8_e4m3.argtypes = [vp, vp, i32, i32, i64, i64, i64, f32, f32, f32, vp, i64,
                                           vp, vp]
            L.or_gemm_fp8_e4m3.restype = i32
            L.or_quantize_grouped_i8.argtypes = [vp, i32, i64, i64, i64, i64, vp, vp]
            L.or_quantize_grouped_i8.restype = i32
            L.or_gemm_i8_grouped.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64,
                                             vp, vp]
            L.or_gemm_i8_grouped.restype = i32
            L.or_gemm_fp8_bias.argtypes = [vp, vp, i32, i32, i64, i64, i64, f32, f32, vp, vp, i64,
                                           vp, vp]
            L.or_gemm_fp8_bias.restype = i32
            L.or_fp8_bias_to_f32.argtypes = [vp, i64, i32, f32, vp]
            L.or_fp8_bias_to_f32.restype = i32
            L.or_colsum_bf16.argtypes = [vp, i64, i64, vp]
            L.or_colsum_bf16.restype = i32
            L.or_num_threads.argtypes = []
            L.or_num_threads.restype = i32
            L.or_set_num_threads.argtypes = [i32]
            L.or_set_num_threads.restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def num_threads() -> int:
    return int(_load().or_num_threads())


def set_num_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops (for timing it on one core)."""
    _load().or_set_num_threads(int(n))


# ------------------------------------------------------------------ codec
def fp8_decode(code: int, fmt: int) -> float:
    return float(_load().or_fp8_decode(int(code) & 0xFF, int(fmt)))


def fp8_decode_table(fmt: int) -> np.ndarray:
    """The 256 decoded values (NaN for NaN codes) as float64."""
    return np.array([fp8_decode(c, fmt) for c in range(256)], dtype=np.float64)


def fp8_code_is_nan(code: int, fmt: int) -> bool:
    return bool(_load().or_fp8_code_is_nan(int(code) & 0xFF, int(fmt)))


def fp8_encode(t, fmt: int) -> np.ndarray:
    """float32 -> FP8 codes (RNE, saturating to the largest finite value)."""
    t = np.asarray(t, dtype=np.float32)
    shape = t.shape
    t = _c(t.reshape(-1), np.float32)
    out = np.empty(t.shape, dtype=np.uint8)
    if _load().or_fp8_encode_array(_ptr(t), t.size, int(fmt), _ptr(out)) != 0:
        raise ValueError("bad fp8 format")
    return out.reshape(shape)


def round_half_even(t: float) -> int:
    return int(_load().or_round_half_even(float(np.float32(t))))


def bf16_round(f: float) -> int:
    return int(_load().or_bf16_round(float(np.float32(f))))


# ------------------------------------------------------------------ quantize
def quantize_rowwise_i8(x: np.ndarray, dtype: int = F32):
    """Per-row symmetric INT8 of a 2-D (or batched 3-D, per head) array.

    x: float32 values (dtype=F32) or uint16 bf16 bits (dtype=BF16), last axis
    is the row.  Returns (q int8 same shape, scales float32 of shape[:-1]).
    """
    x = np.ascontiguousarray(x)
    if dtype == F32 and x.dtype != np.float32:
        raise TypeError("F32 input must be float32")
    if dtype == BF16 and x.dtype != np.uint16:
        raise TypeError("BF16 input must be uint16 bit patterns")
    cols = x.shape[-1]
    rows = x.size // cols if cols else 0
    q = np.empty(x.shape, dtype=np.int8)
    s = np.empty(x.shape[:-1], dtype=np.float32)
    if _load().or_quantize_rowwise_i8(_ptr(x), int(dtype), rows, cols, cols, _ptr(q), _ptr(s)) != 0:
        raise ValueError("bad arguments")
    return q, s


def quantize_grouped_i8(x: np.ndarray, group_rows: int, dtype: int = F32):
    """Row-group INT8 of a 2-D array (groups of group_rows consecutive rows;
    group_rows >= rows is per tensor).  Returns (q, scales[ceil(rows/g)])."""
    x = np.ascontiguousarray(x)
    if (dtype == F32 and x.dtype != np.float32) or (dtype == BF16 and x.dtype != np.uint16):
        raise TypeError("dtype mismatch")
    rows, cols = x.shape
    q = np.empty(x.shape, dtype=np.int8)
    s = np.empty((rows + group_rows - 1) // group_rows, dtype=np.float32)
    if _load().or_quantize_grouped_i8(_ptr(x), int(dtype), rows, cols, cols, int(group_rows),
                                      _ptr(q), _ptr(s)) != 0:
        raise ValueError("bad arguments")
    return q, s


def gemm_i8_grouped(A, B, sa, sb, ga: int, gb: int, rows=None):
    """C[b] = A[b] B[b]^T with row-group scales sa[b][i // ga], sb[b][j // gb].
    A, B 2-D or 3-D int8; sa, sb flat per batch.  Returns (acc, C)."""
    A = _c(A, np.int8)
    B = _c(B, np.int8)
    batched = A.ndim == 3
    if not batched:
        A, B = A[None], B[None]
    nb, M, K = A.shape
    N = B.shape[1]
    sa = _c(np.asarray(sa, dtype=np.float32).reshape(-1), np.float32)
    sb = _c(np.asarray(sb, dtype=np.float32).reshape(-1), np.float32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    acc = np.empty((nb, nr, N), dtype=np.int32)
    C = np.empty((nb, nr, N), dtype=np.float32)
    rc = _load().or_gemm_i8_grouped(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), int(ga), int(gb), nb,
                                    M, N, K, _ptr(r), nr, _ptr(acc), _ptr(C))
    if rc < 0:
        raise ValueError("bad arguments")
    if rc == 1:
        raise OverflowError("an exact INT8 accumulator does not fit int32")
    return (acc, C) if batched else (acc[0], C[0])


def quantize_fp8(x_bf16: np.ndarray, scale: float, fmt: int):
    """Per-tensor FP8 of bf16 bits with the scale divided out.  Returns (x8, amax)."""
    x = _c(x_bf16, np.uint16)
    x8 = np.empty(x.shape, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    if _load().or_quantize_fp8(_ptr(x), x.size, float(np.float32(scale)), int(fmt),
                               _ptr(x8), _ptr(amax)) != 0:
        raise ValueError("bad arguments")
    return x8, np.float32(amax[0])


def quantize_fp8_ring(x_bf16: np.ndarray, fmt: int, ring: np.ndarray, idx: int, margin: int = 0):
    """Delayed-scaling quantize: uses ring[H] as the step, records the amax in
    ring[idx] and publishes the next step in ring[H] (in place).
    ring = float32[H + 2] laid out [hist | scale | counter].  Returns (x8, amax)."""
    x = _c(x_bf16, np.uint16)
    if ring.dtype != np.float32 or not ring.flags.c_contiguous or ring.size < 3:
        raise TypeError("ring must be a contiguous float32 array of H + 2 entries")
    H = ring.size - 2
    x8 = np.empty(x.shape, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    if _load().or_quantize_fp8_ring(_ptr(x), x.size, int(fmt), _ptr(x8), _ptr(amax), _ptr(ring),
                                    H, int(idx), int(margin)) != 0:
        raise ValueError("bad arguments")
    return x8, np.float32(amax[0])


# ------------------------------------------------------------------ GEMMs
def gemm_i8(A, B, sa=None, sb=None, rows=None):
    """C[b] = A[b] B[b]^T on int8 codes (2-D or batched 3-D).

    Returns (acc int32, C float32 or None).  rows selects output rows of every
    batch (None = all).  Raises OverflowError if an exact sum leaves int32.
    """
    A = _c(A, np.int8)
    B = _c(B, np.int8)
    batched = A.ndim == 3
    if not batched:
        A, B = A[None], B[None]
        if sa is not None:
            sa, sb = np.asarray(sa)[None], np.asarray(sb)[None]
    nb, M, K = A.shape
    _, N, K2 = B.shape
    assert K == K2 and B.shape[0] == nb
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    acc = np.empty((nb, nr, N), dtype=np.int32)
    C = None
    if sa is not None:
        sa = _c(np.asarray(sa, dtype=np.float32), np.float32)
        sb = _c(np.asarray(sb, dtype=np.float32), np.float32)
        C = np.empty((nb, nr, N), dtype=np.float32)
    rc = _load().or_gemm_i8(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), nb, M, N, K, M * K, N * K,
                            _ptr(r), nr, _ptr(acc), _ptr(C))
    if rc < 0:
        raise ValueError("bad arguments")
    if rc == 1:
        raise OverflowError("an exact INT8 accumulator does not fit int32")
    if not batched:
        acc = acc[0]
        C = None if C is None else C[0]
    return acc, C


def gemm_fp8(A8, B8, fmt: int, layout: int, sa: float, sb: float, rows=None, want_bf16=True):
    """FP8 GEMM reference.  Returns (ref float64 [rows, N], bf16 bits or None).

    layout NT: A[M,K], B[N,K]; NN: A[M,K], B[K,N]; TN: A[K,M], B[K,N].
    """
    A8 = _c(A8, np.uint8)
    B8 = _c(B8, np.uint8)
    if layout == NT:
        M, K = A8.shape
        N = B8.shape[0]
        assert B8.shape[1] == K
    elif layout == NN:
        M, K = A8.shape
        N = B8.shape[1]
        assert B8.shape[0] == K
    elif layout == TN:
        K, M = A8.shape
        N = B8.shape[1]
        assert B8.shape[0] == K
    else:
        raise ValueError("layout must be NT, NN or TN")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    ref = np.empty((nr, N), dtype=np.float64)
    bf = np.empty((nr, N), dtype=np.uint16) if want_bf16 else None
    rc = _load().or_gemm_fp8(_ptr(A8), _ptr(B8), int(fmt), int(layout), M, N, K,
                             float(np.float32(sa)), float(np.float32(sb)), _ptr(r), nr,
                             _ptr(ref), _ptr(bf))
    if rc != 0:
        raise ValueError("bad arguments")
    return ref, bf


def gemm_fp8_e4m3(A8, B8, fmt: int, layout: int, sa: float, sb: float, out_scale: float,
                  rows=None):
    """FP8 GEMM with E4M3 output.  Returns (t_ref float64 = ref / out_scale,
    codes uint8 from the oracle's own float32 scaling)."""
    A8 = _c(A8, np.uint8)
    B8 = _c(B8, np.uint8)
    if layout == NT:
        (M, K), N = A8.shape, B8.shape[0]
    elif layout == NN:
        (M, K), N = A8.shape, B8.shape[1]
    elif layout == TN:
        (K, M), N = A8.shape, B8.shape[1]
    else:
        raise ValueError("layout must be NT, NN or TN")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    t = np.empty((nr, N), dtype=np.float64)
    codes = np.empty((nr, N), dtype=np.uint8)
    rc = _load().or_gemm_fp8_e4m3(_ptr(A8), _ptr(B8), int(fmt), int(layout), M, N, K,
                                  float(np.float32(sa)), float(np.float32(sb)),
                                  float(np.float32(out_scale)), _ptr(r), nr, _ptr(t), _ptr(codes))
    if rc != 0:
        raise ValueError("bad arguments")
    return t, codes


def e4m3_acceptable(codes, t_ref, slack):
    """True where the E4M3 code's value lies between the representable values
    bracketing [t_ref - slack, t_ref + slack] (what RNE of any value in that
    interval can give), saturating at +-448."""
    tab = fp8_decode_table(E4M3)
    vals = np.unique(tab[np.isfinite(tab)])
    lo = np.clip(t_ref - slack, -448.0, 448.0)
    hi = np.clip(t_ref + slack, -448.0, 448.0)
    lo_rep = vals[np.clip(np.searchsorted(vals, lo, side="right") - 1, 0, vals.size - 1)]
    hi_rep = vals[np.clip(np.searchsorted(vals, hi, side="left"), 0, vals.size - 1)]
    got = tab[codes]
    return (got >= lo_rep) & (got <= hi_rep)


def gemm_fp8_bias(A8, B8, fmt: int, layout: int, sa: float, sb: float, bias_f32=None, rows=None):
    """FP8 GEMM plus a float32 bias per output column.  Returns (ref, bf16 bits)."""
    A8 = _c(A8, np.uint8)
    B8 = _c(B8, np.uint8)
    if layout == NT:
        (M, K), N = A8.shape, B8.shape[0]
    elif layout == NN:
        (M, K), N = A8.shape, B8.shape[1]
    elif layout == TN:
        (K, M), N = A8.shape, B8.shape[1]
    else:
        raise ValueError("layout must be NT, NN or TN")
    bias = None if bias_f32 is None else _c(np.asarray(bias_f32, dtype=np.float32), np.float32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    ref = np.empty((nr, N), dtype=np.float64)
    bf = np.empty((nr, N), dtype=np.uint16)
    if _load().or_gemm_fp8_bias(_ptr(A8), _ptr(B8), int(fmt), int(layout), M, N, K,
                                float(np.float32(sa)), float(np.float32(sb)), _ptr(bias), _ptr(r),
                                nr, _ptr(ref), _ptr(bf)) != 0:
        raise ValueError("bad arguments")
    return ref, bf


def fp8_bias_to_f32(codes, fmt: int, step: float) -> np.ndarray:
    codes = _c(np.asarray(codes, dtype=np.uint8), np.uint8)
    out = np.empty(codes.shape, dtype=np.float32)
    if _load().or_fp8_bias_to_f32(_ptr(codes), codes.size, int(fmt), float(np.float32(step)),
                                  _ptr(out)) != 0:
        raise ValueError("bad arguments")
    return out


def colsum_bf16(g_bf16: np.ndarray) -> np.ndarray:
    g = _c(g_bf16, np.uint16)
    T, N = g.shape
    out = np.empty(N, dtype=np.float64)
    if _load().or_colsum_bf16(_ptr(g), T, N, _ptr(out)) != 0:
        raise ValueError("bad arguments")
    return out


def fp8_gemm_bound(ref: np.ndarray, K: int, sa: float, sb: float, maxa8: float, maxb8: float):
    """Allowed |err| per element for a bf16 FP8-GEMM output against the fp64 reference:
    1e-2*|ref| + 1e-3*sqrt(K)*sa*sb*max|a8|*max|b8|."""
    return 1e-2 * np.abs(ref) + 1e-3 * np.sqrt(K) * float(sa) * float(sb) * maxa8 * maxb8
