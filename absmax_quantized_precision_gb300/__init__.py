"""absmax-scaled quantization and scaled low-precision GEMM on GB300 (sm_103a).

Thin binding over libsq.so, whose C ABI is declared in include/sq.h.  Every
function here only marshals arguments (torch tensors -> device pointers, the
current CUDA stream) and turns a non-OK status into an exception; all
arithmetic runs in the library's CUDA kernels.  There is no CPU fallback: if
libsq.so has not been built, importing the library raises.

Entry points (names as in the C ABI):
  sq_quantize_rowwise_i8  per-row symmetric INT8 (absmax/127, half-to-even)
  sq_quantize_fp8         per-tensor FP8 E4M3/E5M2 with the amax fused in
  sq_gemm_i8_rowscaled    exact INT8 GEMM, fp32 = acc * sA[i] * sB[j]
  sq_gemm_fp8_scaled      FP8 GEMM, bf16 = acc * sa * sb, layouts NT/NN/TN
  sq_gemm_fp8_scaled_pair two independent FP8 GEMMs in one call (e.g. dX and dW)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsq.so")

SQ_OK, SQ_ERR_INVALID_ARG, SQ_ERR_UNSUPPORTED, SQ_ERR_ALIGNMENT, SQ_ERR_CUDA, \
    SQ_ERR_DEVICE_TIMEOUT = range(6)
SQ_F32, SQ_BF16 = 0, 1
SQ_FMT_E4M3, SQ_FMT_E5M2 = 0, 1
SQ_NT, SQ_NN, SQ_TN = 0, 1, 2
SQ_BIAS_NONE, SQ_BIAS_BF16, SQ_BIAS_FP8 = 0, 1, 2
SQ_GRAD_INPUT, SQ_GRAD_WEIGHT, SQ_GRAD_BIAS = 1, 2, 4

# every symbol include/sq.h declares
EXPORTS = ("sq_status_string", "sq_workspace_bytes", "sq_quantize_rowwise_i8", "sq_quantize_fp8",
           "sq_quantize_fp8_multi", "sq_quantize_rowwise_i8_staged_pair",
           "sq_gemm_i8_workspace_bytes", "sq_gemm_i8_rowscaled", "sq_gemm_fp8_scaled", "sq_gemm_fp8_scaled_pair",
           "sq_get_last_device_error", "sq_gemm_i8_rowscaled_noalloc", "sq_quantize_fp8_ring",
           "sq_gemm_fp8_scaled_e4m3", "sq_quantize_grouped_i8_workspace_bytes",
           "sq_quantize_grouped_i8", "sq_gemm_i8_grouped", "sq_linear_workspace_bytes",
           "sq_linear_forward_fp8", "sq_linear_backward_fp8", "sq_selftest_bounded_wait",
           "sq_gemm_i8_stage", "sq_gemm_i8_rowscaled_staged", "sq_quantize_rowwise_i8_staged",
           "sq_set_clock_probe")

# size of the fixed scratch array behind sq_gemm_i8_rowscaled_noalloc
GEMM_I8_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

_lib = None


class SQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


def load_library():
    """Load libsq.so (raises if it has not been built: no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsq.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.sq_status_string.argtypes = [i32]
    L.sq_status_string.restype = ctypes.c_char_p
    L.sq_workspace_bytes.argtypes = []
    L.sq_workspace_bytes.restype = sz
    L.sq_quantize_rowwise_i8.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp]
    L.sq_quantize_rowwise_i8.restype = i32
    L.sq_quantize_fp8.argtypes = [vp, i64, vp, i32, vp, vp, vp, vp]
    L.sq_quantize_fp8.restype = i32
    L.sq_quantize_fp8_multi.argtypes = [i32, vp, vp, vp, i32, vp, vp, vp, vp]
    L.sq_quantize_fp8_multi.restype = i32
    L.sq_quantize_rowwise_i8_staged_pair.argtypes = [vp, i64, vp, i64, i32, i64, i64, i64, i64, vp, vp,
                                                     vp, vp, vp, sz, vp]
    L.sq_quantize_rowwise_i8_staged_pair.restype = i32
    L.sq_gemm_i8_workspace_bytes.argtypes = [i64, i64, i64, i64]
    L.sq_gemm_i8_workspace_bytes.restype = sz
    L.sq_gemm_i8_rowscaled.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, vp, vp,
                                       vp, sz, vp]
    L.sq_gemm_i8_rowscaled.restype = i32
    L.sq_gemm_fp8_scaled.argtypes = [vp, vp, vp, vp, i32, i32, i64, i64, i64, vp, vp]
    L.sq_gemm_fp8_scaled.restype = i32
    # host arrays of two entries each
    L.sq_gemm_fp8_scaled_pair.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
    L.sq_gemm_fp8_scaled_pair.restype = i32
    L.sq_get_last_device_error.argtypes = [vp]
    L.sq_get_last_device_error.restype = i32
    L.sq_gemm_i8_rowscaled_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                               vp, vp, vp]
    L.sq_gemm_i8_rowscaled_noalloc.restype = i32
    L.sq_quantize_fp8_ring.argtypes = [vp, i64, i32, vp, vp, vp, i64, i64, i32, vp, vp]
    L.sq_quantize_fp8_ring.restype = i32
    L.sq_gemm_fp8_scaled_e4m3.argtypes = [vp, vp, vp, vp, i32, i32, i64, i64, i64, vp, vp, vp]
    L.sq_gemm_fp8_scaled_e4m3.restype = i32
    L.sq_quantize_grouped_i8_workspace_bytes.argtypes = [i64, i64]
    L.sq_quantize_grouped_i8_workspace_bytes.restype = sz
    L.sq_quantize_grouped_i8.argtypes = [vp, i32, i64, i64, i64, i64, vp, vp, vp, sz, vp]
    L.sq_quantize_grouped_i8.restype = i32
    L.sq_gemm_i8_grouped.argtypes = [vp, vp, i64, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
                                     vp, vp, vp, sz, vp]
    L.sq_gemm_i8_grouped.restype = i32
    L.sq_linear_workspace_bytes.argtypes = [i64, i64, i64]
    L.sq_linear_workspace_bytes.restype = sz
    L.sq_linear_forward_fp8.argtypes = [vp, i64, i64, vp, i32, i64, vp, i32, vp, vp, vp, i32,
                                        vp, i64, i64, i32, vp, i64, i64, i32,
                                        vp, vp, vp, vp, vp, vp, sz, vp]
    L.sq_linear_forward_fp8.restype = i32
    L.sq_linear_backward_fp8.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp, vp, i32,
                                         vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.sq_linear_backward_fp8.restype = i32
    L.sq_gemm_i8_stage.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, vp, sz, vp]
    L.sq_gemm_i8_stage.restype = i32
    L.sq_gemm_i8_rowscaled_staged.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, sz, vp]
    L.sq_gemm_i8_rowscaled_staged.restype = i32
    L.sq_quantize_rowwise_i8_staged.argtypes = [vp, i32, i64, i64, i64, vp, vp, i32, i64, i64, i64,
                                                i64, vp, sz, vp]
    L.sq_quantize_rowwise_i8_staged.restype = i32
    L.sq_set_clock_probe.argtypes = [vp, vp, i32]
    L.sq_set_clock_probe.restype = i32
    L.sq_selftest_bounded_wait.argtypes = [ctypes.c_uint64, vp]
    L.sq_selftest_bounded_wait.restype = i32
    _lib = L
    return L


def status_string(status: int) -> str:
    return load_library().sq_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != SQ_OK:
        raise SQError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    """All given tensors on one CUDA device; returns that device.  The library
    works on the current device, so every call runs under this device."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libsq works on CUDA tensors only")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices: {dev} and {t.device}")
    return dev


def _need(t, dtype, numel=None, shape=None, what="tensor"):
    """A caller-passed tensor of the given dtype, contiguous, and of the given
    number of elements or shape: the library reads or writes exactly that many."""
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{what} must hold {numel} elements, got {t.numel()}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _i8_operands(A, B, sA, sB, group_a=1, group_b=1):
    """Shapes of the INT8 GEMM operands, checked against each other and against
    the scale vectors the epilogue reads (batch * ceil(M / group_a) and
    batch * ceil(N / group_b) floats)."""
    if A.dtype != torch.int8 or B.dtype != torch.int8:
        raise TypeError("A and B must be int8 codes")
    if A.dim() not in (2, 3) or B.dim() != A.dim():
        raise ValueError("A and B must both be [rows, K] or both [batch, rows, K]")
    batched = A.dim() == 3
    A3 = A if batched else A.unsqueeze(0)
    B3 = B if batched else B.unsqueeze(0)
    nb, M, K = A3.shape
    if B3.shape[0] != nb or B3.shape[2] != K:
        raise ValueError(f"A {tuple(A.shape)} and B {tuple(B.shape)} do not share batch and K")
    N = B3.shape[1]
    if not (A3.is_contiguous() and B3.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    ga, gb = max(1, min(int(group_a), M)), max(1, min(int(group_b), N))
    _need(sA, torch.float32, numel=nb * ((M + ga - 1) // ga), what="sA")
    _need(sB, torch.float32, numel=nb * ((N + gb - 1) // gb), what="sB")
    return A3, B3, nb, M, N, K, batched


def _i8_outputs(C, acc_out, want_c, shape, dev):
    if C is not None:
        _need(C, torch.float32, shape=shape, what="C")
    elif want_c:
        C = torch.empty(shape, dtype=torch.float32, device=dev)
    if acc_out is True:
        acc_out = torch.empty(shape, dtype=torch.int32, device=dev)
    elif acc_out is False:
        acc_out = None
    elif acc_out is not None:
        _need(acc_out, torch.int32, shape=shape, what="acc_out")
    if C is None and acc_out is None:
        raise ValueError("ask for C, acc_out or both")
    return C, acc_out


def _fp8_shape(A, B, layout):
    if A.dtype != torch.uint8 or B.dtype != torch.uint8:
        raise TypeError("A and B must be FP8 codes (uint8)")
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    if layout == SQ_NT:
        (M, K), (N, K2) = A.shape, B.shape
    elif layout == SQ_NN:
        (M, K), (K2, N) = A.shape, B.shape
    elif layout == SQ_TN:
        (K, M), (K2, N) = A.shape, B.shape
    else:
        raise ValueError("layout must be SQ_NT, SQ_NN or SQ_TN")
    if K2 != K:
        raise ValueError(f"A {tuple(A.shape)} and B {tuple(B.shape)} do not share K in this layout")
    return M, N, K


# ---------------------------------------------------------------- workspaces
def workspace_bytes() -> int:
    return int(load_library().sq_workspace_bytes())


def new_workspace(device=None) -> torch.Tensor:
    """A zeroed workspace for sq_quantize_fp8 (allocate once per stream)."""
    return torch.zeros(workspace_bytes(), dtype=torch.uint8, device=device or "cuda")


def gemm_i8_workspace_bytes(batch: int, M: int, N: int, K: int) -> int:
    return int(load_library().sq_gemm_i8_workspace_bytes(batch, M, N, K))


# ---------------------------------------------------------------- entry points
def sq_quantize_rowwise_i8(x: torch.Tensor, q: torch.Tensor = None, scales: torch.Tensor = None,
                           stream=None):
    """Per-row INT8 of x (float32 or bfloat16, last dim = row, rows may be
    strided).  Returns (q int8 packed, scales float32 of shape x.shape[:-1])."""
    dev = _need_cuda(x, q, scales)
    if x.dtype == torch.float32:
        dt = SQ_F32
    elif x.dtype == torch.bfloat16:
        dt = SQ_BF16
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    cols = x.shape[-1]
    x2 = x.reshape(-1, cols) if x.dim() != 2 else x
    if x2.numel() and x2.stride(-1) != 1:
        raise ValueError("rows of x must be contiguous")
    rows = x2.shape[0]
    ld = x2.stride(0) if rows > 1 else cols
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    _need(q, torch.int8, numel=rows * cols, what="q")
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(scales, torch.float32, numel=rows, what="scales")
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_rowwise_i8(_ptr(x2), dt, rows, cols, ld, _ptr(q),
                                                     _ptr(scales), _stream(stream)),
               "sq_quantize_rowwise_i8")
    return q, scales


def sq_quantize_fp8(x: torch.Tensor, scale: torch.Tensor, fmt: int, workspace: torch.Tensor,
                    x8: torch.Tensor = None, amax: torch.Tensor = None, stream=None):
    """Per-tensor FP8 of bf16 x with the step `scale` (1-element float32 on the
    device) divided out.  Returns (x8 uint8 codes, amax 1-element float32)."""
    dev = _need_cuda(x, scale, workspace, x8, amax)
    _need(x, torch.bfloat16, what="x")
    _need(scale, torch.float32, numel=1, what="scale")
    if workspace.numel() * workspace.element_size() < workspace_bytes():
        raise ValueError("workspace is smaller than sq_workspace_bytes()")
    if x8 is None:
        x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _need(x8, torch.uint8, numel=x.numel(), what="x8")
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _need(amax, torch.float32, numel=1, what="amax")
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_fp8(_ptr(x), x.numel(), _ptr(scale), int(fmt), _ptr(x8),
                                              _ptr(amax), _ptr(workspace), _stream(stream)),
               "sq_quantize_fp8")
    return x8, amax


def sq_quantize_fp8_multi(xs, scales, fmt: int, workspace: torch.Tensor, x8s=None, amaxs=None,
                          stream=None):
    """sq_quantize_fp8 on 1-4 bf16 tensors in one launch, each with its own
    step (1-element float32) and amax.  Returns (list of x8, list of amax)."""
    xs, scales = list(xs), list(scales)
    if not 1 <= len(xs) <= 4 or len(scales) != len(xs):
        raise ValueError("1 to 4 tensors, one step each")
    x8s = [None] * len(xs) if x8s is None else list(x8s)
    amaxs = [None] * len(xs) if amaxs is None else list(amaxs)
    if len(x8s) != len(xs) or len(amaxs) != len(xs):
        raise ValueError("one output and one amax per tensor")
    dev = _need_cuda(workspace, *xs, *scales, *[t for t in x8s + amaxs if t is not None])
    if workspace.numel() * workspace.element_size() < workspace_bytes():
        raise ValueError("workspace is smaller than sq_workspace_bytes()")
    for t, (x, sc) in enumerate(zip(xs, scales)):
        _need(x, torch.bfloat16, what=f"xs[{t}]")
        _need(sc, torch.float32, numel=1, what=f"scales[{t}]")
        if x8s[t] is None:
            x8s[t] = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        _need(x8s[t], torch.uint8, numel=x.numel(), what=f"x8s[{t}]")
        if amaxs[t] is None:
            amaxs[t] = torch.empty(1, dtype=torch.float32, device=x.device)
        _need(amaxs[t], torch.float32, numel=1, what=f"amaxs[{t}]")
    n = len(xs)
    P = ctypes.c_void_p * n
    ptrs = lambda ts: P(*[_ptr(t) for t in ts])
    numel = (ctypes.c_int64 * n)(*[x.numel() for x in xs])
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_fp8_multi(n, ptrs(xs), numel, ptrs(scales), int(fmt),
                                                    ptrs(x8s), ptrs(amaxs), _ptr(workspace),
                                                    _stream(stream)),
               "sq_quantize_fp8_multi")
    return x8s, amaxs


def new_ring(hist_len: int, scale: float, device=None) -> torch.Tensor:
    """A delayed-scaling ring float32[hist_len + 2] = [hist | scale | counter]
    with an empty history, the given step, and a zero counter."""
    r = torch.zeros(hist_len + 2, dtype=torch.float32, device=device or "cuda")
    r[hist_len] = scale
    return r


def sq_quantize_fp8_ring(x: torch.Tensor, fmt: int, ring: torch.Tensor, idx: int, margin: int,
                         workspace: torch.Tensor, x8: torch.Tensor = None,
                         amax: torch.Tensor = None, stream=None):
    """Per-tensor FP8 of bf16 x with the step ring[H]; records the amax in
    ring[idx] and publishes the next step in ring[H] on the device."""
    dev = _need_cuda(x, ring, workspace, x8, amax)
    _need(x, torch.bfloat16, what="x")
    if ring.dtype != torch.float32 or not ring.is_contiguous() or ring.numel() < 3:
        raise TypeError("ring must be a contiguous float32 tensor of hist_len + 2 entries")
    if workspace.numel() * workspace.element_size() < workspace_bytes():
        raise ValueError("workspace is smaller than sq_workspace_bytes()")
    if x8 is None:
        x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _need(x8, torch.uint8, numel=x.numel(), what="x8")
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _need(amax, torch.float32, numel=1, what="amax")
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_fp8_ring(_ptr(x), x.numel(), int(fmt), _ptr(x8),
                                                   _ptr(amax), _ptr(ring), ring.numel() - 2,
                                                   int(idx), int(margin), _ptr(workspace),
                                                   _stream(stream)),
               "sq_quantize_fp8_ring")
    return x8, amax


def sq_quantize_grouped_i8(x: torch.Tensor, group_rows: int, q: torch.Tensor = None,
                           scales: torch.Tensor = None, workspace: torch.Tensor = None,
                           stream=None):
    """Row-group INT8 of a 2-D float32/bfloat16 x: groups of group_rows rows
    share a scale (group_rows >= rows: per tensor).  Returns (q, scales)."""
    dev = _need_cuda(x, q, scales, workspace)
    dt = {torch.float32: SQ_F32, torch.bfloat16: SQ_BF16}.get(x.dtype)
    if dt is None or x.dim() != 2 or (x.numel() and x.stride(1) != 1):
        raise TypeError("x must be 2-D float32 or bfloat16 with contiguous rows")
    rows, cols = x.shape
    g = max(1, min(int(group_rows), rows)) if rows else 1
    ng = (rows + g - 1) // g
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    _need(q, torch.int8, numel=rows * cols, what="q")
    if scales is None:
        scales = torch.empty(ng, dtype=torch.float32, device=x.device)
    _need(scales, torch.float32, numel=ng, what="scales")
    if workspace is None and g > 1:
        workspace = torch.empty(int(load_library().sq_quantize_grouped_i8_workspace_bytes(rows, g)),
                                dtype=torch.uint8, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ld = x.stride(0) if rows > 1 else cols
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_grouped_i8(_ptr(x), dt, rows, cols, ld, g, _ptr(q),
                                                     _ptr(scales), _ptr(workspace), nbytes,
                                                     _stream(stream)),
               "sq_quantize_grouped_i8")
    return q, scales


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size()


def sq_gemm_i8_grouped(A: torch.Tensor, sA: torch.Tensor, group_a: int, B: torch.Tensor,
                       sB: torch.Tensor, group_b: int, workspace: torch.Tensor,
                       C: torch.Tensor = None, acc_out=None, want_c: bool = True, stream=None):
    """INT8 GEMM with row-group scales sA[b][i // group_a], sB[b][j // group_b]."""
    dev = _need_cuda(A, B, sA, sB, workspace, C,
                     acc_out if isinstance(acc_out, torch.Tensor) else None)
    A3, B3, nb, M, N, K, batched = _i8_operands(A, B, sA, sB, group_a, group_b)
    shape = (nb, M, N) if batched else (M, N)
    C, acc_out = _i8_outputs(C, acc_out, want_c, shape, A.device)
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_i8_grouped(
            _ptr(A3), _ptr(sA), int(group_a), _ptr(B3), _ptr(sB), int(group_b), nb, M, N, K,
            M * K, N * K, M * N, _ptr(C), _ptr(acc_out), _ptr(workspace), _ws_bytes(workspace),
            _stream(stream)), "sq_gemm_i8_grouped")
    return C, acc_out


def sq_gemm_i8_rowscaled(A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor, sB: torch.Tensor,
                         workspace: torch.Tensor, C: torch.Tensor = None, acc_out=None,
                         want_c: bool = True, stream=None):
    """C[b] = A[b] B[b]^T on int8 codes with fp32 (acc * sA[i]) * sB[j].

    A: [M,K] or [batch,M,K] int8, B: [N,K] or [batch,N,K].  Returns (C, acc_out);
    pass acc_out=True to get the exact int32 accumulators too."""
    dev = _need_cuda(A, B, sA, sB, workspace, C,
                     acc_out if isinstance(acc_out, torch.Tensor) else None)
    A3, B3, nb, M, N, K, batched = _i8_operands(A, B, sA, sB)
    shape = (nb, M, N) if batched else (M, N)
    C, acc_out = _i8_outputs(C, acc_out, want_c, shape, A.device)
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_i8_rowscaled(
            _ptr(A3), _ptr(sA), _ptr(B3), _ptr(sB), nb, M, N, K, M * K, N * K, M * N,
            _ptr(C), _ptr(acc_out), _ptr(workspace), _ws_bytes(workspace),
            _stream(stream)), "sq_gemm_i8_rowscaled")
    return C, acc_out


def sq_gemm_i8_stage(A: torch.Tensor, B: torch.Tensor, workspace: torch.Tensor, stream=None):
    """First phase of sq_gemm_i8_rowscaled: stage the int8 codes of A and B
    (shapes as there) in `workspace` for sq_gemm_i8_rowscaled_staged."""
    dev = _need_cuda(A, B, workspace)
    if A.dtype != torch.int8 or B.dtype != torch.int8:
        raise TypeError("A and B must be int8 codes")
    if A.dim() not in (2, 3) or B.dim() != A.dim():
        raise ValueError("A and B must both be [rows, K] or both [batch, rows, K]")
    A3 = A if A.dim() == 3 else A.unsqueeze(0)
    B3 = B if B.dim() == 3 else B.unsqueeze(0)
    nb, M, K = A3.shape
    if B3.shape[0] != nb or B3.shape[2] != K or not (A3.is_contiguous() and B3.is_contiguous()):
        raise ValueError("A and B must be contiguous and share batch and K")
    N = B3.shape[1]
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_i8_stage(_ptr(A3), _ptr(B3), nb, M, N, K, M * K, N * K,
                                               _ptr(workspace), _ws_bytes(workspace),
                                               _stream(stream)), "sq_gemm_i8_stage")


def sq_gemm_i8_rowscaled_staged(sA: torch.Tensor, sB: torch.Tensor, shape, workspace: torch.Tensor,
                                C: torch.Tensor = None, acc_out=None, want_c: bool = True,
                                stream=None):
    """Second phase of sq_gemm_i8_rowscaled on a workspace staged by
    sq_gemm_i8_stage for operands of shape = (batch, M, N, K) (batch 0: the
    2-D form).  Returns (C, acc_out)."""
    dev = _need_cuda(sA, sB, workspace, C, acc_out if isinstance(acc_out, torch.Tensor) else None)
    nb, M, N, K = (int(v) for v in shape)
    batched = nb > 0
    nb = max(nb, 1)
    _need(sA, torch.float32, numel=nb * M, what="sA")
    _need(sB, torch.float32, numel=nb * N, what="sB")
    oshape = (nb, M, N) if batched else (M, N)
    C, acc_out = _i8_outputs(C, acc_out, want_c, oshape, sA.device)
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_i8_rowscaled_staged(
            _ptr(sA), _ptr(sB), nb, M, N, K, M * N, _ptr(C), _ptr(acc_out),
            _ptr(workspace), _ws_bytes(workspace), _stream(stream)), "sq_gemm_i8_rowscaled_staged")
    return C, acc_out


def sq_quantize_rowwise_i8_staged(x: torch.Tensor, operand: int, shape, workspace: torch.Tensor,
                                  q: torch.Tensor = None, scales: torch.Tensor = None,
                                  stream=None):
    """sq_quantize_rowwise_i8 of x that also stages its codes in an INT8 GEMM
    workspace for operands of shape = (batch, M, N, K) (batch 0: the 2-D
    form); operand 0 is A, 1 is B.  Returns (q, scales)."""
    dev = _need_cuda(x, q, scales, workspace)
    if x.dtype == torch.float32:
        dt = SQ_F32
    elif x.dtype == torch.bfloat16:
        dt = SQ_BF16
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    nb, M, N, K = (int(v) for v in shape)
    nb = max(nb, 1)
    cols = x.shape[-1]
    x2 = x.reshape(-1, cols) if x.dim() != 2 else x
    if x2.numel() and x2.stride(-1) != 1:
        raise ValueError("rows of x must be contiguous")
    rows = x2.shape[0]
    if rows != nb * (N if operand else M) or cols != K:
        raise ValueError(f"x {tuple(x.shape)} is not operand {'B' if operand else 'A'} of {shape}")
    ld = x2.stride(0) if rows > 1 else cols
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    _need(q, torch.int8, numel=rows * cols, what="q")
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(scales, torch.float32, numel=rows, what="scales")
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_rowwise_i8_staged(
            _ptr(x2), dt, rows, cols, ld, _ptr(q), _ptr(scales), int(operand), nb, M, N, K,
            _ptr(workspace), _ws_bytes(workspace), _stream(stream)), "sq_quantize_rowwise_i8_staged")
    return q, scales


def sq_quantize_rowwise_i8_staged_pair(xa: torch.Tensor, xb: torch.Tensor, shape,
                                       workspace: torch.Tensor, qa: torch.Tensor = None,
                                       sa: torch.Tensor = None, qb: torch.Tensor = None,
                                       sb: torch.Tensor = None, stream=None):
    """sq_quantize_rowwise_i8_staged of A (xa) and B (xb) in one call (one
    launch when both fit the register-resident kernel).  Returns
    (qa, sa, qb, sb)."""
    dev = _need_cuda(xa, xb, qa, sa, qb, sb, workspace)
    if xa.dtype != xb.dtype:
        raise TypeError("xa and xb must have the same dtype")
    if xa.dtype == torch.float32:
        dt = SQ_F32
    elif xa.dtype == torch.bfloat16:
        dt = SQ_BF16
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {xa.dtype}")
    nb, M, N, K = (int(v) for v in shape)
    nb = max(nb, 1)
    views = []
    for x, rows, name in ((xa, nb * M, "A"), (xb, nb * N, "B")):
        cols = x.shape[-1]
        x2 = x.reshape(-1, cols) if x.dim() != 2 else x
        if x2.numel() and x2.stride(-1) != 1:
            raise ValueError("rows of x must be contiguous")
        if x2.shape[0] != rows or cols != K:
            raise ValueError(f"x {tuple(x.shape)} is not operand {name} of {shape}")
        views.append((x2, x2.stride(0) if rows > 1 else cols))
    if qa is None:
        qa = torch.empty(xa.shape, dtype=torch.int8, device=xa.device)
    if qb is None:
        qb = torch.empty(xb.shape, dtype=torch.int8, device=xb.device)
    if sa is None:
        sa = torch.empty(xa.shape[:-1], dtype=torch.float32, device=xa.device)
    if sb is None:
        sb = torch.empty(xb.shape[:-1], dtype=torch.float32, device=xb.device)
    _need(qa, torch.int8, numel=nb * M * K, what="qa")
    _need(qb, torch.int8, numel=nb * N * K, what="qb")
    _need(sa, torch.float32, numel=nb * M, what="sa")
    _need(sb, torch.float32, numel=nb * N, what="sb")
    (xa2, lda), (xb2, ldb) = views
    with torch.cuda.device(dev):
        _check(load_library().sq_quantize_rowwise_i8_staged_pair(
            _ptr(xa2), lda, _ptr(xb2), ldb, dt, nb, M, N, K, _ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb),
            _ptr(workspace), _ws_bytes(workspace), _stream(stream)), "sq_quantize_rowwise_i8_staged_pair")
    return qa, sa, qb, sb


def sq_gemm_i8_rowscaled_noalloc(A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor,
                                 sB: torch.Tensor, C: torch.Tensor = None, acc_out=None,
                                 want_c: bool = True, stream=None):
    """sq_gemm_i8_rowscaled without a workspace argument: the library stages the
    operands in its own fixed 16 MiB device array, so this call allocates
    nothing (the output tensors are created here only when not passed in).
    Problems whose staged operands exceed the array raise SQError
    (SQ_ERR_UNSUPPORTED).  Calls that overlap on the GPU race on the array."""
    dev = _need_cuda(A, B, sA, sB, C, acc_out if isinstance(acc_out, torch.Tensor) else None)
    A3, B3, nb, M, N, K, batched = _i8_operands(A, B, sA, sB)
    shape = (nb, M, N) if batched else (M, N)
    C, acc_out = _i8_outputs(C, acc_out, want_c, shape, A.device)
    with torch.cuda.device(dev):
        st = load_library().sq_gemm_i8_rowscaled_noalloc(
            _ptr(A3), _ptr(sA), _ptr(B3), _ptr(sB), nb, M, N, K, M * K, N * K, M * N, _ptr(C),
            _ptr(acc_out), _stream(stream))
    if st == SQ_ERR_UNSUPPORTED:
        raise SQError(st, "sq_gemm_i8_rowscaled_noalloc: staged operands "
                          f"({gemm_i8_workspace_bytes(nb, M, N, K)} bytes) exceed the "
                          f"{GEMM_I8_NOALLOC_SCRATCH_BYTES}-byte scratch array, or K > 2^17")
    _check(st, "sq_gemm_i8_rowscaled_noalloc")
    return C, acc_out


def sq_gemm_fp8_scaled(A: torch.Tensor, B: torch.Tensor, sa: torch.Tensor, sb: torch.Tensor,
                       fmt: int, layout: int, C: torch.Tensor = None, stream=None):
    """bf16 C = (acc * sa) * sb for FP8 codes A, B (uint8) in layout NT/NN/TN."""
    dev = _need_cuda(A, B, sa, sb, C)
    M, N, K = _fp8_shape(A, B, layout)
    _need(sa, torch.float32, numel=1, what="sa")
    _need(sb, torch.float32, numel=1, what="sb")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, torch.bfloat16, shape=(M, N), what="C")
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_fp8_scaled(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb), int(fmt),
                                                 int(layout), M, N, K, _ptr(C), _stream(stream)),
               "sq_gemm_fp8_scaled")
    return C


def sq_gemm_fp8_scaled_pair(As, Bs, sas, sbs, fmt: int, layouts, Cs=None, stream=None):
    """Two independent FP8 GEMMs in one call: problem i is
    sq_gemm_fp8_scaled(As[i], Bs[i], sas[i], sbs[i], fmt, layouts[i], Cs[i])."""
    if len(As) != 2 or len(Bs) != 2 or len(sas) != 2 or len(sbs) != 2 or len(layouts) != 2:
        raise ValueError("two problems expected")
    Cs = list(Cs) if Cs is not None else [None, None]
    if len(Cs) != 2:
        raise ValueError("two outputs expected")
    dev = _need_cuda(*As, *Bs, *sas, *sbs, *[c for c in Cs if c is not None])
    dims = []
    for i in range(2):
        M, N, K = _fp8_shape(As[i], Bs[i], layouts[i])
        _need(sas[i], torch.float32, numel=1, what="sa")
        _need(sbs[i], torch.float32, numel=1, what="sb")
        if Cs[i] is None:
            Cs[i] = torch.empty((M, N), dtype=torch.bfloat16, device=As[i].device)
        _need(Cs[i], torch.bfloat16, shape=(M, N), what="C")
        dims.append((M, N, K))
    arr = ctypes.c_void_p * 2
    i64x2 = ctypes.c_int64 * 2
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_fp8_scaled_pair(
            arr(*[_ptr(t) for t in As]), arr(*[_ptr(t) for t in Bs]),
            arr(*[_ptr(t) for t in sas]), arr(*[_ptr(t) for t in sbs]), int(fmt),
            (ctypes.c_int * 2)(*[int(x) for x in layouts]), i64x2(*[d[0] for d in dims]),
            i64x2(*[d[1] for d in dims]), i64x2(*[d[2] for d in dims]),
            arr(*[_ptr(t) for t in Cs]), _stream(stream)), "sq_gemm_fp8_scaled_pair")
    return Cs


def sq_gemm_fp8_scaled_e4m3(A: torch.Tensor, B: torch.Tensor, sa: torch.Tensor, sb: torch.Tensor,
                            fmt: int, layout: int, out_scale: torch.Tensor, C: torch.Tensor = None,
                            stream=None):
    """E4M3 codes C = e4m3((acc * sa) * sb / out_scale) for FP8 codes A, B."""
    dev = _need_cuda(A, B, sa, sb, out_scale, C)
    M, N, K = _fp8_shape(A, B, layout)
    for t, n in ((sa, "sa"), (sb, "sb"), (out_scale, "out_scale")):
        _need(t, torch.float32, numel=1, what=n)
    if C is None:
        C = torch.empty((M, N), dtype=torch.uint8, device=A.device)
    _need(C, torch.uint8, shape=(M, N), what="C")
    with torch.cuda.device(dev):
        _check(load_library().sq_gemm_fp8_scaled_e4m3(_ptr(A), _ptr(B), _ptr(sa), _ptr(sb),
                                                      int(fmt), int(layout), M, N, K,
                                                      _ptr(out_scale), _ptr(C), _stream(stream)),
               "sq_gemm_fp8_scaled_e4m3")
    return C


def linear_workspace(T: int, N: int, K: int, device=None) -> torch.Tensor:
    """A zeroed workspace for the fused linear forward / backward."""
    n = int(load_library().sq_linear_workspace_bytes(T, N, K))
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ring_args(ring, idx, margin):
    if ring is None:
        return None, 0, 0, 0
    if ring.dtype != torch.float32 or not ring.is_contiguous() or ring.numel() < 3:
        raise TypeError("a ring is a contiguous float32 tensor of hist_len + 2 entries")
    return ring, ring.numel() - 2, int(idx), int(margin)


def sq_linear_forward_fp8(x: torch.Tensor, w: torch.Tensor, bias, sx, sw, fmt: int,
                          workspace: torch.Tensor, bias_scale=None, w_prequantized: bool = False,
                          x_ring=None, x_ring_idx: int = 0, x_ring_margin: int = 0,
                          w_ring=None, w_ring_idx: int = 0, w_ring_margin: int = 0, stream=None):
    """Fused FP8 linear forward.  x bf16 [M, K]; w bf16 [N, K] (or FP8 codes
    uint8 when w_prequantized); bias None, bf16 [N], or FP8 codes uint8 [N]
    (with bias_scale).  Returns (out bf16 [M, N], x8, w8, amax_x, amax_w)."""
    dev = _need_cuda(x, w, workspace, bias, sx, sw, bias_scale, x_ring, w_ring)
    _need(x, torch.bfloat16, what="x")
    if x.dim() != 2 or w.dim() != 2:
        raise ValueError("x and w must be 2-D")
    M, K = x.shape
    N = w.shape[0]
    _need(w, torch.uint8 if w_prequantized else torch.bfloat16, shape=(N, K), what="w")
    if bias is not None:
        _need(bias, bias.dtype, numel=N, what="bias")
    for t, n in ((sx, "sx"), (sw, "sw"), (bias_scale, "bias_scale")):
        if t is not None:
            _need(t, torch.float32, numel=1, what=n)
    if bias is None:
        bkind = SQ_BIAS_NONE
    elif bias.dtype == torch.bfloat16:
        bkind = SQ_BIAS_BF16
    elif bias.dtype == torch.uint8:
        bkind = SQ_BIAS_FP8
    else:
        raise TypeError("bias must be bf16, FP8 codes (uint8) or None")
    dev = x.device
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    x8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    w8 = None if w_prequantized else torch.empty((N, K), dtype=torch.uint8, device=dev)
    amax_x = torch.empty(1, dtype=torch.float32, device=dev)
    amax_w = torch.empty(1, dtype=torch.float32, device=dev)
    xr, xh, xi, xm = _ring_args(x_ring, x_ring_idx, x_ring_margin)
    wr, wh, wi, wm = _ring_args(w_ring, w_ring_idx, w_ring_margin)
    with torch.cuda.device(dev):
        _check(load_library().sq_linear_forward_fp8(
            _ptr(x), M, K, _ptr(w), int(bool(w_prequantized)), N, _ptr(bias), bkind,
            _ptr(bias_scale), _ptr(sx), _ptr(sw), int(fmt), _ptr(xr), xh, xi, xm, _ptr(wr), wh, wi,
            wm, _ptr(out), _ptr(x8), _ptr(w8), _ptr(amax_x), _ptr(amax_w), _ptr(workspace),
            _ws_bytes(workspace), _stream(stream)), "sq_linear_forward_fp8")
    return out, x8, (w if w_prequantized else w8), amax_x, amax_w


def sq_linear_backward_fp8(g: torch.Tensor, x: torch.Tensor, w: torch.Tensor, masks, sg, sw, sx,
                           fmt: int, workspace: torch.Tensor, g_ring=None, g_ring_idx: int = 0,
                           g_ring_margin: int = 0, stream=None):
    """Fused FP8 linear backward for out = x w^T.  g bf16 [T, N], x bf16 [T, K],
    w bf16 [N, K]; masks = (grad_input, grad_weight, grad_bias) booleans.
    Returns (gx [T, K] or None, gw [N, K] or None, gb [N] or None, amax_g)."""
    dev = _need_cuda(g, x, w, workspace, sg, sw, sx, g_ring)
    if g.dim() != 2 or x.dim() != 2 or w.dim() != 2:
        raise ValueError("g, x and w must be 2-D")
    T, N = g.shape
    K = x.shape[1]
    _need(g, torch.bfloat16, what="g")
    _need(x, torch.bfloat16, shape=(T, K), what="x")
    _need(w, torch.bfloat16, shape=(N, K), what="w")
    for t, n in ((sg, "sg"), (sw, "sw"), (sx, "sx")):
        if t is not None:
            _need(t, torch.float32, numel=1, what=n)
    m = (SQ_GRAD_INPUT if masks[0] else 0) | (SQ_GRAD_WEIGHT if masks[1] else 0) | \
        (SQ_GRAD_BIAS if masks[2] else 0)
    dev = g.device
    gx = torch.empty((T, K), dtype=torch.bfloat16, device=dev) if masks[0] else None
    gw = torch.empty((N, K), dtype=torch.bfloat16, device=dev) if masks[1] else None
    gb = torch.empty(N, dtype=torch.bfloat16, device=dev) if masks[2] else None
    amax_g = torch.empty(1, dtype=torch.float32, device=dev)
    g8 = torch.empty((T, N), dtype=torch.uint8, device=dev)
    w8 = torch.empty((N, K), dtype=torch.uint8, device=dev) if masks[0] else None
    x8 = torch.empty((T, K), dtype=torch.uint8, device=dev) if masks[1] else None
    gr, gh, gi, gm = _ring_args(g_ring, g_ring_idx, g_ring_margin)
    with torch.cuda.device(dev):
        _check(load_library().sq_linear_backward_fp8(
            _ptr(g), _ptr(x), _ptr(w), T, N, K, m, _ptr(sg), _ptr(sw), _ptr(sx), int(fmt),
            _ptr(gr), gh, gi, gm, _ptr(gx), _ptr(gw), _ptr(gb), _ptr(amax_g), _ptr(g8), _ptr(w8),
            _ptr(x8), _ptr(workspace), _ws_bytes(workspace), _stream(stream)),
            "sq_linear_backward_fp8")
    return gx, gw, gb, amax_g


def sq_set_clock_probe(fp8_records: torch.Tensor = None, i8_records: torch.Tensor = None):
    """Diagnostics: let the GEMM launches record their CTAs' SM cycles and
    nanoseconds (int64 tensors of 4 * max_ctas words on the current device);
    no arguments stop the records."""
    dev = _need_cuda(fp8_records, i8_records)
    caps = [t.numel() // 4 for t in (fp8_records, i8_records) if t is not None]
    for t in (fp8_records, i8_records):
        if t is not None:
            _need(t, torch.int64, what="records")
    with torch.cuda.device(dev or torch.cuda.current_device()):
        _check(load_library().sq_set_clock_probe(_ptr(fp8_records), _ptr(i8_records),
                                                 min(caps) if caps else 0), "sq_set_clock_probe")


def clock_probe_mhz(records: torch.Tensor) -> dict:
    """Median, minimum and maximum mean SM clock (MHz) over the CTAs that
    wrote records (zero rows are unused slots), their median cycle count, and
    the launch's span from the first CTA's start to the last one's end."""
    r = records.view(-1, 4).cpu()
    r = r[r[:, 3] > r[:, 2]]
    if r.numel() == 0:
        return {}
    cyc = (r[:, 1] - r[:, 0]).double()
    mhz = cyc / (r[:, 3] - r[:, 2]).double() * 1e3
    return {"median": float(mhz.median()), "min": float(mhz.min()), "max": float(mhz.max()),
            "ctas": int(r.shape[0]), "cycles_median": float(cyc.median()),
            "span_ns": int(r[:, 3].max() - r[:, 2].min())}


def sq_selftest_bounded_wait(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test kernel (see include/sq.h)."""
    _check(load_library().sq_selftest_bounded_wait(int(limit_ns), _stream(stream)),
           "sq_selftest_bounded_wait")


def sq_get_last_device_error(stream=None) -> int:
    return int(load_library().sq_get_last_device_error(_stream(stream)))
