"""The INT8 GEMM entry point that allocates nothing.

sq_gemm_i8_rowscaled_noalloc is for callers that cannot allocate device
memory where they run the GEMM (code inside a host engine or framework that
owns the whole device memory pool and only hands over the tensors to work
on, or callers holding device pointers but no allocator).  It stages its
operands in a fixed 16 MiB array inside libsq.  These tests call it through
the C ABI and compare it with sq_gemm_i8_rowscaled (which takes a caller
workspace): INT8 results are exact, so the two must agree bit for bit, on
two calls in a row of different sizes that share the one array.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__
import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, guard_intact, guarded, to_dev

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def noalloc_via_cabi(qa, sa, qb, sb):
    """Direct C-ABI call; returns (C, acc) as numpy."""
    lib = sq.load_library()
    batched = qa.dim() == 3
    nb, M, K = qa.shape if batched else (1, *qa.shape)
    N = qb.shape[-2]
    shape = (nb, M, N) if batched else (M, N)
    C = torch.empty(shape, dtype=torch.float32, device=DEV)
    acc = torch.empty(shape, dtype=torch.int32, device=DEV)
    st = lib.sq_gemm_i8_rowscaled_noalloc(
        _p(qa), _p(sa), _p(qb), _p(sb), nb, M, N, K, M * K, N * K, M * N, _p(C), _p(acc),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == sq.SQ_OK, sq.status_string(st)
    return C.cpu().numpy(), acc.cpu().numpy()


def with_workspace(qa, sa, qb, sb):
    batched = qa.dim() == 3
    nb, M, K = qa.shape if batched else (1, *qa.shape)
    N = qb.shape[-2]
    ws = torch.empty(sq.gemm_i8_workspace_bytes(nb, M, N, K), dtype=torch.uint8, device=DEV)
    C, acc = sq.sq_gemm_i8_rowscaled(qa, sa, qb, sb, ws, acc_out=True)
    return C.cpu().numpy(), acc.cpu().numpy()


def quantized(seed, a_shape, b_shape):
    a = to_dev(synth.normal(seed, a_shape))
    b = to_dev(synth.normal(seed + 1, b_shape))
    qa, sa = sq.sq_quantize_rowwise_i8(a)
    qb, sb = sq.sq_quantize_rowwise_i8(b)
    return qa, sa.reshape(-1).contiguous(), qb, sb.reshape(-1).contiguous()


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    # call 1: A 128x1024, B 512x1024 (per row); call 2: 16 heads of 196x64
    first = quantized(701, (128, 1024), (512, 1024))
    second = quantized(703, (16, 196, 64), (16, 196, 64))
    c1, a1 = noalloc_via_cabi(*first)
    c2, a2 = noalloc_via_cabi(*second)
    w1, wa1 = with_workspace(*first)
    w2, wa2 = with_workspace(*second)
    assert np.array_equal(a1, wa1) and np.array_equal(c1, w1)
    assert np.array_equal(a2, wa2) and np.array_equal(c2, w2)
    # and both agree with the oracle
    qa, sa, qb, sb = (t.cpu().numpy() for t in second)
    oacc, oC = oracle.gemm_i8(qa, qb, sa.reshape(16, 196), sb.reshape(16, 196))
    assert np.array_equal(a2, oacc) and np.array_equal(c2, oC)
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    torch.cuda.set_device(DEV)
    M = N = 4096
    K = 2048           # staged operands: (4096 + 4096) * 2048 * 2 B = 32 MiB > 16 MiB
    assert sq.gemm_i8_workspace_bytes(1, M, N, K) > sq.GEMM_I8_NOALLOC_SCRATCH_BYTES
    qa = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    qb = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    s = torch.ones(M, device=DEV)
    C, cbuf, n = guarded((M, N), torch.float32, 9.0)
    lib = sq.load_library()
    st = lib.sq_gemm_i8_rowscaled_noalloc(_p(qa), _p(s), _p(qb), _p(s), 1, M, N, K, M * K, N * K,
                                          M * N, _p(C), None, None)
    assert st == sq.SQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool(torch.all(C == 9.0).item()) and guard_intact(cbuf, n, 9.0)
    with pytest.raises(sq.SQError, match="scratch array"):
        sq.sq_gemm_i8_rowscaled_noalloc(qa, s, qb, s)
