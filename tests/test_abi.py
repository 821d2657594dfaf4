"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/sq.h declares, and rejects bad arguments before touching a
device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import absmax_quantized_precision_gb300 as sq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return sq.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(sq.EXPORTS)


def test_exported_symbols_are_c_linkage():
    out = os.popen(f"nm -D --defined-only {sq.LIB_PATH}").read()
    for n in declared_functions():
        assert re.search(rf"\sT\s{n}$", out, flags=re.M), n


def test_status_strings_and_sizes(lib):
    for s in range(6):
        assert sq.status_string(s).startswith("SQ_")
    assert sq.workspace_bytes() >= 8
    # fp16 copies of A and B, then two bound regions of 1024 words
    assert sq.gemm_i8_workspace_bytes(1, 128, 512, 1024) == 128 * 1024 * 2 + 512 * 1024 * 2 + 8192
    assert sq.gemm_i8_workspace_bytes(0, 1, 1, 1) == 0


def test_invalid_arguments_are_rejected_without_a_device(lib):
    null = ctypes.c_void_p(0)
    # bad dtype / negative sizes
    assert lib.sq_quantize_rowwise_i8(null, 7, 1, 1, 1, null, null, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8(null, 0, -1, 1, 1, null, null, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8(null, 0, 2, 8, 4, null, null, null) == sq.SQ_ERR_INVALID_ARG
    # empty input is a no-op
    assert lib.sq_quantize_rowwise_i8(null, 0, 0, 8, 8, null, null, null) == sq.SQ_OK
    # fp8: bad fmt, missing scale
    assert lib.sq_quantize_fp8(null, 16, null, 5, null, null, null, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8(null, 16, null, 0, null, null, null, null) == sq.SQ_ERR_INVALID_ARG
    # misaligned FP8 operands
    p1 = ctypes.c_void_p(0x1001)
    p = ctypes.c_void_p(0x1000)
    assert lib.sq_quantize_fp8(p1, 16, p, 0, p, p, p, null) == sq.SQ_ERR_ALIGNMENT
    # several tensors in one launch: count 1..4, entries as for one tensor
    arr = (ctypes.c_void_p * 2)(p, p)
    arr_mis = (ctypes.c_void_p * 2)(p, p1)
    arr_null = (ctypes.c_void_p * 2)(p, null)
    n2 = (ctypes.c_int64 * 2)(16, 16)
    n_neg = (ctypes.c_int64 * 2)(16, -1)
    assert lib.sq_quantize_fp8_multi(0, arr, n2, arr, 0, arr, arr, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8_multi(5, arr, n2, arr, 0, arr, arr, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8_multi(2, arr, n2, arr, 3, arr, arr, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8_multi(2, arr, n_neg, arr, 0, arr, arr, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8_multi(2, arr, n2, arr_null, 0, arr, arr, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_fp8_multi(2, arr_mis, n2, arr, 0, arr, arr, p, null) == sq.SQ_ERR_ALIGNMENT
    # both INT8 operands quantized and staged: bad dtype, short pitch, missing output
    assert lib.sq_quantize_rowwise_i8_staged_pair(p, 16, p, 16, 7, 1, 4, 4, 16, p, p, p, p, p, 1 << 20,
                                                  null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8_staged_pair(p, 8, p, 16, 0, 1, 4, 4, 16, p, p, p, p, p, 1 << 20,
                                                  null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8_staged_pair(p, 16, p, 16, 0, 1, 4, 4, 16, p, p, null, p, p,
                                                  1 << 20, null) == sq.SQ_ERR_INVALID_ARG
    # two GEMMs in one call: each problem checked as one GEMM, and an output
    # may not meet the other problem's operands or output
    def q(*vals, t=ctypes.c_void_p):
        return (t * 2)(*vals)
    PA, PB = q(0x10000, 0x20000), q(0x30000, 0x40000)
    P16 = q(16, 16, t=ctypes.c_int64)
    assert lib.sq_gemm_fp8_scaled_pair(PA, PB, PA, PB, 0, q(0, 9, t=ctypes.c_int), P16, P16, P16,
                                       q(0x50000, 0x60000), null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_fp8_scaled_pair(PA, PB, PA, PB, 0, q(0, 0, t=ctypes.c_int), P16, P16,
                                       q(16, 24, t=ctypes.c_int64), q(0x50000, 0x60000),
                                       null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_fp8_scaled_pair(PA, PB, PA, PB, 0, q(0, 1, t=ctypes.c_int), P16, P16, P16,
                                       q(0x50000, 0x10000), null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_fp8_scaled_pair(PA, PB, PA, PB, 0, q(0, 2, t=ctypes.c_int), P16, P16, P16,
                                       q(0x50000, 0x50100), null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_fp8_scaled_pair(null, PB, PA, PB, 0, q(0, 0, t=ctypes.c_int), P16, P16, P16,
                                       q(0x50000, 0x60000), null) == sq.SQ_ERR_INVALID_ARG
    # gemm: bad layout, K not a multiple of 16, K too long
    assert lib.sq_gemm_fp8_scaled(p, p, p, p, 0, 9, 16, 16, 16, p, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_fp8_scaled(p, p, p, p, 0, 0, 16, 16, 24, p, null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_fp8_scaled(p, p, p, p, 0, 1, 16, 24, 32, p, null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_fp8_scaled(p, p, p, p, 0, 2, 24, 16, 32, p, null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_fp8_scaled(p1, p, p, p, 0, 0, 16, 16, 16, p, null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_i8_rowscaled(p, p, p, p, 1, 4, 4, 24, 96, 96, 16, p, null, p, 1 << 20,
                                    null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_i8_rowscaled(p, p, p, p, 1, 4, 4, 1 << 18, 1 << 20, 1 << 20, 16, p, null,
                                    p, 1 << 30, null) == sq.SQ_ERR_UNSUPPORTED
    assert lib.sq_gemm_i8_rowscaled(p, p, p, p, 1, 4, 4, 16, 64, 64, 16, null, null, p, 1 << 20,
                                    null) == sq.SQ_ERR_INVALID_ARG
    # workspace too small
    assert lib.sq_gemm_i8_rowscaled(p, p, p, p, 1, 4, 4, 16, 64, 64, 16, p, null, p, 8,
                                    null) == sq.SQ_ERR_INVALID_ARG
    # the two phases check the same sizes, strides and workspace
    assert lib.sq_gemm_i8_stage(p, p, 1, 4, 4, 24, 96, 96, p, 1 << 20, null) == sq.SQ_ERR_ALIGNMENT
    assert lib.sq_gemm_i8_stage(null, p, 1, 4, 4, 16, 64, 64, p, 1 << 20,
                                null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_i8_stage(p, p, 1, 4, 4, 16, 64, 64, p, 8, null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_i8_rowscaled_staged(p, p, 1, 4, 4, 16, 16, null, null, p, 1 << 20,
                                           null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_i8_rowscaled_staged(p, p, 1, 4, 4, 16, 8, p, null, p, 1 << 20,
                                           null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_gemm_i8_rowscaled_staged(p, p, 1, 4, 4, 16, 16, p1, null, p, 1 << 20,
                                           null) == sq.SQ_ERR_ALIGNMENT
    # the fused quantize-and-stage: operand, rows and cols must match the GEMM's shape
    assert lib.sq_quantize_rowwise_i8_staged(p, 0, 4, 16, 16, p, p, 2, 1, 4, 4, 16, p, 1 << 20,
                                             null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8_staged(p, 0, 5, 16, 16, p, p, 0, 1, 4, 4, 16, p, 1 << 20,
                                             null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8_staged(p, 0, 4, 32, 32, p, p, 1, 1, 4, 4, 16, p, 1 << 20,
                                             null) == sq.SQ_ERR_INVALID_ARG
    assert lib.sq_quantize_rowwise_i8_staged(p, 0, 4, 16, 16, p, p, 1, 1, 4, 4, 16, p, 8,
                                             null) == sq.SQ_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        sq.sq_quantize_rowwise_i8(torch.zeros(4, 16))


def test_binding_checks_dtypes_and_sizes_before_calling(lib, monkeypatch):
    """The wrappers reject wrong dtypes, scale lengths and output shapes before
    anything reaches the library (the CUDA checks are bypassed: these tensors
    are on the CPU and the library is never called)."""
    import torch
    monkeypatch.setattr(sq, "_need_cuda", lambda *ts: None)
    a = torch.zeros(4, 16, dtype=torch.int8)
    b = torch.zeros(6, 16, dtype=torch.int8)
    with pytest.raises(TypeError):
        sq._i8_operands(a.float(), b, torch.ones(4), torch.ones(6))
    with pytest.raises(ValueError, match="sA"):
        sq._i8_operands(a, b, torch.ones(3), torch.ones(6))
    with pytest.raises(ValueError, match="sB"):
        sq._i8_operands(a, b, torch.ones(4), torch.ones(4))
    with pytest.raises(TypeError, match="sA"):
        sq._i8_operands(a, b, torch.ones(4, dtype=torch.float64), torch.ones(6))
    with pytest.raises(ValueError, match="share"):
        sq._i8_operands(a, torch.zeros(6, 32, dtype=torch.int8), torch.ones(4), torch.ones(6))
    # grouped scales: ceil(rows / group) per batch
    sq._i8_operands(a, b, torch.ones(2), torch.ones(1), group_a=2, group_b=6)
    with pytest.raises(ValueError, match="C"):
        sq._i8_outputs(torch.zeros(4, 5), None, True, (4, 6), "cpu")
    with pytest.raises(TypeError, match="acc_out"):
        sq._i8_outputs(None, torch.zeros(4, 6, dtype=torch.int64), False, (4, 6), "cpu")
    with pytest.raises(ValueError, match="acc_out"):
        sq._i8_outputs(None, torch.zeros(4, 5, dtype=torch.int32), False, (4, 6), "cpu")
    u = torch.zeros(8, 32, dtype=torch.uint8)
    assert sq._fp8_shape(u, torch.zeros(16, 32, dtype=torch.uint8), sq.SQ_NT) == (8, 16, 32)
    assert sq._fp8_shape(u, torch.zeros(32, 16, dtype=torch.uint8), sq.SQ_NN) == (8, 16, 32)
    assert sq._fp8_shape(u.t().contiguous(), torch.zeros(32, 16, dtype=torch.uint8),
                         sq.SQ_TN) == (8, 16, 32)
    with pytest.raises(ValueError, match="share K"):
        sq._fp8_shape(u, torch.zeros(16, 48, dtype=torch.uint8), sq.SQ_NT)
    with pytest.raises(TypeError):
        sq._fp8_shape(u.to(torch.int8), torch.zeros(16, 32, dtype=torch.uint8), sq.SQ_NT)


def test_clock_record_summary_on_the_host():
    """clock_probe_mhz: cycles over nanoseconds per CTA, unused (zero) rows
    left out, and the launch's span from first start to last end."""
    import torch
    rec = torch.zeros(8 * 4, dtype=torch.int64)
    # CTA 0: 2000 cycles in 1000 ns (2000 MHz); CTA 1: 1500 cycles in 1000 ns
    rec[0:4] = torch.tensor([100, 2100, 5000, 6000])
    rec[4:8] = torch.tensor([7, 1507, 5100, 6100])
    s = sq.clock_probe_mhz(rec)
    assert s["ctas"] == 2 and s["max"] == 2000.0 and s["min"] == 1500.0
    assert s["span_ns"] == 1100 and s["cycles_median"] in (1500.0, 2000.0, 1750.0)
    assert sq.clock_probe_mhz(torch.zeros(16, dtype=torch.int64)) == {}


def test_quantize_and_stage_binding_checks_the_operand_shape(lib, monkeypatch):
    import torch
    monkeypatch.setattr(sq, "_need_cuda", lambda *ts: None)
    x = torch.zeros(4, 16, dtype=torch.float32)
    ws = torch.zeros(1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="operand"):
        sq.sq_quantize_rowwise_i8_staged(x, 0, (0, 5, 4, 16), ws)      # A must have M rows
    with pytest.raises(ValueError, match="operand"):
        sq.sq_quantize_rowwise_i8_staged(x, 1, (0, 4, 4, 32), ws)      # cols must equal K
    with pytest.raises(TypeError):
        sq.sq_quantize_rowwise_i8_staged(x.to(torch.float64), 0, (0, 4, 4, 16), ws)
