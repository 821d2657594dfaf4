"""Full-size parity for the large workload (M=16384, N=8192, K=8192, bf16
Student-t(3) inputs), run through the same entry points and launch
configuration the benchmark times: quantized tensors and amax compared in
full, GEMM outputs on a seeded sample of rows."""
import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, bf16_to_f64, to_dev

pytestmark = pytest.mark.gpu

M, N, K = 16384, 8192, 8192
SAMPLE_ROWS = 48


@pytest.fixture(scope="module")
def inputs():
    a = synth.student_t(501, (M, K), df=3, dtype=synth.BF16)
    b = synth.student_t(502, (N, K), df=3, dtype=synth.BF16)
    return a, b


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def test_large_fp8_e4m3_nt(inputs):
    a, b = inputs
    pa = synth.bf16_bits_to_f32(synth.student_t(601, (M, K), df=3, dtype=synth.BF16))
    pb = synth.bf16_bits_to_f32(synth.student_t(602, (N, K), df=3, dtype=synth.BF16))
    sa = np.float32(np.abs(pa).max()) / np.float32(448.0)
    sb = np.float32(np.abs(pb).max()) / np.float32(448.0)
    del pa, pb
    ws = sq.new_workspace(DEV)
    tsa, tsb = torch.tensor([sa], device=DEV), torch.tensor([sb], device=DEV)
    a8, amax_a = sq.sq_quantize_fp8(to_dev(a, bf16=True), tsa, 0, ws)
    b8, amax_b = sq.sq_quantize_fp8(to_dev(b, bf16=True), tsb, 0, ws)
    oa8, oamax_a = oracle.quantize_fp8(a, sa, 0)
    ob8, oamax_b = oracle.quantize_fp8(b, sb, 0)
    assert amax_a.item() == float(oamax_a) and amax_b.item() == float(oamax_b)
    assert np.array_equal(a8.cpu().numpy(), oa8)
    assert np.array_equal(b8.cpu().numpy(), ob8)
    C = sq.sq_gemm_fp8_scaled(a8, b8, tsa, tsb, 0, sq.SQ_NT)
    rows = np.sort(np.random.default_rng(7).choice(M, SAMPLE_ROWS, replace=False))
    ref, _ = oracle.gemm_fp8(oa8, ob8, 0, oracle.NT, sa, sb, rows=rows, want_bf16=False)
    tab = oracle.fp8_decode_table(0)
    bound = oracle.fp8_gemm_bound(ref, K, sa, sb, np.abs(tab[oa8]).max(), np.abs(tab[ob8]).max())
    got = bf16_to_f64(C[torch.from_numpy(rows).to(DEV)])
    assert np.all(np.abs(got - ref) <= bound)


def test_large_int8_per_row(inputs):
    a, b = inputs
    qa, sa = sq.sq_quantize_rowwise_i8(to_dev(a, bf16=True))
    qb, sb = sq.sq_quantize_rowwise_i8(to_dev(b, bf16=True))
    oqa, osa = oracle.quantize_rowwise_i8(a, oracle.BF16)
    oqb, osb = oracle.quantize_rowwise_i8(b, oracle.BF16)
    assert np.array_equal(sa.cpu().numpy(), osa) and np.array_equal(sb.cpu().numpy(), osb)
    assert np.array_equal(qa.cpu().numpy(), oqa)
    assert np.array_equal(qb.cpu().numpy(), oqb)
    ws = torch.empty(sq.gemm_i8_workspace_bytes(1, M, N, K), dtype=torch.uint8, device=DEV)
    C, acc = sq.sq_gemm_i8_rowscaled(qa, sa, qb, sb, ws, acc_out=True)
    rows = np.sort(np.random.default_rng(8).choice(M, SAMPLE_ROWS, replace=False))
    oacc, oC = oracle.gemm_i8(oqa, oqb, osa, osb, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert np.array_equal(acc[ridx].cpu().numpy(), oacc)
    assert np.array_equal(C[ridx].cpu().numpy(), oC)


def test_large_int8_per_row_quantized_and_staged(inputs):
    """The benchmark's INT8 path: each operand quantized and staged in one
    launch (sq_quantize_rowwise_i8_staged), then the staged GEMM; codes and
    scales in full, GEMM outputs on sampled rows, and the same bits as the
    one-call form on those rows."""
    a, b = inputs
    ws = torch.empty(sq.gemm_i8_workspace_bytes(1, M, N, K), dtype=torch.uint8, device=DEV)
    shape = (0, M, N, K)
    A, B = to_dev(a, bf16=True), to_dev(b, bf16=True)
    qa, sa = sq.sq_quantize_rowwise_i8_staged(A, 0, shape, ws)
    qb, sb = sq.sq_quantize_rowwise_i8_staged(B, 1, shape, ws)
    C, acc = sq.sq_gemm_i8_rowscaled_staged(sa, sb, shape, ws, acc_out=True)
    oqa, osa = oracle.quantize_rowwise_i8(a, oracle.BF16)
    oqb, osb = oracle.quantize_rowwise_i8(b, oracle.BF16)
    assert np.array_equal(sa.cpu().numpy(), osa) and np.array_equal(sb.cpu().numpy(), osb)
    assert np.array_equal(qa.cpu().numpy(), oqa)
    assert np.array_equal(qb.cpu().numpy(), oqb)
    rows = np.sort(np.random.default_rng(9).choice(M, SAMPLE_ROWS, replace=False))
    oacc, oC = oracle.gemm_i8(oqa, oqb, osa, osb, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert np.array_equal(acc[ridx].cpu().numpy(), oacc)
    assert np.array_equal(C[ridx].cpu().numpy(), oC)
    ws1 = torch.empty_like(ws)
    C1, acc1 = sq.sq_gemm_i8_rowscaled(qa, sa, qb, sb, ws1, acc_out=True)
    assert torch.equal(C1[ridx], C[ridx]) and torch.equal(acc1[ridx], acc[ridx])
