"""GPU parity of the fused FP8 linear forward and backward against the oracle.

Forward: quantized operands and amax bit-exact, output within the FP8 GEMM
bound (plus the bias), rings bit-exact, pre-quantized weights and bias.
Backward: one gradient quantization feeding dX (NN) and dW (TN), the bias
gradient, the masks, and a gradient ring.
"""
import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, bf16_to_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def prev_step(seed, shape, std, fmt):
    p = synth.bf16_bits_to_f32(synth.normal(seed, shape, std=std, dtype=synth.BF16))
    return np.float32(np.abs(p).max()) / np.float32(448.0 if fmt == 0 else 57344.0)


def check_out(out, ref, K, sa, sb, a8, b8, fmt, rows=None):
    tab = oracle.fp8_decode_table(fmt)
    bound = oracle.fp8_gemm_bound(ref, K, sa, sb, np.abs(tab[a8]).max(), np.abs(tab[b8]).max())
    got = bf16_to_f64(out)
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"


def sample_rows(M, n, seed):
    r = np.random.default_rng(seed).choice(M, min(n, M), replace=False)
    return np.unique(np.concatenate([r, [0, M - 1]]))


@pytest.mark.parametrize("fmt", [0, 1], ids=["e4m3", "e5m2"])
def test_forward_with_bf16_bias(fmt):
    M, K, N = 2048, 1024, 1024
    x = synth.normal(201, (M, K), std=1.0, dtype=synth.BF16)
    w = synth.normal(202, (N, K), std=0.02, dtype=synth.BF16)
    b = synth.normal(203, (N,), std=0.5, dtype=synth.BF16)
    sx, sw = prev_step(204, (M, K), 1.0, fmt), prev_step(205, (N, K), 0.02, fmt)
    ws = sq.linear_workspace(M, N, K, DEV)
    out, x8, w8, ax, aw = sq.sq_linear_forward_fp8(
        to_dev(x, True), to_dev(w, True), to_dev(b, True), torch.tensor([sx], device=DEV),
        torch.tensor([sw], device=DEV), fmt, ws)
    ox8, oax = oracle.quantize_fp8(x, sx, fmt)
    ow8, oaw = oracle.quantize_fp8(w, sw, fmt)
    assert np.array_equal(x8.cpu().numpy(), ox8) and np.array_equal(w8.cpu().numpy(), ow8)
    assert ax.item() == float(oax) and aw.item() == float(oaw)
    rows = sample_rows(M, 200, 1)
    ref, obf = oracle.gemm_fp8_bias(ox8, ow8, fmt, oracle.NT, sx, sw,
                                    synth.bf16_bits_to_f32(b), rows=rows)
    check_out(out, ref, K, sx, sw, ox8, ow8, fmt, rows)
    same = np.mean(out.view(torch.int16).cpu().numpy().astype(np.uint16)[rows] == obf)
    assert same > 0.9


def test_forward_rings_use_the_old_step_and_publish_the_next():
    M, K, N = 512, 256, 384
    fmt = 0
    H = 4
    xr_o = np.zeros(H + 2, np.float32)
    wr_o = np.zeros(H + 2, np.float32)
    xr_o[H], wr_o[H] = 0.01, 0.0001
    xr, wr = sq.new_ring(H, 0.01, DEV), sq.new_ring(H, 0.0001, DEV)
    ws = sq.linear_workspace(M, N, K, DEV)
    for step in range(3):
        x = synth.normal(210 + step, (M, K), std=1.0 + step, dtype=synth.BF16)
        w = synth.normal(220 + step, (N, K), std=0.02, dtype=synth.BF16)
        sx_used, sw_used = xr_o[H], wr_o[H]
        out, x8, w8, ax, aw = sq.sq_linear_forward_fp8(
            to_dev(x, True), to_dev(w, True), None, None, None, fmt, ws,
            x_ring=xr, x_ring_idx=step % H, w_ring=wr, w_ring_idx=step % H, w_ring_margin=1)
        ox8, oax = oracle.quantize_fp8_ring(x, fmt, xr_o, idx=step % H)
        ow8, oaw = oracle.quantize_fp8_ring(w, fmt, wr_o, idx=step % H, margin=1)
        assert np.array_equal(x8.cpu().numpy(), ox8) and np.array_equal(w8.cpu().numpy(), ow8)
        assert np.array_equal(xr.cpu().numpy().view(np.uint32), xr_o.view(np.uint32))
        assert np.array_equal(wr.cpu().numpy().view(np.uint32), wr_o.view(np.uint32))
        ref, _ = oracle.gemm_fp8_bias(ox8, ow8, fmt, oracle.NT, sx_used, sw_used, None)
        check_out(out, ref, K, sx_used, sw_used, ox8, ow8, fmt)


def test_forward_prequantized_weight_and_fp8_bias():
    M, K, N = 300, 512, 272
    fmt = 0
    x = synth.normal(231, (M, K), dtype=synth.BF16)
    w = synth.normal(232, (N, K), std=0.02, dtype=synth.BF16)
    sx, sw = prev_step(233, (M, K), 1.0, fmt), prev_step(234, (N, K), 0.02, fmt)
    ow8, _ = oracle.quantize_fp8(w, sw, fmt)
    bias_step = np.float32(0.01)
    b = synth.normal(235, (N,), std=0.5, dtype=synth.BF16)
    ob8, _ = oracle.quantize_fp8(b, bias_step, fmt)
    ws = sq.linear_workspace(M, N, K, DEV)
    out, x8, w8, ax, aw = sq.sq_linear_forward_fp8(
        to_dev(x, True), to_dev(ow8), to_dev(ob8), torch.tensor([sx], device=DEV),
        torch.tensor([sw], device=DEV), fmt, ws, bias_scale=torch.tensor([bias_step], device=DEV),
        w_prequantized=True)
    assert aw.item() == 0.0
    ox8, _ = oracle.quantize_fp8(x, sx, fmt)
    assert np.array_equal(x8.cpu().numpy(), ox8)
    bias_f = oracle.fp8_bias_to_f32(ob8, fmt, bias_step)
    ref, _ = oracle.gemm_fp8_bias(ox8, ow8, fmt, oracle.NT, sx, sw, bias_f)
    check_out(out, ref, K, sx, sw, ox8, ow8, fmt)


@pytest.mark.parametrize("fmt", [1, 0], ids=["e5m2", "e4m3"])
def test_backward_mlp_shapes(fmt):
    """dim 1024, hidden 4096, 2048 tokens: out = x w^T, g = dout."""
    T, N, K = 2048, 4096, 1024
    g = synth.normal(241, (T, N), std=1e-3, dtype=synth.BF16)
    w = synth.normal(242, (N, K), std=0.02, dtype=synth.BF16)
    x = synth.normal(243, (T, K), std=1.0, dtype=synth.BF16)
    sg, sw, sx = prev_step(244, (T, N), 1e-3, fmt), prev_step(245, (N, K), 0.02, fmt), \
        prev_step(246, (T, K), 1.0, fmt)
    ws = sq.linear_workspace(T, N, K, DEV)
    gx, gw, gb, ag = sq.sq_linear_backward_fp8(
        to_dev(g, True), to_dev(x, True), to_dev(w, True), (True, True, True),
        torch.tensor([sg], device=DEV), torch.tensor([sw], device=DEV),
        torch.tensor([sx], device=DEV), fmt, ws)
    og8, oag = oracle.quantize_fp8(g, sg, fmt)
    ow8, _ = oracle.quantize_fp8(w, sw, fmt)
    ox8, _ = oracle.quantize_fp8(x, sx, fmt)
    assert ag.item() == float(oag)
    rows = sample_rows(T, 96, 2)
    ref, _ = oracle.gemm_fp8(og8, ow8, fmt, oracle.NN, sg, sw, rows=rows, want_bf16=False)
    check_out(gx, ref, N, sg, sw, og8, ow8, fmt, rows)
    rows = sample_rows(N, 96, 3)
    ref, _ = oracle.gemm_fp8(og8, ox8, fmt, oracle.TN, sg, sx, rows=rows, want_bf16=False)
    check_out(gw, ref, T, sg, sx, og8, ox8, fmt, rows)
    want = oracle.colsum_bf16(g)
    gmax = np.abs(synth.bf16_bits_to_f32(g)).max()
    tol = 2.0 ** -8 * np.abs(want) + T * gmax * 2.0 ** -22
    assert np.all(np.abs(bf16_to_f64(gb) - want) <= tol)


def test_backward_masks_ragged_tokens_and_gradient_ring():
    T, N, K = 2000, 256, 512
    fmt = 1
    g = synth.normal(251, (T, N), std=1e-2, dtype=synth.BF16)
    w = synth.normal(252, (N, K), std=0.02, dtype=synth.BF16)
    x = synth.normal(253, (T, K), dtype=synth.BF16)
    sw, sx = prev_step(254, (N, K), 0.02, fmt), prev_step(255, (T, K), 1.0, fmt)
    H = 3
    gr_o = np.zeros(H + 2, np.float32)
    gr_o[H] = 1e-6
    gr = sq.new_ring(H, 1e-6, DEV)
    ws = sq.linear_workspace(T, N, K, DEV)
    # only the weight gradient and the bias gradient; the step comes from the ring
    gx, gw, gb, ag = sq.sq_linear_backward_fp8(
        to_dev(g, True), to_dev(x, True), to_dev(w, True), (False, True, True), None,
        torch.tensor([sw], device=DEV), torch.tensor([sx], device=DEV), fmt, ws,
        g_ring=gr, g_ring_idx=1)
    assert gx is None
    sg_used = gr_o[H]
    og8, oag = oracle.quantize_fp8_ring(g, fmt, gr_o, idx=1)
    assert np.array_equal(gr.cpu().numpy().view(np.uint32), gr_o.view(np.uint32))
    assert ag.item() == float(oag)
    ox8, _ = oracle.quantize_fp8(x, sx, fmt)
    ref, _ = oracle.gemm_fp8(og8, ox8, fmt, oracle.TN, sg_used, sx, want_bf16=False)
    check_out(gw, ref, T, sg_used, sx, og8, ox8, fmt)
    want = oracle.colsum_bf16(g)
    gmax = np.abs(synth.bf16_bits_to_f32(g)).max()
    tol = 2.0 ** -8 * np.abs(want) + T * gmax * 2.0 ** -22
    assert np.all(np.abs(bf16_to_f64(gb) - want) <= tol)
    # only the input gradient
    gx, gw, gb, _ = sq.sq_linear_backward_fp8(
        to_dev(g, True), to_dev(x, True), to_dev(w, True), (True, False, False),
        torch.tensor([sg_used], device=DEV), torch.tensor([sw], device=DEV),
        torch.tensor([sx], device=DEV), fmt, ws)
    assert gw is None and gb is None
    og8b, _ = oracle.quantize_fp8(g, sg_used, fmt)
    ow8, _ = oracle.quantize_fp8(w, sw, fmt)
    ref, _ = oracle.gemm_fp8(og8b, ow8, fmt, oracle.NN, sg_used, sw, want_bf16=False)
    check_out(gx, ref, N, sg_used, sw, og8b, ow8, fmt)


@pytest.mark.parametrize("T,N", [(5, 1008), (1000, 1008), (64, 16)],
                         ids=["T5 empty slabs", "T1000", "N16 one partial block"])
def test_backward_bias_gradient_ragged_columns(T, N):
    """The bias gradient alone, on a partial 128-column block and on fewer
    tokens than row slabs; the same bits on a second call."""
    K = 64
    fmt = 0
    g = synth.normal(261 + T, (T, N), std=1e-2, dtype=synth.BF16)
    x = synth.normal(262, (T, K), dtype=synth.BF16)
    w = synth.normal(263, (N, K), std=0.02, dtype=synth.BF16)
    ws = sq.linear_workspace(T, N, K, DEV)
    sg = torch.tensor([prev_step(264, (T, N), 1e-2, fmt)], device=DEV)
    args = (to_dev(g, True), to_dev(x, True), to_dev(w, True), (False, False, True), sg, None, None,
            fmt, ws)
    gx, gw, gb, _ = sq.sq_linear_backward_fp8(*args)
    assert gx is None and gw is None and gb.shape == (N,)
    want = oracle.colsum_bf16(g)
    gmax = np.abs(synth.bf16_bits_to_f32(g)).max()
    tol = 2.0 ** -8 * np.abs(want) + T * gmax * 2.0 ** -22
    assert np.all(np.abs(bf16_to_f64(gb) - want) <= tol)
    _, _, gb2, _ = sq.sq_linear_backward_fp8(*args)
    assert torch.equal(gb.view(torch.int16), gb2.view(torch.int16))
