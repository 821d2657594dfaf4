"""The stream argument: the FP8 and INT8 paths running at the same time on
two streams, each with its own workspaces, give bit-for-bit the results of
the same calls made one after another on one stream (every kernel here is
deterministic)."""
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import synth
from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def run_fp8(x, w, sx, sw, ws, stream):
    x8, ax = sq.sq_quantize_fp8(x, sx, sq.SQ_FMT_E4M3, ws, stream=stream)
    w8, aw = sq.sq_quantize_fp8(w, sw, sq.SQ_FMT_E4M3, ws, stream=stream)
    c = sq.sq_gemm_fp8_scaled(x8, w8, sx, sw, sq.SQ_FMT_E4M3, sq.SQ_NT, stream=stream)
    return x8, ax, c


def run_i8(a, b, wsi, stream):
    qa, sa = sq.sq_quantize_rowwise_i8(a, stream=stream)
    qb, sb = sq.sq_quantize_rowwise_i8(b, stream=stream)
    c, _ = sq.sq_gemm_i8_rowscaled(qa, sa, qb, sb, wsi, stream=stream)
    return qa, sa, c


def test_two_streams_match_one_stream():
    M, N, K = 2048, 1536, 2048
    x = to_dev(synth.normal(71, (M, K), dtype=synth.BF16), True)
    w = to_dev(synth.normal(72, (N, K), std=0.02, dtype=synth.BF16), True)
    a = to_dev(synth.student_t(73, (M, K), dtype=synth.BF16), True)
    b = to_dev(synth.student_t(74, (N, K), dtype=synth.BF16), True)
    sx = torch.tensor([float(x.float().abs().max()) / 448.0], device=DEV)
    sw = torch.tensor([float(w.float().abs().max()) / 448.0], device=DEV)
    nbytes = sq.gemm_i8_workspace_bytes(1, M, N, K)

    main = torch.cuda.current_stream()
    ref_fp8 = run_fp8(x, w, sx, sw, sq.new_workspace(DEV), main)
    ref_i8 = run_i8(a, b, torch.empty(nbytes, dtype=torch.uint8, device=DEV), main)
    torch.cuda.synchronize()

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = sq.new_workspace(DEV)
    wsi2 = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    s1.wait_stream(main)
    s2.wait_stream(main)
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            f = run_fp8(x, w, sx, sw, ws1, s1)
        with torch.cuda.stream(s2):
            i = run_i8(a, b, wsi2, s2)
        outs.append((f, i))
    main.wait_stream(s1)
    main.wait_stream(s2)
    torch.cuda.synchronize()
    for f, i in outs:
        for got, want in zip(f, ref_fp8):
            assert torch.equal(got, want)
        for got, want in zip(i, ref_i8):
            assert torch.equal(got, want)
