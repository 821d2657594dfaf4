"""One long stream of mixed calls that share their workspaces.

Every quantize (FP8 and INT8, small and streamed sizes) and every GEMM shape
(single-CTA 128- and 256-wide tiles, CTA pairs, batched heads; NT, NN, TN)
runs back to back on one stream. One FP8 workspace and one INT8 GEMM
workspace serve all of them, and nothing is read back until the end. Each
result must still equal the oracle, which shows that no call leaves state
behind for the next: the self-resetting amax words, the INT8 staging buffers
and bounds, and the per-device launch set-up. A repeated call must reproduce
its first result bit for bit.
"""
import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, bf16_to_f64, to_dev

pytestmark = pytest.mark.gpu


def _step(seed, shape, std, fmt):
    """A delayed step: the amax of a second draw of the same distribution."""
    prev = synth.bf16_bits_to_f32(synth.normal(seed + 1, shape, std=std, dtype=synth.BF16))
    fmax = 448.0 if fmt == sq.SQ_FMT_E4M3 else 57344.0
    return np.float32(np.abs(prev).max()) / np.float32(fmax)


def _check_fp8_gemm(out, A8, B8, fmt, layout, K, sa, sb, rows):
    ref, _ = oracle.gemm_fp8(A8, B8, fmt, layout, sa, sb, rows=rows)
    tab = oracle.fp8_decode_table(fmt)
    bound = oracle.fp8_gemm_bound(ref, K, sa, sb, np.abs(tab[A8]).max(), np.abs(tab[B8]).max())
    got = bf16_to_f64(out)[rows]
    assert np.all(np.abs(got - ref) <= bound)


def test_mixed_call_sequence_shares_workspaces():
    fp8_ws = sq.new_workspace(DEV)
    i8_shapes = [(1, 300, 260, 2048), (16, 196, 196, 64), (1, 2200, 2300, 1040), (1, 128, 512, 1024)]
    i8_ws = torch.empty(max(sq.gemm_i8_workspace_bytes(*s) for s in i8_shapes),
                        dtype=torch.uint8, device=DEV)

    # ---- inputs (host arrays for the oracle, device copies for the calls)
    fp8_in = {
        "X": (synth.normal(901, (2048, 1024), dtype=synth.BF16), 1.0, sq.SQ_FMT_E4M3),
        "W": (synth.normal(903, (1024, 1024), std=0.02, dtype=synth.BF16), 0.02, sq.SQ_FMT_E4M3),
        "tiny": (synth.normal(905, (33,), dtype=synth.BF16), 1.0, sq.SQ_FMT_E5M2),
        "G": (synth.normal(907, (2048, 4096), std=1e-3, dtype=synth.BF16), 1e-3, sq.SQ_FMT_E4M3),
        "P": (synth.normal(909, (2200, 384), dtype=synth.BF16), 1.0, sq.SQ_FMT_E4M3),
        "Q": (synth.normal(911, (384, 2208), std=0.02, dtype=synth.BF16), 0.02, sq.SQ_FMT_E4M3),
    }
    seeds = {"X": 901, "W": 903, "tiny": 905, "G": 907, "P": 909, "Q": 911}
    steps = {k: _step(seeds[k], v[0].shape, v[1], v[2]) for k, v in fp8_in.items()}
    i8_in = {
        "a1": synth.student_t(921, (300, 2048), dtype=synth.BF16),
        "b1": synth.normal(922, (260, 2048)),
        "qh": synth.normal(923, (16, 196, 64)),
        "kh": synth.normal(924, (16, 196, 64)),
        "a3": synth.normal(925, (2200, 1040)),
        "b3": synth.normal(926, (2300, 1040)),
        "a4": synth.normal(927, (128, 1024)),
        "b4": synth.normal(928, (512, 1024)),
    }
    bf16_keys = {"a1"}

    # ---- the sequence: no host synchronisation until every call is queued
    out = {}
    d_step = {k: torch.tensor([v], dtype=torch.float32, device=DEV) for k, v in steps.items()}

    def q8(key):
        x8, amax = sq.sq_quantize_fp8(to_dev(fp8_in[key][0], bf16=True), d_step[key],
                                      fp8_in[key][2], fp8_ws)
        out["x8_" + key], out["amax_" + key] = x8, amax
        return x8

    def qi8(key):
        q, s = sq.sq_quantize_rowwise_i8(to_dev(i8_in[key], bf16=(key in bf16_keys)))
        out["q_" + key], out["s_" + key] = q, s
        return q, s

    def gi8(name, ka, kb):
        qa, sa = out["q_" + ka], out["s_" + ka]
        qb, sb = out["q_" + kb], out["s_" + kb]
        out["C_" + name], out["acc_" + name] = sq.sq_gemm_i8_rowscaled(
            qa, sa.reshape(-1), qb, sb.reshape(-1), i8_ws, acc_out=True)

    x8 = q8("X")
    q8("tiny")
    qi8("a1")
    qi8("b1")
    gi8("1", "a1", "b1")                                   # 128-wide single tiles, staged store
    w8 = q8("W")
    out["fwd"] = sq.sq_gemm_fp8_scaled(x8, w8, d_step["X"], d_step["W"], sq.SQ_FMT_E4M3, sq.SQ_NT)
    qi8("qh")
    qi8("kh")
    gi8("heads", "qh", "kh")                               # batched heads
    p8, q8_ = q8("P"), q8("Q")
    out["nn_pair"] = sq.sq_gemm_fp8_scaled(p8, q8_, d_step["P"], d_step["Q"],
                                           sq.SQ_FMT_E4M3, sq.SQ_NN)  # CTA pairs, MN-major B
    qi8("a3")
    qi8("b3")
    gi8("pair", "a3", "b3")                                # CTA pairs, some CTAs run two tiles
    g8 = q8("G")                                           # streamed FP8 quantize
    out["tn"] = sq.sq_gemm_fp8_scaled(g8, x8, d_step["G"], d_step["X"],
                                      sq.SQ_FMT_E4M3, sq.SQ_TN)  # dW = G^T X
    qi8("a4")
    qi8("b4")
    gi8("cfg1", "a4", "b4")
    first_C1 = out["C_1"].clone()
    gi8("1", "a1", "b1")                                   # the first INT8 GEMM again
    torch.cuda.synchronize()
    assert sq.sq_get_last_device_error() == sq.SQ_OK

    # ---- every result against the oracle
    for key, (x, _, fmt) in fp8_in.items():
        ox8, oamax = oracle.quantize_fp8(x, steps[key], fmt)
        assert np.array_equal(out["x8_" + key].cpu().numpy(), ox8), key
        assert out["amax_" + key].item() == float(oamax), key
    assert int(fp8_ws.sum().item()) == 0

    oq = {}
    for key, x in i8_in.items():
        q, s = oracle.quantize_rowwise_i8(x, oracle.BF16 if key in bf16_keys else oracle.F32)
        assert np.array_equal(out["q_" + key].cpu().numpy(), q), key
        assert np.array_equal(out["s_" + key].cpu().numpy(), s), key
        oq[key] = (q, s)

    for name, ka, kb, rows in (("1", "a1", "b1", None), ("heads", "qh", "kh", None),
                               ("pair", "a3", "b3", np.r_[0:4, 1100:1104, 2196:2200]),
                               ("cfg1", "a4", "b4", None)):
        (qa, sa), (qb, sb) = oq[ka], oq[kb]
        oacc, oC = oracle.gemm_i8(qa, qb, sa.reshape(-1), sb.reshape(-1), rows=rows)
        acc, C = out["acc_" + name].cpu().numpy(), out["C_" + name].cpu().numpy()
        if rows is not None:
            acc, C = acc[rows], C[rows]
        assert np.array_equal(acc, oacc), name
        assert np.array_equal(C, oC), name
    assert torch.equal(out["C_1"], first_C1)

    x8h, w8h = out["x8_X"].cpu().numpy(), out["x8_W"].cpu().numpy()
    _check_fp8_gemm(out["fwd"], x8h, w8h, 0, sq.SQ_NT, 1024, steps["X"], steps["W"],
                    np.r_[0:8, 1000:1008, 2040:2048])
    _check_fp8_gemm(out["nn_pair"], out["x8_P"].cpu().numpy(), out["x8_Q"].cpu().numpy(), 0,
                    sq.SQ_NN, 384, steps["P"], steps["Q"], np.r_[0:8, 1024:1032, 2192:2200])
    g8h = out["x8_G"].cpu().numpy()
    _check_fp8_gemm(out["tn"], g8h, x8h, 0, sq.SQ_TN, 2048, steps["G"], steps["X"],
                    np.r_[0:8, 2048:2056, 4088:4096])
