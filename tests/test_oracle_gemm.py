"""Pins for the oracle's INT8 and FP8 GEMMs: brute force on tiny shapes, library
products, closed forms, layout equivalences and the lossless special case."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


def rand_i8(rng, shape):
    return rng.integers(-127, 128, size=shape, dtype=np.int64).astype(np.int8)


def test_i8_tiny_brute_force():
    rng = np.random.default_rng(1)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (8, 8, 8), (2, 7, 3)]:
        A, B = rand_i8(rng, (M, K)), rand_i8(rng, (N, K))
        acc, _ = oracle.gemm_i8(A, B)
        for i in range(M):
            for j in range(N):
                assert acc[i, j] == sum(int(A[i, k]) * int(B[j, k]) for k in range(K))


def test_i8_against_numpy_int64_and_extremes():
    rng = np.random.default_rng(2)
    A, B = rand_i8(rng, (37, 300)), rand_i8(rng, (29, 300))
    acc, _ = oracle.gemm_i8(A, B)
    assert np.array_equal(acc, A.astype(np.int64) @ B.astype(np.int64).T)
    K = 8192
    A = np.full((2, K), 127, np.int8)
    A[1] = -127
    B = np.full((3, K), 127, np.int8)
    acc, _ = oracle.gemm_i8(A, B)
    assert acc[0, 0] == 127 * 127 * K and acc[1, 2] == -127 * 127 * K


def test_i8_overflow_is_reported():
    K = 140_000   # 127^2 * K > 2^31 - 1
    A = np.full((1, K), 127, np.int8)
    with pytest.raises(OverflowError):
        oracle.gemm_i8(A, A)


def test_i8_identity_and_dequant_closed_form():
    rng = np.random.default_rng(3)
    K = 64
    A = np.zeros((K, K), np.int8)
    np.fill_diagonal(A, 1)
    B = rand_i8(rng, (10, K))
    acc, _ = oracle.gemm_i8(A, B)
    assert np.array_equal(acc, B.T.astype(np.int32))
    # power-of-two scales and small sums: the dequant is exact
    sa = (2.0 ** rng.integers(-10, 10, K)).astype(np.float32)
    sb = (2.0 ** rng.integers(-10, 10, 10)).astype(np.float32)
    acc, C = oracle.gemm_i8(A, B, sa, sb)
    assert np.array_equal(C.astype(np.float64),
                          acc.astype(np.float64) * sa[:, None].astype(np.float64) * sb[None, :])


def test_i8_dequant_rounds_left_to_right():
    """(float(acc) * sa) * sb in float32, each product rounded: numpy float32
    arithmetic does the same two IEEE multiplies."""
    rng = np.random.default_rng(4)
    A, B = rand_i8(rng, (20, 2048)), rand_i8(rng, (30, 2048))
    sa = synth.normal(5, (20,)) ** 2 + np.float32(0.01)
    sb = synth.normal(6, (30,)) ** 2 + np.float32(0.01)
    acc, C = oracle.gemm_i8(A, B, sa, sb)
    want = (acc.astype(np.float32) * sa[:, None]) * sb[None, :]
    assert np.array_equal(C, want)


def test_i8_batched_and_row_subset():
    rng = np.random.default_rng(7)
    A, B = rand_i8(rng, (4, 19, 64)), rand_i8(rng, (4, 23, 64))
    sa = np.abs(synth.normal(8, (4, 19))) + np.float32(0.1)
    sb = np.abs(synth.normal(9, (4, 23))) + np.float32(0.1)
    acc, C = oracle.gemm_i8(A, B, sa, sb)
    for h in range(4):
        a2, c2 = oracle.gemm_i8(A[h], B[h], sa[h], sb[h])
        assert np.array_equal(acc[h], a2) and np.array_equal(C[h], c2)
    rows = np.array([0, 5, 18])
    accr, Cr = oracle.gemm_i8(A, B, sa, sb, rows=rows)
    assert np.array_equal(accr, acc[:, rows]) and np.array_equal(Cr, C[:, rows])


# ------------------------------------------------------------------ FP8
def rand_codes(rng, shape, fmt):
    tab = oracle.fp8_decode_table(fmt)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c])], dtype=np.uint8)
    return rng.choice(ok, size=shape)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_fp8_nt_tiny_exact_rationals(fmt):
    rng = np.random.default_rng(10 + fmt)
    tab = oracle.fp8_decode_table(fmt)
    M, N, K = 5, 6, 8
    A, B = rand_codes(rng, (M, K), fmt), rand_codes(rng, (N, K), fmt)
    sa, sb = np.float32(0.37), np.float32(1.9)
    ref, _ = oracle.gemm_fp8(A, B, fmt, oracle.NT, sa, sb)
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(tab[A[i, k]]) * Fraction(tab[B[j, k]]) for k in range(K))
            exact = exact * Fraction(float(sa)) * Fraction(float(sb))
            assert abs(Fraction(ref[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_fp8_layouts_agree_with_numpy(fmt):
    rng = np.random.default_rng(20 + fmt)
    tab = oracle.fp8_decode_table(fmt)
    M, N, K = 33, 17, 96
    A, B = rand_codes(rng, (M, K), fmt), rand_codes(rng, (N, K), fmt)
    want = tab[A] @ tab[B].T * 0.5 * 0.25
    nt, _ = oracle.gemm_fp8(A, B, fmt, oracle.NT, 0.5, 0.25)
    nn, _ = oracle.gemm_fp8(A, np.ascontiguousarray(B.T), fmt, oracle.NN, 0.5, 0.25)
    tn, _ = oracle.gemm_fp8(np.ascontiguousarray(A.T), np.ascontiguousarray(B.T), fmt,
                            oracle.TN, 0.5, 0.25)
    scale = np.abs(tab[A]) @ np.abs(tab[B]).T * 0.125
    for got in (nt, nn, tn):
        assert np.all(np.abs(got - want) <= 1e-12 * scale + 1e-300)
    # a plausible slip (NN fed the NT operand) is caught
    if M == N:
        bad, _ = oracle.gemm_fp8(A, B, fmt, oracle.NN, 0.5, 0.25)
        assert not np.allclose(bad, want)


def test_fp8_layout_slip_is_caught():
    rng = np.random.default_rng(30)
    tab = oracle.fp8_decode_table(oracle.E4M3)
    A, B = rand_codes(rng, (16, 16), 0), rand_codes(rng, (16, 16), 0)
    want = tab[A] @ tab[B].T
    for layout in (oracle.NN, oracle.TN):
        bad, _ = oracle.gemm_fp8(A, B, 0, layout, 1.0, 1.0)
        assert not np.allclose(bad, want)


def test_fp8_identity_closed_form():
    rng = np.random.default_rng(31)
    K = 32
    I = np.zeros((K, K), np.uint8)
    np.fill_diagonal(I, 0x38)   # E4M3 1.0
    B = rand_codes(rng, (9, K), 0)
    tab = oracle.fp8_decode_table(0)
    ref, _ = oracle.gemm_fp8(I, B, 0, oracle.NT, 2.0, 0.5)
    assert np.array_equal(ref, tab[B].T)


def test_fp8_bf16_output_is_rne_of_scaled_float32():
    rng = np.random.default_rng(32)
    A, B = rand_codes(rng, (12, 64), 0), rand_codes(rng, (14, 64), 0)
    sa, sb = np.float32(0.013), np.float32(0.77)
    ref, bf = oracle.gemm_fp8(A, B, 0, oracle.NT, sa, sb)
    import torch
    raw = (ref / float(sa) / float(sb))  # the unscaled fp64 sums (exact here)
    f = (raw.astype(np.float32) * sa) * sb
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(bf, want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_quantized_gemm_lossless_special_case(fmt):
    """Inputs equal to code * 2^e with power-of-two scales quantize exactly, so
    the quantized GEMM equals the fp64 GEMM of the raw inputs."""
    rng = np.random.default_rng(40 + fmt)
    M, N, K = 24, 20, 64
    tab = oracle.fp8_decode_table(fmt)
    ca = rand_codes(rng, (M, K), fmt)
    cb = rand_codes(rng, (N, K), fmt)
    ea, eb = -3, 2
    xa = (tab[ca] * 2.0 ** ea).astype(np.float32)
    xb = (tab[cb] * 2.0 ** eb).astype(np.float32)
    bits_a = (xa.view(np.uint32) >> 16).astype(np.uint16)
    bits_b = (xb.view(np.uint32) >> 16).astype(np.uint16)
    a8, _ = oracle.quantize_fp8(bits_a, 2.0 ** ea, fmt)
    b8, _ = oracle.quantize_fp8(bits_b, 2.0 ** eb, fmt)
    ref, _ = oracle.gemm_fp8(a8, b8, fmt, oracle.NT, 2.0 ** ea, 2.0 ** eb)
    direct = xa.astype(np.float64) @ xb.astype(np.float64).T
    scale = np.abs(xa.astype(np.float64)) @ np.abs(xb.astype(np.float64)).T
    assert np.all(np.abs(ref - direct) <= 1e-13 * scale)


def test_fp8_row_subset():
    rng = np.random.default_rng(50)
    A, B = rand_codes(rng, (40, 32), 0), rand_codes(rng, (16, 32), 0)
    full, fb = oracle.gemm_fp8(A, B, 0, oracle.NT, 1.0, 1.0)
    rows = np.array([0, 7, 39])
    part, pb = oracle.gemm_fp8(A, B, 0, oracle.NT, 1.0, 1.0, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pb, fb[rows])


# ------------------------------------------------------------------ E4M3 output
def test_fp8_e4m3_output_identity_closed_form():
    """A = identity (E4M3 1.0), sa = sb = 1: the output codes are B^T's codes
    scaled by 1/out_scale -- identical for out_scale = 1, one binade down for
    out_scale = 2 (so a multiply-instead-of-divide slip shows)."""
    rng = np.random.default_rng(60)
    K = 48
    I = np.zeros((K, K), np.uint8)
    np.fill_diagonal(I, 0x38)
    tab = oracle.fp8_decode_table(0)
    # B codes with magnitudes in [2^-5, 2^7] so halving stays exact in E4M3
    ok = np.array([c for c in range(256) if np.isfinite(tab[c]) and 2 ** -5 <= abs(tab[c]) <= 2 ** 7],
                  dtype=np.uint8)
    B = rng.choice(ok, size=(20, K))
    _, codes1 = oracle.gemm_fp8_e4m3(I, B, 0, oracle.NT, 1.0, 1.0, 1.0)
    assert np.array_equal(codes1, B.T)
    t2, codes2 = oracle.gemm_fp8_e4m3(I, B, 0, oracle.NT, 1.0, 1.0, 2.0)
    assert np.array_equal(tab[codes2], tab[B.T] / 2) and np.array_equal(t2, tab[B.T] / 2)


def test_fp8_e4m3_output_saturates_and_brackets():
    rng = np.random.default_rng(61)
    A, B = rand_codes(rng, (30, 64), 0), rand_codes(rng, (24, 64), 0)
    t, codes = oracle.gemm_fp8_e4m3(A, B, 0, oracle.NT, 0.5, 0.25, 1e-3)
    tab = oracle.fp8_decode_table(0)
    assert np.all(np.abs(tab[codes][np.abs(t) > 500]) == 448.0)
    assert np.all(oracle.e4m3_acceptable(codes, t, 1e-9 * np.abs(t) + 1e-30))


def test_grouped_gemm_reduces_to_rowscaled_and_broadcasts_group_scales():
    rng = np.random.default_rng(70)
    A, B = rand_i8(rng, (2, 20, 64)), rand_i8(rng, (2, 30, 64))
    sa = np.abs(synth.normal(71, (2, 20))) + np.float32(0.1)
    sb = np.abs(synth.normal(72, (2, 30))) + np.float32(0.1)
    acc1, C1 = oracle.gemm_i8(A, B, sa, sb)
    acc2, C2 = oracle.gemm_i8_grouped(A, B, sa, sb, 1, 1)
    assert np.array_equal(acc1, acc2) and np.array_equal(C1, C2)
    # group sizes 8 (A) and 30 (B, per tensor): the same as expanding the scales
    ga_s = np.abs(synth.normal(73, (2, 3))) + np.float32(0.1)
    gb_s = np.abs(synth.normal(74, (2, 1))) + np.float32(0.1)
    _, Cg = oracle.gemm_i8_grouped(A, B, ga_s, gb_s, 8, 30)
    _, Ce = oracle.gemm_i8(A, B, np.repeat(ga_s, 8, axis=1)[:, :20], np.repeat(gb_s, 30, axis=1))
    assert np.array_equal(Cg, Ce)


# ------------------------------------------------------------------ linear layer pieces
def test_gemm_bias_adds_the_bias_after_scaling():
    rng = np.random.default_rng(80)
    A, B = rand_codes(rng, (17, 64), 0), rand_codes(rng, (23, 64), 0)
    bias = synth.normal(81, (23,), std=3.0)
    ref0, bf0 = oracle.gemm_fp8(A, B, 0, oracle.NT, 0.3, 0.7)
    ref1, bf1 = oracle.gemm_fp8_bias(A, B, 0, oracle.NT, 0.3, 0.7, bias)
    assert np.allclose(ref1 - ref0, bias[None, :].astype(np.float64), rtol=0, atol=1e-12)
    refn, bfn = oracle.gemm_fp8_bias(A, B, 0, oracle.NT, 0.3, 0.7, None)
    assert np.array_equal(refn, ref0) and np.array_equal(bfn, bf0)


def test_fp8_bias_decode_is_code_times_step():
    tab = oracle.fp8_decode_table(1)
    codes = np.array([0x00, 0x3C, 0xBC, 0x7B, 0x01], dtype=np.uint8)
    out = oracle.fp8_bias_to_f32(codes, 1, 0.5)
    assert list(out) == [0.0, 0.5, -0.5, 57344.0 * 0.5, 2.0 ** -16 * 0.5]
    assert np.array_equal(out, (tab[codes] * 0.5).astype(np.float32))


def test_colsum_matches_numpy():
    g = synth.normal(82, (300, 40), dtype=synth.BF16)
    want = synth.bf16_bits_to_f32(g).astype(np.float64).sum(axis=0)
    assert np.allclose(oracle.colsum_bf16(g), want, rtol=1e-15, atol=1e-15)


def test_oracle_results_do_not_depend_on_the_thread_count():
    """The OpenMP loops split rows between threads; every output element is
    still summed in one fixed order, so one thread and all threads agree bit
    for bit (the one-core timing in bench.py relies on this too)."""
    rng = np.random.default_rng(91)
    qa = rng.integers(-127, 128, (37, 300)).astype(np.int8)
    qb = rng.integers(-127, 128, (41, 300)).astype(np.int8)
    sa = rng.uniform(0.1, 2.0, 37).astype(np.float32)
    sb = rng.uniform(0.1, 2.0, 41).astype(np.float32)
    a8 = rng.integers(0, 0x7F, (33, 256)).astype(np.uint8)
    b8 = rng.integers(0, 0x7F, (29, 256)).astype(np.uint8)
    n = oracle.num_threads()
    try:
        many = (oracle.gemm_i8(qa, qb, sa, sb), oracle.gemm_fp8(a8, b8, 0, oracle.NT, 0.01, 0.02))
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1
        one = (oracle.gemm_i8(qa, qb, sa, sb), oracle.gemm_fp8(a8, b8, 0, oracle.NT, 0.01, 0.02))
    finally:
        oracle.set_num_threads(n)
    for x, y in zip(many[0] + many[1], one[0] + one[1]):
        assert np.array_equal(np.asarray(x), np.asarray(y))
