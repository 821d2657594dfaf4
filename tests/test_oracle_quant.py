"""Pins for the oracle's INT8 per-row and FP8 per-tensor quantizers."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden


def brute_force_int8(t):
    """argmin over n in [-127, 127] of |t - n|, ties to the even n."""
    n = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(t.astype(np.float64)[..., None] - n)
    dmin = d.min(axis=-1, keepdims=True)
    score = np.where(d == dmin, np.abs(n) % 2, 2)
    return (np.argmin(score, axis=-1) - 127).astype(np.int8)


def test_printed_ties_through_the_quantizer():
    """A row whose absmax is 127 has scale exactly 1, so x/scale = x and the
    printed tie examples (POPCORNBENCH trace, rounding discussion) pass
    through the quantizer unchanged."""
    ties = read_golden("round_half_even_ties.txt")
    x = np.array([[127.0] + [float(t) for t, _, _ in ties]], dtype=np.float32)
    q, s = oracle.quantize_rowwise_i8(x)
    assert s[0] == np.float32(1.0)
    assert list(q[0]) == [127] + [int(e) for _, e, _ in ties]


def test_int8_matches_brute_force_and_rint():
    x = synth.normal(101, (64, 333))
    x[3] *= 1e-3
    x[5, 7] = 40.0        # outlier row
    q, s = oracle.quantize_rowwise_i8(x)
    t = x / s[:, None]    # numpy float32 division is one IEEE operation
    assert t.dtype == np.float32
    assert np.array_equal(q, brute_force_int8(t))
    assert np.array_equal(q, np.clip(np.rint(t), -127, 127).astype(np.int8))


def test_int8_many_exact_ties():
    # absmax 127 -> scale 1; every other element is an exact half
    rng = np.random.default_rng(5)
    x = (rng.integers(-250, 251, size=(16, 64)) / 2).astype(np.float32)
    x[:, 0] = 127.0
    q, s = oracle.quantize_rowwise_i8(x)
    assert np.all(s == 1.0)
    assert np.array_equal(q, brute_force_int8(x))


def test_int8_invariants():
    x = synth.student_t(102, (200, 257), df=3)
    q, s = oracle.quantize_rowwise_i8(x)
    assert np.abs(q.astype(np.int32)).max() <= 127
    amax = np.abs(x).max(axis=1)
    # the absmax element of every row encodes to +-127
    idx = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(200), idx].astype(np.int32)) == 127)
    assert np.all(np.sign(q[np.arange(200), idx]) == np.sign(x[np.arange(200), idx]))
    # scale is the absmax step: amax/127 rounded once
    assert np.array_equal(s, (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32))
    # dequantized error is at most half a step (values never clip: |t| <= 127ish)
    err = np.abs(q.astype(np.float64) * s[:, None] - x)
    assert np.all(err <= 0.5 * s[:, None].astype(np.float64) * (1 + 1e-6))


def test_int8_power_of_two_scaling_invariance():
    x = synth.normal(103, (8, 100))
    q1, s1 = oracle.quantize_rowwise_i8(x)
    for k in (-20, -3, 5, 30):
        q2, s2 = oracle.quantize_rowwise_i8((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(q1, q2)
        assert np.array_equal(s2, s1 * np.float32(2.0 ** k))


def test_int8_zero_and_tiny_rows_use_the_floor():
    x = np.zeros((3, 40), dtype=np.float32)
    x[1, 5] = 1e-12           # below the 1e-8 floor
    x[2, :] = -0.0
    q, s = oracle.quantize_rowwise_i8(x)
    floor_scale = np.float32(1e-8) / np.float32(127.0)
    assert np.all(s == floor_scale)
    assert np.all(q == 0)


def test_int8_per_row_not_per_tensor():
    x = synth.normal(104, (4, 64))
    x[0] *= 100.0
    q, s = oracle.quantize_rowwise_i8(x)
    assert len(set(s.tolist())) == 4
    assert np.all(np.abs(q.astype(np.int32)).max(axis=1) == 127)


def test_int8_bf16_input_equals_widened_f32():
    xb = synth.normal(105, (32, 96), dtype=synth.BF16)
    xf = synth.bf16_bits_to_f32(xb)
    qb, sb = oracle.quantize_rowwise_i8(xb, oracle.BF16)
    qf, sf = oracle.quantize_rowwise_i8(xf, oracle.F32)
    assert np.array_equal(qb, qf) and np.array_equal(sb, sf)
    # bf16 widening agrees with torch's
    tw = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(tw, xf)


def test_per_head_is_per_row_within_each_head():
    x = synth.normal(106, (16, 196, 64))
    q3, s3 = oracle.quantize_rowwise_i8(x)
    q2, s2 = oracle.quantize_rowwise_i8(x.reshape(-1, 64))
    assert q3.shape == (16, 196, 64) and s3.shape == (16, 196)
    assert np.array_equal(q3.reshape(-1, 64), q2) and np.array_equal(s3.reshape(-1), s2)


# ------------------------------------------------------------------ FP8 per tensor
@pytest.mark.parametrize("fmt,tdt", [(oracle.E4M3, torch.float8_e4m3fn),
                                     (oracle.E5M2, torch.float8_e5m2)])
def test_fp8_quantize_against_torch(fmt, tdt):
    x = synth.normal(107, (257, 129), std=1.0, dtype=synth.BF16)
    xf = synth.bf16_bits_to_f32(x)
    prev = synth.bf16_bits_to_f32(synth.normal(108, (257, 129), dtype=synth.BF16))
    fmax = 448.0 if fmt == oracle.E4M3 else 57344.0
    scale = np.float32(np.abs(prev).max()) / np.float32(fmax)
    x8, amax = oracle.quantize_fp8(x, scale, fmt)
    # amax is the raw max|x| (library reduction)
    assert amax == np.abs(xf).max()
    t = xf / scale
    inr = np.abs(t) <= fmax
    want = torch.from_numpy(t[inr]).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(x8[inr], want)
    # outside the range the codes saturate with the input's sign
    mc = 0x7E if fmt == oracle.E4M3 else 0x7B
    sat = x8[~inr]
    assert np.all((sat & 0x7F) == mc)
    assert np.array_equal(sat >> 7, np.signbit(t[~inr]).astype(np.uint8))


def test_fp8_amax_permutation_invariant_and_raw():
    x = synth.student_t(109, (5000,), dtype=synth.BF16)
    _, a1 = oracle.quantize_fp8(x, 0.01, oracle.E4M3)
    perm = np.random.default_rng(0).permutation(x.size)
    _, a2 = oracle.quantize_fp8(x[perm], 0.01, oracle.E4M3)
    assert a1 == a2 == np.abs(synth.bf16_bits_to_f32(x)).max()
    _, a0 = oracle.quantize_fp8(np.zeros(100, dtype=np.uint16), 1.0, oracle.E4M3)
    assert a0 == 0.0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_fp8_lossless_when_input_is_code_times_power_of_two(fmt):
    """x = decode(c) * 2^e with scale = 2^e quantizes back to c exactly."""
    tab = oracle.fp8_decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(tab[c])], dtype=np.uint8)
    for e in (-4, 0, 3):
        vals = (tab[codes] * 2.0 ** e).astype(np.float32)
        bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
        # these values are exact in bf16 (<= 4 significant bits)
        assert np.array_equal(synth.bf16_bits_to_f32(bits), vals)
        x8, amax = oracle.quantize_fp8(bits, np.float32(2.0 ** e), fmt)
        # +0 and -0 both decode to 0; the encoder keeps the sign of the input
        assert np.array_equal(x8, codes)
        assert amax == np.abs(vals).max()
