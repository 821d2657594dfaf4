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


# ------------------------------------------------------------------ delayed-scaling ring
def _ring(H, scale, hist=None):
    r = np.zeros(H + 2, dtype=np.float32)
    if hist is not None:
        r[:H] = hist
    r[H] = scale
    return r


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_ring_quantizes_with_the_ring_scale_and_records_amax(fmt):
    x = synth.normal(120, (300, 64), dtype=synth.BF16)
    ring = _ring(8, 0.01, hist=[0.5, 0, 0, 0, 0, 0, 0, 0])
    x8, amax = oracle.quantize_fp8_ring(x, fmt, ring, idx=3)
    plain8, plain_amax = oracle.quantize_fp8(x, 0.01, fmt)
    assert np.array_equal(x8, plain8) and amax == plain_amax
    assert ring[3] == amax and ring[0] == np.float32(0.5)
    assert np.all(ring[[1, 2, 4, 5, 6, 7]] == 0) and ring[9] == 0   # counter untouched


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_published_step_maps_the_window_max_to_the_largest_code(fmt):
    """At margin 0 the next step sends the history's max to the largest finite
    FP8 code, not past it (no saturation of the window max)."""
    rng = np.random.default_rng(3)
    for _ in range(50):
        hist = rng.uniform(1e-3, 1e3, size=16).astype(np.float32)
        ring = _ring(16, 1.0, hist)
        x = (np.zeros(32, dtype=np.uint16))
        oracle.quantize_fp8_ring(x, fmt, ring, idx=int(rng.integers(0, 16)), margin=0)
        m = np.float32(ring[:16].max())
        code = int(oracle.fp8_encode(np.float32(m) / ring[16], fmt))
        assert code == (0x7E if fmt == oracle.E4M3 else 0x7B)


def test_ring_margin_doubles_the_step_and_follows_the_delayed_recipe():
    x = synth.normal(121, (512,), std=2.0, dtype=synth.BF16)
    steps = []
    for margin in (0, 1, 2, 5):
        ring = _ring(4, 0.02)
        oracle.quantize_fp8_ring(x, oracle.E4M3, ring, idx=0, margin=margin)
        steps.append(ring[4])
    assert steps[1] == 2 * steps[0] and steps[2] == 4 * steps[0] and steps[3] == 32 * steps[0]
    # margin 0 with one entry: the previous-amax / 448 recipe of the delayed-scale workload
    amax = np.abs(synth.bf16_bits_to_f32(x)).max()
    assert steps[0] == np.float32(amax) / np.float32(448.0)


def test_ring_keeps_the_scale_when_the_history_is_zero_and_rolls_the_window():
    ring = _ring(3, 0.125)
    oracle.quantize_fp8_ring(np.zeros(64, dtype=np.uint16), oracle.E4M3, ring, idx=1)
    assert ring[3] == np.float32(0.125) and np.all(ring[:3] == 0)
    # a large amax leaves the window after H further steps
    big = synth.normal(122, (64,), std=100.0, dtype=synth.BF16)
    small = synth.normal(123, (64,), std=0.01, dtype=synth.BF16)
    oracle.quantize_fp8_ring(big, oracle.E4M3, ring, idx=0)
    s_big = ring[3]
    oracle.quantize_fp8_ring(small, oracle.E4M3, ring, idx=1)
    oracle.quantize_fp8_ring(small, oracle.E4M3, ring, idx=2)
    assert ring[3] == s_big                 # the big amax is still in the window
    oracle.quantize_fp8_ring(small, oracle.E4M3, ring, idx=0)
    assert ring[3] < s_big / 100            # now it has rolled out


# ------------------------------------------------------------------ row groups / per tensor
def test_grouped_with_one_row_per_group_is_per_row():
    x = synth.normal(130, (37, 96))
    qg, sg = oracle.quantize_grouped_i8(x, 1)
    qr, sr = oracle.quantize_rowwise_i8(x)
    assert np.array_equal(qg, qr) and np.array_equal(sg, sr)


def test_per_tensor_follows_the_printed_fake_quant_formula():
    """The POPCORNBENCH trace's reference model: amax = max|x| clamped at 1e-8,
    scale = amax / 127, q = clamp(round_half_even(x / scale), -127, 127)."""
    x = synth.student_t(131, (50, 70), df=3)
    q, s = oracle.quantize_grouped_i8(x, 50)
    assert s.shape == (1,)
    amax = np.float32(max(np.abs(x).max(), np.float32(1e-8)))
    assert s[0] == amax / np.float32(127.0)
    t = x / s[0]
    assert np.array_equal(q, brute_force_int8(t))
    # only the tensor's absmax element reaches +-127
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert abs(int(q[i])) == 127


def test_groups_are_independent_and_row_order_inside_a_group_does_not_matter():
    x = synth.normal(132, (40, 64))
    x[10:20] *= 50.0                          # group 1 (rows 8..15 with g=8) gets a big row
    q, s = oracle.quantize_grouped_i8(x, 8)
    assert s.shape == (5,)
    for g in range(5):
        qg, sg = oracle.quantize_grouped_i8(np.ascontiguousarray(x[8 * g:8 * g + 8]), 8)
        assert sg[0] == s[g] and np.array_equal(qg, q[8 * g:8 * g + 8])
    perm = np.concatenate([np.random.default_rng(1).permutation(8) + 8 * g for g in range(5)])
    qp, sp = oracle.quantize_grouped_i8(np.ascontiguousarray(x[perm]), 8)
    assert np.array_equal(sp, s) and np.array_equal(qp, q[perm])
    # ragged last group
    q7, s7 = oracle.quantize_grouped_i8(x, 7)
    assert s7.shape == (6,)
    qlast, slast = oracle.quantize_grouped_i8(np.ascontiguousarray(x[35:]), 5)
    assert slast[0] == s7[5] and np.array_equal(qlast, q7[35:])
