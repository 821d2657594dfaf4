"""Pins for the oracle's FP8 codec, its bf16 rounding and its integer rounding.

The codec is checked against what does not depend on it: torch's float8 and
bfloat16 dtypes (library routines), the format's closed-form special values,
and a brute-force nearest-value search over the 256 decoded codes.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

FMTS = [(oracle.E4M3, torch.float8_e4m3fn, 448.0, 2.0 ** -9),
        (oracle.E5M2, torch.float8_e5m2, 57344.0, 2.0 ** -16)]


@pytest.mark.parametrize("fmt,tdt,fmax,fmin", FMTS)
def test_decode_matches_torch_float8(fmt, tdt, fmax, fmin):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(tdt).to(torch.float64).numpy()
    got = oracle.fp8_decode_table(fmt)
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(want[~nan], got[~nan])


@pytest.mark.parametrize("fmt,tdt,fmax,fmin", FMTS)
def test_special_values(fmt, tdt, fmax, fmin):
    tab = oracle.fp8_decode_table(fmt)
    finite = tab[np.isfinite(tab)]
    assert finite.max() == fmax and finite.min() == -fmax
    assert np.min(finite[finite > 0]) == fmin
    one = 0x38 if fmt == oracle.E4M3 else 0x3C
    assert tab[one] == 1.0
    assert tab[0x00] == 0.0 and np.signbit(tab[0x80])
    if fmt == oracle.E5M2:
        assert tab[0x7C] == np.inf and tab[0xFC] == -np.inf
        assert all(oracle.fp8_code_is_nan(c, fmt) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    else:
        assert oracle.fp8_code_is_nan(0x7F, fmt) and oracle.fp8_code_is_nan(0xFF, fmt)
        assert np.sum(np.isnan(tab)) == 2
    # positive finite codes decode strictly increasing
    pos = tab[:0x80]
    pos = pos[np.isfinite(pos)]
    assert np.all(np.diff(pos) > 0)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_every_code_round_trips(fmt):
    tab = oracle.fp8_decode_table(fmt)
    for c in range(256):
        v = tab[c]
        if np.isnan(v):
            nan_bits = np.uint32(0xFFC00000 if c & 0x80 else 0x7FC00000)
            e = oracle.fp8_encode(nan_bits.view(np.float32), fmt)
            assert oracle.fp8_code_is_nan(int(e), fmt) and (int(e) & 0x80) == (c & 0x80)
            continue
        if np.isinf(v):
            # infinity saturates to the largest finite value of the same sign
            assert int(oracle.fp8_encode(np.float32(v), fmt)) == (c & 0x80) | 0x7B
            continue
        assert int(oracle.fp8_encode(np.float32(v), fmt)) == c, hex(c)


def brute_force_encode(t, fmt):
    """Nearest finite code of the same sign; ties go to the even code."""
    tab = oracle.fp8_decode_table(fmt)
    codes = np.arange(256)
    ok = np.isfinite(tab)
    out = np.empty(t.shape, dtype=np.uint8)
    fmax = np.max(tab[ok])
    # beyond 2*fmax every value has the same nearest finite code (fmax); clipping
    # there keeps the fp64 distances exact enough to compare
    td = np.clip(t.astype(np.float64), -2 * fmax, 2 * fmax)
    for sgn in (0, 1):
        sel = ok & ((codes >> 7) == sgn)
        cand_c = codes[sel]
        cand_v = tab[sel]
        m = np.signbit(t) == bool(sgn)
        if not m.any():
            continue
        tt = td[m][:, None]
        d = np.abs(tt - cand_v[None, :])
        dmin = d.min(axis=1, keepdims=True)
        tie = d == dmin
        # among equally near codes prefer the even one (mantissa LSB 0)
        score = np.where(tie, (cand_c[None, :] & 1), 2)
        pick = np.argmin(score, axis=1)
        out[m] = cand_c[pick]
    return out


def probe_points(fmt):
    tab = oracle.fp8_decode_table(fmt)
    vals = np.unique(tab[np.isfinite(tab)])
    mids = (vals[:-1] + vals[1:]) / 2
    fmax = vals.max()
    base = np.concatenate([vals, mids, [fmax * 1.0001, fmax * 1.5, fmax * 2, 1e30, 3e38]])
    base32 = base.astype(np.float32)
    pts = [base32]
    for k in range(1, 5):  # +-4 ulp around every code value and every midpoint
        pts.append(np.nextafter(base32, np.float32(np.inf)))
        pts.append(np.nextafter(base32, np.float32(-np.inf)))
        base32 = np.concatenate([np.nextafter(base32, np.float32(np.inf)),
                                 np.nextafter(base32, np.float32(-np.inf))])
    p = np.concatenate(pts)
    return np.unique(np.concatenate([p, -p]))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encoder_equals_brute_force_near_codes_and_ties(fmt):
    t = probe_points(fmt)
    assert np.array_equal(oracle.fp8_encode(t, fmt), brute_force_encode(t, fmt))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encoder_equals_brute_force_random(fmt):
    fmax = 448.0 if fmt == oracle.E4M3 else 57344.0
    rng = np.random.default_rng(1234 + fmt)
    for _ in range(10):
        t = rng.uniform(-2 * fmax, 2 * fmax, size=100_000).astype(np.float32)
        # also log-uniform magnitudes so every binade and the subnormals are hit
        mag = np.exp(rng.uniform(np.log(1e-9), np.log(2 * fmax), size=100_000))
        t2 = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
        for tt in (t, t2):
            assert np.array_equal(oracle.fp8_encode(tt, fmt), brute_force_encode(tt, fmt))


@pytest.mark.parametrize("fmt,tdt,fmax,fmin", FMTS)
def test_encoder_matches_torch_in_range(fmt, tdt, fmax, fmin):
    """torch's float32 -> float8 cast rounds to nearest even; it agrees with the
    saturating encoder on every value that does not overflow."""
    rng = np.random.default_rng(99)
    mag = np.exp(rng.uniform(np.log(1e-8), np.log(fmax), size=200_000))
    t = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    t = np.concatenate([t, probe_points(fmt)])
    t = t[np.abs(t) <= fmax]
    want = torch.from_numpy(t).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_encode(t, fmt), want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_saturation_and_signed_zero(fmt):
    big = np.array([1e6, -1e6, np.inf, -np.inf, 3.4e38], dtype=np.float32)
    mc = 0x7E if fmt == oracle.E4M3 else 0x7B
    assert list(oracle.fp8_encode(big, fmt)) == [mc, 0x80 | mc, mc, 0x80 | mc, mc]
    z = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-45, -1e-45], dtype=np.float32)
    assert list(oracle.fp8_encode(z, fmt)) == [0, 0x80, 0, 0x80, 0, 0x80]


def test_round_half_even_printed_examples():
    """The tie examples printed on the POPCORNBENCH trace page."""
    for t, even, away in read_golden("round_half_even_ties.txt"):
        assert oracle.round_half_even(float(t)) == int(even)
        assert oracle.round_half_even(float(t)) == int(np.rint(np.float32(t)))
        assert int(away) != int(even) or abs(float(t)) == 1.5


def test_round_half_even_vs_rint():
    rng = np.random.default_rng(7)
    t = np.concatenate([rng.uniform(-200, 200, 20000).astype(np.float32),
                        (np.arange(-400, 401) / 2).astype(np.float32),
                        np.nextafter(np.float32(np.arange(-300, 301) / 2 + 0.0),
                                     np.float32(np.inf)),
                        np.nextafter(np.float32(np.arange(-300, 301) / 2 + 0.0),
                                     np.float32(-np.inf))])
    got = np.array([oracle.round_half_even(v) for v in t])
    assert np.array_equal(got, np.rint(t).astype(np.int64))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 1e3,
                        # exact ties: low 16 bits = 0x8000
                        (rng.integers(0, 2**15, 2000, dtype=np.uint32) << 16 | 0x8000)
                        .astype(np.uint32).view(np.float32)])
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_round(v) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)
