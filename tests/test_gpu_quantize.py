"""GPU parity of the quantize kernels against the oracle: bit-exact INT8 codes,
row scales, FP8 codes and amax, on the pages' shapes plus ragged, strided,
degenerate and long-row cases."""
import zlib

import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, guard_intact, guarded, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert sq.sq_get_last_device_error() == sq.SQ_OK


ROW_CASES = [
    # (name, shape, dtype, draw)
    ("int8 per-row A 128x1024 f32", (128, 1024), "f32", "normal"),
    ("int8 per-row B 512x1024 f32", (512, 1024), "f32", "normal"),
    ("int8 per-head Q 16x196x64 f32", (16, 196, 64), "f32", "normal"),
    ("bf16 t3 300x8192 (CTA per row)", (300, 8192), "bf16", "t3"),
    ("bf16 64x2048", (64, 2048), "bf16", "normal"),
    ("f32 7x4096", (7, 4096), "f32", "t3"),
    ("f32 ragged 37x17 (scalar path)", (37, 17), "f32", "normal"),
    ("bf16 long rows 5x40000 (scalar path)", (5, 40000), "bf16", "t3"),
    ("f32 tiny rows 1000x16", (1000, 16), "f32", "normal"),
    ("bf16 1x8", (1, 8), "bf16", "normal"),
    # enough rows of 4-16 KB to take the bulk-copy pipeline
    ("bulk bf16 1000x2048", (1000, 2048), "bf16", "normal"),
    ("bulk f32 700x4096", (700, 4096), "f32", "t3"),
    ("bulk bf16 t3 900x6144", (900, 6144), "bf16", "t3"),
]


def draw(seed, shape, dt, kind):
    d = synth.F32 if dt == "f32" else synth.BF16
    if kind == "t3":
        return synth.student_t(seed, shape, df=3, dtype=d)
    return synth.normal(seed, shape, dtype=d)


@pytest.mark.parametrize("name,shape,dt,kind", ROW_CASES, ids=[c[0] for c in ROW_CASES])
def test_rowwise_i8_parity(name, shape, dt, kind):
    x = draw(zlib.crc32(name.encode()) % 1000 + 10, shape, dt, kind)
    oq, osc = oracle.quantize_rowwise_i8(x, oracle.F32 if dt == "f32" else oracle.BF16)
    q, s = sq.sq_quantize_rowwise_i8(to_dev(x, bf16=(dt == "bf16")))
    assert np.array_equal(s.cpu().numpy(), osc)
    assert np.array_equal(q.cpu().numpy(), oq)


def test_rowwise_i8_strided_rows_and_guard():
    full = synth.normal(21, (96, 1040))
    xd = to_dev(full)[:, :1024]          # row stride 1040 elements
    oq, osc = oracle.quantize_rowwise_i8(np.ascontiguousarray(full[:, :1024]))
    q, qbuf, n = guarded((96, 1024), torch.int8, 77)
    s, sbuf, ns = guarded((96,), torch.float32, -5.0)
    sq.sq_quantize_rowwise_i8(xd, q=q, scales=s)
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), osc)
    assert guard_intact(qbuf, n, 77) and guard_intact(sbuf, ns, -5.0)


def test_rowwise_i8_bulk_path_strided_rows_and_guard():
    full = synth.normal(23, (800, 4096 + 64), dtype=synth.BF16)
    xd = to_dev(full, bf16=True)[:, :4096]          # rows 8 KB, row stride 8320 B
    oq, osc = oracle.quantize_rowwise_i8(np.ascontiguousarray(full[:, :4096]), oracle.BF16)
    q, qbuf, n = guarded((800, 4096), torch.int8, 55)
    s, sbuf, ns = guarded((800,), torch.float32, -3.0)
    sq.sq_quantize_rowwise_i8(xd, q=q, scales=s)
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), osc)
    assert guard_intact(qbuf, n, 55) and guard_intact(sbuf, ns, -3.0)


def test_rowwise_i8_degenerate_rows_and_ties():
    x = synth.normal(22, (6, 64))
    x[0] = 0.0                              # all-zero row -> floor scale, zeros
    x[1] = 1e-12                            # below the 1e-8 floor
    x[2] = (np.arange(64) - 32) / 2.0       # many exact ties after scaling
    x[2, 0] = 127.0
    x[3] = -x[3]
    x[4] = np.float32(3.0e38) * np.sign(x[4])   # huge but finite
    x = x.astype(np.float32)
    oq, osc = oracle.quantize_rowwise_i8(x)
    q, s = sq.sq_quantize_rowwise_i8(to_dev(x))
    assert np.array_equal(s.cpu().numpy(), osc) and np.array_equal(q.cpu().numpy(), oq)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_rowwise_i8_degenerate_rows_in_streamed_rows(dt):
    """The same special rows scattered through a tall matrix of 4-8 KB rows,
    the shape rows are streamed through shared memory at."""
    rows, cols = 2333, 1024 if dt == "f32" else 4096
    x = synth.normal(24, (rows, cols), dtype=synth.BF16 if dt == "bf16" else synth.F32)
    xf = synth.bf16_bits_to_f32(x) if dt == "bf16" else x
    pick = np.random.default_rng(5).choice(rows, 60, replace=False)
    for n, r in enumerate(pick):
        kind = n % 5
        if kind == 0:
            xf[r] = 0.0
        elif kind == 1:
            xf[r] = 1e-12
        elif kind == 2:
            xf[r] = (np.arange(cols) % 64 - 32) / 2.0
            xf[r, 0] = 127.0
        elif kind == 3:
            xf[r] *= np.float32(1e30)          # scales above 2^40
        else:
            xf[r] = np.float32(3.0e38) * np.sign(xf[r])
    if dt == "bf16":
        x = (xf.view(np.uint32) >> 16).astype(np.uint16)   # truncated to bf16; both sides see it
        oq, osc = oracle.quantize_rowwise_i8(x, oracle.BF16)
        q, s = sq.sq_quantize_rowwise_i8(to_dev(x, True))
    else:
        x = xf.astype(np.float32)
        oq, osc = oracle.quantize_rowwise_i8(x)
        q, s = sq.sq_quantize_rowwise_i8(to_dev(x))
    assert np.array_equal(s.cpu().numpy(), osc) and np.array_equal(q.cpu().numpy(), oq)


def test_rowwise_i8_empty():
    q, s = sq.sq_quantize_rowwise_i8(torch.empty((0, 64), device=DEV))
    assert q.shape == (0, 64) and s.shape == (0,)


# ------------------------------------------------------------------ FP8
def delayed_scale(seed, shape, std, fmt):
    prev = synth.bf16_bits_to_f32(synth.normal(seed + 1, shape, std=std, dtype=synth.BF16))
    fmax = 448.0 if fmt == sq.SQ_FMT_E4M3 else 57344.0
    return np.float32(np.abs(prev).max()) / np.float32(fmax)


FP8_CASES = [
    ("X 2048x1024 N(0,1)", (2048, 1024), 1.0),
    ("W 1024x1024 N(0,0.02)", (1024, 1024), 0.02),
    ("G 2048x4096 N(0,1e-3)", (2048, 4096), 1e-3),
    ("tail 1000003", (1000003,), 1.0),
    # 65537 chunks of 1024 (every warp of a full grid takes 17-18) and a
    # 112-element tail
    ("full grid and tail 67110000", (67110000,), 1.0),
    ("tail 33", (33,), 1.0),
    ("one", (1,), 1.0),
]


@pytest.mark.parametrize("fmt", [sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("name,shape,std", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_fp8_quantize_parity(name, shape, std, fmt):
    seed = zlib.crc32(name.encode()) % 1000 + 100
    x = synth.normal(seed, shape, std=std, dtype=synth.BF16)
    scale = delayed_scale(seed, shape, std, fmt)
    ox8, oamax = oracle.quantize_fp8(x, scale, fmt)
    ws = sq.new_workspace(DEV)
    x8, amax = sq.sq_quantize_fp8(to_dev(x, bf16=True),
                                  torch.tensor([scale], dtype=torch.float32, device=DEV), fmt, ws)
    assert np.array_equal(x8.cpu().numpy(), ox8)
    assert amax.item() == float(oamax)
    assert int(ws.sum().item()) == 0        # the last block reset the workspace


MULTI = [
    ("X 2048x1024 and W 1024x1024", [((2048, 1024), 1.0), ((1024, 1024), 0.02)]),
    ("G, W, X of the MLP backward", [((2048, 4096), 1e-3), ((4096, 1024), 0.02), ((2048, 1024), 1.0)]),
    ("four ragged, one empty", [((1000003,), 1.0), ((0,), 1.0), ((33,), 1.0), ((3, 5127), 2.0)]),
    ("8192x8192 (full grid) and a 129-element tail", [((8192, 8192), 1.0), ((129,), 1.0)]),
]


@pytest.mark.parametrize("fmt", [sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("name,specs", MULTI, ids=[c[0] for c in MULTI])
def test_fp8_multi_quantize_equals_one_call_per_tensor(name, specs, fmt):
    """sq_quantize_fp8_multi: every tensor's codes and amax equal the
    oracle's, whatever tensor its chunks follow in the launch, ragged tails
    and empty tensors included, and the shared workspace ends zeroed."""
    seed = zlib.crc32(name.encode()) % 1000 + 100
    xs = [synth.normal(seed + 3 * i, shape, std=std, dtype=synth.BF16)
          for i, (shape, std) in enumerate(specs)]
    steps = [delayed_scale(seed + 3 * i, shape, std, fmt) if np.prod(shape) else np.float32(1.0)
             for i, (shape, std) in enumerate(specs)]
    ws = sq.new_workspace(DEV)
    x8s, amaxs = sq.sq_quantize_fp8_multi(
        [to_dev(x, bf16=True) for x in xs],
        [torch.tensor([s], dtype=torch.float32, device=DEV) for s in steps], fmt, ws)
    for x, s, x8, amax in zip(xs, steps, x8s, amaxs):
        ox8, oamax = oracle.quantize_fp8(x, s, fmt)
        assert np.array_equal(x8.cpu().numpy(), ox8)
        assert amax.item() == float(oamax)
    assert int(ws.sum().item()) == 0


def test_fp8_saturation_and_repeated_calls():
    x = synth.student_t(31, (4096, 512), dtype=synth.BF16)
    ws = sq.new_workspace(DEV)
    xd = to_dev(x, bf16=True)
    for fmt, scale in ((sq.SQ_FMT_E4M3, 1e-3), (sq.SQ_FMT_E5M2, 1e-6), (sq.SQ_FMT_E4M3, 0.5)):
        ox8, oamax = oracle.quantize_fp8(x, scale, fmt)
        x8, amax = sq.sq_quantize_fp8(xd, torch.tensor([scale], dtype=torch.float32, device=DEV),
                                      fmt, ws)
        assert np.array_equal(x8.cpu().numpy(), ox8)
        assert amax.item() == float(oamax)
    # a smaller tensor right after: amax must not leak from the previous call
    y = synth.normal(32, (777,), std=1e-3, dtype=synth.BF16)
    oy8, oyamax = oracle.quantize_fp8(y, 1e-5, 0)
    y8, yamax = sq.sq_quantize_fp8(to_dev(y, bf16=True),
                                   torch.tensor([1e-5], dtype=torch.float32, device=DEV), 0, ws)
    assert np.array_equal(y8.cpu().numpy(), oy8) and yamax.item() == float(oyamax)


def test_fp8_empty_and_zero():
    ws = sq.new_workspace(DEV)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    _, amax = sq.sq_quantize_fp8(torch.empty(0, dtype=torch.bfloat16, device=DEV), one, 0, ws)
    assert amax.item() == 0.0
    z = torch.zeros(4096, dtype=torch.bfloat16, device=DEV)
    z8, amax = sq.sq_quantize_fp8(z, one, 0, ws)
    assert amax.item() == 0.0 and int(z8.sum().item()) == 0


# ------------------------------------------------------------------ division edge cases
def test_rowwise_i8_near_ties_at_general_scales():
    """Elements placed within a few ulps of (n + 1/2) * s for every n, at
    scales that are not powers of two: the integer code depends on the last
    bit of the float32 quotient, so the GPU's quotient must equal IEEE
    division's exactly."""
    rng = np.random.default_rng(17)
    rows = []
    for amax in rng.uniform(0.3, 50.0, size=24).astype(np.float32):
        s = np.float32(amax) / np.float32(127.0)
        mids = ((np.arange(-126, 126) + 0.5) * np.float64(s)).astype(np.float32)
        cand = [mids]
        up, dn = mids.copy(), mids.copy()
        for _ in range(3):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            cand += [up, dn]
        row = np.concatenate(cand)[:1759]
        rows.append(np.concatenate([row, np.array([amax], dtype=np.float32)]))
    x = np.stack(rows).astype(np.float32)
    assert np.all(np.abs(x).max(axis=1) == np.abs(x[:, -1]))
    oq, osc = oracle.quantize_rowwise_i8(x)
    q, s = sq.sq_quantize_rowwise_i8(to_dev(x))
    assert np.array_equal(s.cpu().numpy(), osc)
    assert np.array_equal(q.cpu().numpy(), oq)


@pytest.mark.parametrize("scale", [2.0 ** -40, 2.0 ** 40, 2.0 ** -41, 2.0 ** 41, 3.3e-7, 7e11],
                         ids=["lo_edge", "hi_edge", "below", "above", "small", "large"])
def test_fp8_scales_across_the_division_paths(scale):
    rng = np.random.default_rng(18)
    # magnitudes spread so that x/scale sweeps the FP8 range for this scale
    t = np.exp(rng.uniform(np.log(1e-6), np.log(1e6), 20000)) * rng.choice([-1, 1], 20000)
    xf = (t * scale).astype(np.float32)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)       # truncate to bf16 bits
    x[:64] = 0x8000                                          # negative zeros
    x[64:128] = 0x0000
    ws = sq.new_workspace(DEV)
    for fmt in (sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2):
        ox8, oamax = oracle.quantize_fp8(x, scale, fmt)
        x8, amax = sq.sq_quantize_fp8(to_dev(x, bf16=True),
                                      torch.tensor([scale], dtype=torch.float32, device=DEV), fmt, ws)
        assert np.array_equal(x8.cpu().numpy(), ox8)
        assert amax.item() == float(oamax)
        assert np.all(ox8[:64] == 0x80)


SPECIAL_BF16 = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x0080, 0x8080, 0x7F7F, 0xFF7F,
                         0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x3F80, 0xBF80], dtype=np.uint16)


@pytest.mark.parametrize("scale", [2.0 ** -40, 1e-12, 1.0, 2.0 ** 40, 1e13],
                         ids=["2^-40", "1e-12", "1", "2^40", "1e13"])
def test_fp8_special_values(scale):
    """Zeros of both signs, bf16 subnormals, the largest bf16, infinities and
    NaNs, in the streamed chunks and in the ragged tail, with step sizes at
    and beyond both ends of the reciprocal range (products that overflow
    float32 must still saturate).  A NaN input must give a NaN code; the sign
    of that code is not fixed by the format, so only NaN-ness is compared
    there, and every other code bit for bit."""
    n = 3 * 8192 + 77
    x = synth.normal(19, (n,), std=3.0, dtype=synth.BF16)
    rng = np.random.default_rng(19)
    for pos in np.concatenate([rng.choice(3 * 8192, 200, replace=False), np.arange(3 * 8192, n)]):
        x[pos] = SPECIAL_BF16[pos % len(SPECIAL_BF16)]
    ws = sq.new_workspace(DEV)
    for fmt in (sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2):
        ox8, oamax = oracle.quantize_fp8(x, np.float32(scale), fmt)
        x8, amax = sq.sq_quantize_fp8(to_dev(x, bf16=True),
                                      torch.tensor([scale], dtype=torch.float32, device=DEV), fmt, ws)
        got = x8.cpu().numpy()
        nan_in = (x & 0x7FFF) > 0x7F80
        assert nan_in.sum() > 20
        assert np.array_equal(got[~nan_in], ox8[~nan_in])
        assert all(oracle.fp8_code_is_nan(int(c), fmt) for c in got[nan_in])
        assert amax.item() == float(oamax) == np.inf


# ------------------------------------------------------------------ delayed-scaling ring
@pytest.mark.parametrize("fmt", [sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2], ids=["e4m3", "e5m2"])
def test_fp8_ring_sequence_matches_the_oracle(fmt):
    """Twelve quantize steps through one ring (history 5, rolling index,
    margins 0 and 1): codes, amax and the whole ring bit-exact every step."""
    H = 5
    ring_o = np.zeros(H + 2, dtype=np.float32)
    ring_o[H] = 0.05
    ring_d = sq.new_ring(H, 0.05, DEV)
    ws = sq.new_workspace(DEV)
    rng = np.random.default_rng(40 + fmt)
    for step in range(12):
        std = float(np.exp(rng.uniform(np.log(1e-3), np.log(10.0))))
        n = int(rng.integers(1, 300_000))
        x = synth.normal(900 + step, (n,), std=std, dtype=synth.BF16)
        margin = step % 2
        ox8, oamax = oracle.quantize_fp8_ring(x, fmt, ring_o, idx=step % H, margin=margin)
        x8, amax = sq.sq_quantize_fp8_ring(to_dev(x, bf16=True), fmt, ring_d, step % H, margin, ws)
        assert np.array_equal(x8.cpu().numpy(), ox8), step
        assert amax.item() == float(oamax)
        got = ring_d.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ring_o.view(np.uint32)), (step, got, ring_o)
    assert int(ws.sum().item()) == 0


def test_fp8_ring_zero_history_keeps_the_step():
    ring = sq.new_ring(4, 0.25, DEV)
    ws = sq.new_workspace(DEV)
    z = torch.zeros(10_000, dtype=torch.bfloat16, device=DEV)
    x8, amax = sq.sq_quantize_fp8_ring(z, sq.SQ_FMT_E4M3, ring, 2, 0, ws)
    r = ring.cpu().numpy()
    assert amax.item() == 0.0 and r[4] == np.float32(0.25) and np.all(r[:4] == 0) and r[5] == 0


# ------------------------------------------------------------------ row groups / per tensor
GROUP_CASES = [
    ("per tensor f32 128x1024", (128, 1024), "f32", 128),
    ("per tensor bf16 t3 2048x2048", (2048, 2048), "bf16", 10**9),
    ("groups of 8, ragged last, f32 100x256", (100, 256), "f32", 8),
    ("groups of 3 bf16 64x4096", (64, 4096), "bf16", 3),
    ("scalar path groups of 4 f32 37x17", (37, 17), "f32", 4),
    ("per tensor, one row", (1, 512), "f32", 1),
]


@pytest.mark.parametrize("name,shape,dt,g", GROUP_CASES, ids=[c[0] for c in GROUP_CASES])
def test_grouped_i8_parity(name, shape, dt, g):
    seed = zlib.crc32(name.encode()) % 1000 + 300
    x = draw(seed, shape, dt, "t3" if "t3" in name else "normal")
    rows = shape[0]
    oq, osc = oracle.quantize_grouped_i8(x, min(g, rows), oracle.F32 if dt == "f32" else oracle.BF16)
    q, s = sq.sq_quantize_grouped_i8(to_dev(x, bf16=(dt == "bf16")), g)
    assert np.array_equal(s.cpu().numpy(), osc)
    assert np.array_equal(q.cpu().numpy(), oq)
