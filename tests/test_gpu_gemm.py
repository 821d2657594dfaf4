"""GPU parity of the tcgen05 GEMMs against the oracle.

INT8: int32 accumulators and the fp32 dequantized output bit-exact.
FP8:  bf16 output within 1e-2*|ref| + 1e-3*sqrt(K)*sa*sb*max|a8|*max|b8| of
the fp64 reference, in the NT, NN and TN layouts, E4M3 and E5M2.
Shapes cover several tiles, ragged M/N tails and the pages' workloads.
"""
import zlib

import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, bf16_to_f64, guard_intact, guarded, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def seed_of(name):
    return zlib.crc32(name.encode()) % 10000


# ------------------------------------------------------------------ INT8
def run_i8(qa, sa, qb, sb):
    batch = qa.shape[0] if qa.ndim == 3 else 1
    M, K = qa.shape[-2:]
    N = qb.shape[-2]
    ws = torch.empty(sq.gemm_i8_workspace_bytes(batch, M, N, K), dtype=torch.uint8, device=DEV)
    C, acc = sq.sq_gemm_i8_rowscaled(to_dev(qa), to_dev(sa), to_dev(qb), to_dev(sb), ws,
                                     acc_out=True)
    return C.cpu().numpy(), acc.cpu().numpy()


I8_CASES = [
    ("cfg1 128x512x1024 f32 N(0,1)", (128, 1024), (512, 1024)),
    ("ragged 200x300x160", (200, 160), (300, 160)),
    ("single tile 1x1x16", (1, 16), (1, 16)),
    ("K 3072 (3 chunks) 256x384", (256, 3072), (384, 3072)),
    ("K 1040 (chunk + tail) 130x129", (130, 1040), (129, 1040)),
]


@pytest.mark.parametrize("name,sa_shape,sb_shape", I8_CASES, ids=[c[0] for c in I8_CASES])
def test_i8_gemm_parity(name, sa_shape, sb_shape):
    s = seed_of(name)
    a, b = synth.normal(s, sa_shape), synth.normal(s + 1, sb_shape)
    qa, sa = oracle.quantize_rowwise_i8(a)
    qb, sb = oracle.quantize_rowwise_i8(b)
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb)
    C, acc = run_i8(qa, sa, qb, sb)
    assert np.array_equal(acc, oacc)
    assert np.array_equal(C.view(np.uint32), oC.view(np.uint32))


def test_i8_gemm_per_head_batched():
    """16 heads of (196x64) . (196x64)^T, per-row scales within each head."""
    q = synth.normal(41, (16, 196, 64))
    k = synth.normal(42, (16, 196, 64))
    qq, sq_ = oracle.quantize_rowwise_i8(q)
    qk, sk = oracle.quantize_rowwise_i8(k)
    oacc, oC = oracle.gemm_i8(qq, qk, sq_, sk)
    C, acc = run_i8(qq, sq_, qk, sk)
    assert acc.shape == (16, 196, 196)
    assert np.array_equal(acc, oacc) and np.array_equal(C, oC)


def test_i8_gemm_extreme_codes_stay_exact():
    """All codes +-127 with K = 8192: every chunk sum sits at 127^2*1024 and
    the total at 1.3e8 > 2^24, so any inexact accumulation shows."""
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 8192
    qa = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    qa[:8] = 127
    qb = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    qb[:8] = 127
    qb[8:16] = -127
    sa = np.abs(synth.normal(6, (M,))) + np.float32(1e-3)
    sb = np.abs(synth.normal(7, (N,))) + np.float32(1e-3)
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb)
    C, acc = run_i8(qa, sa, qb, sb)
    assert acc[0, 0] == 127 * 127 * K and acc[0, 8] == -127 * 127 * K
    assert np.array_equal(acc, oacc) and np.array_equal(C, oC)


def test_i8_gemm_random_codes_and_acc_only():
    rng = np.random.default_rng(6)
    qa = rng.integers(-127, 128, (300, 2048)).astype(np.int8)
    qb = rng.integers(-127, 128, (260, 2048)).astype(np.int8)
    oacc, _ = oracle.gemm_i8(qa, qb)
    ws = torch.empty(sq.gemm_i8_workspace_bytes(1, 300, 260, 2048), dtype=torch.uint8, device=DEV)
    ones_a = torch.ones(300, device=DEV)
    ones_b = torch.ones(260, device=DEV)
    acc, abuf, n = guarded((300, 260), torch.int32, -7)
    C, acc = sq.sq_gemm_i8_rowscaled(to_dev(qa), ones_a, to_dev(qb), ones_b, ws, want_c=False,
                                     acc_out=acc)
    assert C is None
    assert np.array_equal(acc.cpu().numpy(), oacc)
    assert guard_intact(abuf, n, -7)


# ------------------------------------------------------------------ INT8 in two phases
TWO_PHASE = [
    ("cfg1 128x512x1024 (plain staging)", 0, (128, 1024), (512, 1024)),
    ("per head 16x196x196x64 (plain staging)", 16, (196, 64), (196, 64)),
    ("2048x1024x1024 (bulk staging, bounds)", 0, (2048, 1024), (1024, 1024)),
]


@pytest.mark.parametrize("name,nb,sa_shape,sb_shape", TWO_PHASE, ids=[c[0] for c in TWO_PHASE])
def test_i8_gemm_stage_then_staged_equals_one_call(name, nb, sa_shape, sb_shape):
    """sq_gemm_i8_stage + sq_gemm_i8_rowscaled_staged give the bits of the
    one-call form and of the oracle; a workspace staged once serves a second
    GEMM with other scales."""
    s = seed_of(name)
    shape_a = (nb,) + sa_shape if nb else sa_shape
    shape_b = (nb,) + sb_shape if nb else sb_shape
    a, b = synth.normal(s, shape_a), synth.normal(s + 1, shape_b)
    qa, sa = oracle.quantize_rowwise_i8(a)
    qb, sb = oracle.quantize_rowwise_i8(b)
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb)
    M, K = sa_shape
    N = sb_shape[0]
    ws = torch.empty(sq.gemm_i8_workspace_bytes(max(nb, 1), M, N, K), dtype=torch.uint8,
                     device=DEV)
    tqa, tqb = to_dev(qa), to_dev(qb)
    sq.sq_gemm_i8_stage(tqa, tqb, ws)
    C, acc = sq.sq_gemm_i8_rowscaled_staged(to_dev(sa.reshape(-1)), to_dev(sb.reshape(-1)),
                                            (nb, M, N, K), ws, acc_out=True)
    assert np.array_equal(acc.cpu().numpy(), oacc)
    assert np.array_equal(C.cpu().numpy(), oC)
    # the same staged operands with doubled scales: exact powers of two, so
    # every output doubles exactly
    C2, _ = sq.sq_gemm_i8_rowscaled_staged(to_dev(2 * sa.reshape(-1)), to_dev(sb.reshape(-1)),
                                           (nb, M, N, K), ws)
    assert np.array_equal(C2.cpu().numpy(), 2 * oC)
    C1, acc1 = sq.sq_gemm_i8_rowscaled(tqa, to_dev(sa.reshape(-1)), tqb, to_dev(sb.reshape(-1)),
                                       ws, acc_out=True)
    assert torch.equal(C1, C) and torch.equal(acc1, acc)


# ------------------------------------------------------------------ INT8 quantized and staged in one pass
def _bf16_signs(seed, shape):
    """bf16 bits of +-1.0 with seeded signs: every code quantizes to +-127."""
    sgn = np.random.default_rng(seed).integers(0, 2, shape)
    return np.where(sgn == 1, 0xBF80, 0x3F80).astype(np.uint16)


FUSED = [
    # (name, batch, A shape, B shape, input kind)
    ("cfg1 f32 128x512x1024 (rows in registers)", 0, (128, 1024), (512, 1024), "f32"),
    ("per head 16x196x196x64 (rows in registers)", 16, (196, 64), (196, 64), "f32"),
    ("bf16 512x384x2048 (row pipeline, row-norm bounds)", 0, (512, 2048), (384, 2048), "bf16"),
    ("bf16 ragged 333x350x4096 (row pipeline)", 0, (333, 4096), (350, 4096), "bf16"),
    ("f32 320x400x1024 (row pipeline)", 0, (320, 1024), (400, 1024), "f32"),
    ("bf16 +-1 codes 320x336x2048 (bounds demand the drains)", 0, (320, 2048), (336, 2048), "signs"),
    ("f32 long rows 40x48x20000 (quantize, then staging)", 0, (40, 20000), (48, 20000), "f32"),
]


@pytest.mark.parametrize("name,nb,sa_shape,sb_shape,kind", FUSED, ids=[c[0] for c in FUSED])
def test_i8_quantize_staged_then_gemm(name, nb, sa_shape, sb_shape, kind):
    """sq_quantize_rowwise_i8_staged on A and B, then the staged GEMM: codes,
    scales, int32 accumulators and fp32 outputs equal the oracle's bit for
    bit, whichever kernel the shape takes (rows in registers, the row
    pipeline with row-norm bounds, or quantize then staging).  With every
    code +-127 the row norms exceed the exactness bound, so the GEMM must
    drain its fp32 sums every 1024 K; a wrong decision loses exactness."""
    s = seed_of(name)
    shape_a = (nb,) + sa_shape if nb else sa_shape
    shape_b = (nb,) + sb_shape if nb else sb_shape
    if kind == "f32":
        a, b = synth.normal(s, shape_a), synth.normal(s + 1, shape_b)
        dt, A, B = oracle.F32, to_dev(a), to_dev(b)
    elif kind == "bf16":
        a = synth.normal(s, shape_a, dtype=synth.BF16)
        b = synth.normal(s + 1, shape_b, dtype=synth.BF16)
        dt, A, B = oracle.BF16, to_dev(a, bf16=True), to_dev(b, bf16=True)
    else:
        a, b = _bf16_signs(s, shape_a), _bf16_signs(s + 1, shape_b)
        dt, A, B = oracle.BF16, to_dev(a, bf16=True), to_dev(b, bf16=True)
    oqa, osa = oracle.quantize_rowwise_i8(a, dt)
    oqb, osb = oracle.quantize_rowwise_i8(b, dt)
    if kind == "signs":
        assert np.all(np.abs(oqa) == 127) and np.all(np.abs(oqb) == 127)
    oacc, oC = oracle.gemm_i8(oqa, oqb, osa, osb)
    M, K = sa_shape
    N = sb_shape[0]
    ws = torch.empty(sq.gemm_i8_workspace_bytes(max(nb, 1), M, N, K), dtype=torch.uint8,
                     device=DEV)
    shape = (nb, M, N, K)
    qa, sa = sq.sq_quantize_rowwise_i8_staged(A, 0, shape, ws)
    qb, sb = sq.sq_quantize_rowwise_i8_staged(B, 1, shape, ws)
    assert np.array_equal(qa.cpu().numpy(), oqa) and np.array_equal(sa.cpu().numpy(), osa)
    assert np.array_equal(qb.cpu().numpy(), oqb) and np.array_equal(sb.cpu().numpy(), osb)
    C, acc = sq.sq_gemm_i8_rowscaled_staged(sa.reshape(-1), sb.reshape(-1), shape, ws,
                                            acc_out=True)
    assert np.array_equal(acc.cpu().numpy(), oacc)
    assert np.array_equal(C.cpu().numpy(), oC)
    # C alone: the same bits
    C_only, none = sq.sq_gemm_i8_rowscaled_staged(sa.reshape(-1), sb.reshape(-1), shape, ws)
    assert none is None and torch.equal(C_only, C)
    # both operands in one call (one launch where both fit the register-
    # resident kernel) into a fresh workspace: the same codes, scales and C
    ws2 = torch.empty_like(ws)
    qa2, sa2, qb2, sb2 = sq.sq_quantize_rowwise_i8_staged_pair(A, B, shape, ws2)
    assert torch.equal(qa2, qa) and torch.equal(sa2, sa)
    assert torch.equal(qb2, qb) and torch.equal(sb2, sb)
    C2, acc2 = sq.sq_gemm_i8_rowscaled_staged(sa2.reshape(-1), sb2.reshape(-1), shape, ws2,
                                              acc_out=True)
    assert torch.equal(C2, C) and torch.equal(acc2, acc)


C_ONLY = [
    # (name, batch, M, N, K, scale groups of A and B or None for per row)
    ("cfg1 128x512x1024", 0, 128, 512, 1024, None),
    ("ragged 200x300x160", 0, 200, 300, 160, None),
    ("per head 16x196x196x64", 16, 196, 196, 64, None),
    ("ragged heads 3x130x132x256", 3, 130, 132, 256, None),
    ("one round of 64 tiles 1024x1024x512", 0, 1024, 1024, 512, None),
    ("groups 8 x 30 ragged 200x300x160", 0, 200, 300, 160, (8, 30)),
]


@pytest.mark.parametrize("name,nb,M,N,K,groups", C_ONLY, ids=[c[0] for c in C_ONLY])
def test_i8_gemm_c_only_into_a_guarded_buffer(name, nb, M, N, K, groups):
    """Only the fp32 C asked for, so no int32 accumulator is formed where one
    K chunk holds the whole sum.  C matches the oracle bit for bit, including
    the sign of zero where a row of zero codes meets a row of negative ones
    (float(0) is +0), and nothing past it is written."""
    s = seed_of(name)
    shp_a, shp_b = ((nb, M, K), (nb, N, K)) if nb else ((M, K), (N, K))
    a, b = synth.normal(s, shp_a), synth.student_t(s + 1, shp_b, df=3)
    if groups:
        qa, sa = oracle.quantize_grouped_i8(a, groups[0])
        qb, sb = oracle.quantize_grouped_i8(b, groups[1])
    else:
        qa, sa = oracle.quantize_rowwise_i8(a)
        qb, sb = oracle.quantize_rowwise_i8(b)
    qa[..., :2, :] = 0
    qb[..., :1, :] = -np.maximum(np.abs(qb[..., :1, :]), 1)
    if groups:
        _, oC = oracle.gemm_i8_grouped(qa, qb, sa, sb, groups[0], groups[1])
    else:
        _, oC = oracle.gemm_i8(qa, qb, sa, sb)
    assert np.all(oC.view(np.uint32)[..., :2, :1] == 0)
    ws = torch.empty(sq.gemm_i8_workspace_bytes(max(nb, 1), M, N, K), dtype=torch.uint8,
                     device=DEV)
    C, cbuf, n = guarded(oC.shape, torch.float32, -3.0)
    if groups:
        C2, acc = sq.sq_gemm_i8_grouped(to_dev(qa), to_dev(sa), groups[0], to_dev(qb), to_dev(sb),
                                        groups[1], ws, C=C)
    else:
        C2, acc = sq.sq_gemm_i8_rowscaled(to_dev(qa), to_dev(sa), to_dev(qb), to_dev(sb), ws, C=C)
    assert acc is None and C2.data_ptr() == C.data_ptr()
    assert np.array_equal(C.cpu().numpy().view(np.uint32), oC.view(np.uint32))
    assert guard_intact(cbuf, n, -3.0)


# ------------------------------------------------------------------ FP8
@pytest.mark.parametrize("c", [42, 47], ids=["bound holds: one K chunk", "bound fails: drained"])
def test_i8_exactness_with_and_without_drains(c):
    """Constant codes c at K = 8192 (staged by the bulk pipeline).  With c = 42
    the staging bound proves every partial sum below 2^24, so K runs as one
    fp32 chunk; with c = 47 the sums reach 8192 * 47^2 > 2^24 with odd steps,
    which only the per-1024-K drains keep exact.  Both must be bit-exact."""
    M, N, K = 256, 320, 8192
    qa = np.full((M, K), c, dtype=np.int8)
    qb = np.full((N, K), c, dtype=np.int8)
    qa[::3] = -c                                   # signs vary by row
    sa = np.linspace(0.5, 2.0, M).astype(np.float32)
    sb = np.linspace(0.25, 1.0, N).astype(np.float32)
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb)
    assert np.abs(oacc).max() == K * c * c
    C, acc = run_i8(qa, sa, qb, sb)
    assert np.array_equal(acc, oacc)
    assert np.array_equal(C.view(np.uint32), oC.view(np.uint32))


@pytest.mark.parametrize("cmax", [127, 11], ids=["+-127: 128 drained chunks", "|q|<=11: one chunk"])
def test_i8_gemm_at_the_maximum_k(cmax):
    """K = 2^17, the largest the call accepts.  With codes up to 127 the
    sums reach ~2^31 and every 1024-long chunk is drained; with |q| <= 11
    the staging bound lets the whole K run as one fp32 chunk.  Bit-exact."""
    M, N, K = 64, 96, 1 << 17
    rng = np.random.default_rng(97 + cmax)
    qa = rng.integers(-cmax, cmax + 1, (M, K)).astype(np.int8)
    qb = rng.integers(-cmax, cmax + 1, (N, K)).astype(np.int8)
    if cmax == 127:
        qa[0] = 127
        qb[0] = 127                               # one output at exactly 127^2 * 2^17
    sa = rng.uniform(0.5, 1.5, M).astype(np.float32)
    sb = rng.uniform(0.5, 1.5, N).astype(np.float32)
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb)
    C, acc = run_i8(qa, sa, qb, sb)
    assert np.array_equal(acc, oacc)
    assert np.array_equal(C.view(np.uint32), oC.view(np.uint32))


def fp8_inputs(name, M, N, K, fmt, std_a=1.0, std_b=0.02):
    s = seed_of(name)
    xa = synth.normal(s, (M, K), std=std_a, dtype=synth.BF16)
    xb = synth.normal(s + 1, (N, K), std=std_b, dtype=synth.BF16)
    fmax = 448.0 if fmt == 0 else 57344.0
    pa = synth.bf16_bits_to_f32(synth.normal(s + 2, (M, K), std=std_a, dtype=synth.BF16))
    pb = synth.bf16_bits_to_f32(synth.normal(s + 3, (N, K), std=std_b, dtype=synth.BF16))
    sa = np.float32(np.abs(pa).max()) / np.float32(fmax)
    sb = np.float32(np.abs(pb).max()) / np.float32(fmax)
    a8, _ = oracle.quantize_fp8(xa, sa, fmt)
    b8, _ = oracle.quantize_fp8(xb, sb, fmt)
    return a8, b8, sa, sb


def check_fp8(out, A8, B8, fmt, layout, K, sa, sb, rows=None):
    ref, obf = oracle.gemm_fp8(A8, B8, fmt, layout, sa, sb, rows=rows)
    tab = oracle.fp8_decode_table(fmt)
    bound = oracle.fp8_gemm_bound(ref, K, sa, sb, np.abs(tab[A8]).max(), np.abs(tab[B8]).max())
    got = bf16_to_f64(out)
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"
    # the bf16 codes agree with the oracle's rounding of the fp32 result almost everywhere
    same = np.mean(out.view(torch.int16).cpu().numpy().astype(np.uint16)[
        rows if rows is not None else slice(None)] == obf)
    assert same > 0.9, same


FP8_SHAPES = [
    ("one tile 128x128x128", 128, 128, 128),
    ("multi 256x384x512", 256, 384, 512),
    ("ragged 200x176x320", 200, 176, 320),
    ("wide 128x1024x256", 128, 1024, 256),
    ("deep 130x144x2048", 130, 144, 2048),
    ("short K 160x96x16", 160, 96, 16),
]


@pytest.mark.parametrize("layout", [sq.SQ_NT, sq.SQ_NN, sq.SQ_TN], ids=["NT", "NN", "TN"])
@pytest.mark.parametrize("name,M,N,K", FP8_SHAPES, ids=[c[0] for c in FP8_SHAPES])
def test_fp8_gemm_layouts(name, M, N, K, layout):
    fmt = sq.SQ_FMT_E4M3
    if layout == sq.SQ_TN and M % 16:
        M += 16 - M % 16
    a8, b8, sa, sb = fp8_inputs(name, M, N, K, fmt)
    if layout == sq.SQ_NT:
        A, B = a8, b8
    elif layout == sq.SQ_NN:
        A, B = a8, np.ascontiguousarray(b8.T)
    else:
        A, B = np.ascontiguousarray(a8.T), np.ascontiguousarray(b8.T)
    C, cbuf, n = guarded((M, N), torch.bfloat16, 3.0)
    sq.sq_gemm_fp8_scaled(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), fmt, layout, C=C)
    check_fp8(C, A, B, fmt, layout, K, sa, sb)
    assert guard_intact(cbuf, n, 3.0)


def test_fp8_gemm_long_k():
    """K = 65536 in one fp32 accumulation, within the bound, which grows with
    sqrt(K)."""
    M, N, K = 128, 160, 1 << 16
    fmt = sq.SQ_FMT_E4M3
    a8, b8, sa, sb = fp8_inputs("long K", M, N, K, fmt)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.sq_gemm_fp8_scaled(to_dev(a8), to_dev(b8), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), fmt, sq.SQ_NT, C=C)
    check_fp8(C, a8, b8, fmt, sq.SQ_NT, K, sa, sb)


@pytest.mark.parametrize("N", [100, 104, 2056], ids=["N100 thread stores", "N104 clipped box", "N2056 pair"])
def test_fp8_gemm_nt_output_widths(N):
    """Output rows that are not a multiple of 8 bf16 are stored by the threads;
    multiples of 8 leave through 32x32 TMA boxes whose last column box is
    clipped.  The guard band after C must stay untouched either way."""
    M, K = 2304 if N > 1000 else 136, 256   # 2304 x 2056: 81 tile pairs, the CTA-pair kernel
    fmt = sq.SQ_FMT_E4M3
    a8, b8, sa, sb = fp8_inputs(f"width {N}", M, N, K, fmt)
    C, cbuf, n = guarded((M, N), torch.bfloat16, -2.0)
    sq.sq_gemm_fp8_scaled(to_dev(a8), to_dev(b8), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), fmt, sq.SQ_NT, C=C)
    check_fp8(C, a8, b8, fmt, sq.SQ_NT, K, sa, sb)
    assert guard_intact(cbuf, n, -2.0)


@pytest.mark.parametrize("layout", [sq.SQ_NT, sq.SQ_NN, sq.SQ_TN], ids=["NT", "NN", "TN"])
def test_fp8_gemm_e5m2(layout):
    M, N, K = 256, 256, 1024
    fmt = sq.SQ_FMT_E5M2
    a8, b8, sa, sb = fp8_inputs("e5m2", M, N, K, fmt)
    A = a8 if layout != sq.SQ_TN else np.ascontiguousarray(a8.T)
    B = b8 if layout == sq.SQ_NT else np.ascontiguousarray(b8.T)
    C = sq.sq_gemm_fp8_scaled(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                              torch.tensor([sb], device=DEV), fmt, layout)
    check_fp8(C, A, B, fmt, layout, K, sa, sb)


def test_fp8_forward_nt_2048x1024x1024():
    """X bf16 2048x1024 N(0,1), W bf16 1024x1024 N(0,0.02), delayed scales."""
    M, N, K = 2048, 1024, 1024
    a8, b8, sa, sb = fp8_inputs("fwd", M, N, K, 0)
    C = sq.sq_gemm_fp8_scaled(to_dev(a8), to_dev(b8), torch.tensor([sa], device=DEV),
                              torch.tensor([sb], device=DEV), 0, sq.SQ_NT)
    rows = np.sort(np.random.default_rng(1).choice(M, 256, replace=False))
    check_fp8(C, a8, b8, 0, sq.SQ_NT, K, sa, sb, rows=rows)


def test_fp8_backward_dx_nn_and_dw_tn():
    """MLP backward, dim 1024, hidden 4096, 2048 tokens, all E4M3:
    dX = G W (NN) with G 2048x4096, W 4096x1024; dW = G^T X (TN)."""
    T, H, D = 2048, 4096, 1024
    fmt = 0
    g = synth.normal(51, (T, H), std=1e-3, dtype=synth.BF16)
    w = synth.normal(52, (H, D), std=0.02, dtype=synth.BF16)
    x = synth.normal(53, (T, D), std=1.0, dtype=synth.BF16)

    def scale_of(seed, shape, std):
        p = synth.bf16_bits_to_f32(synth.normal(seed, shape, std=std, dtype=synth.BF16))
        return np.float32(np.abs(p).max()) / np.float32(448.0)

    sg, sw, sx = scale_of(61, (T, H), 1e-3), scale_of(62, (H, D), 0.02), scale_of(63, (T, D), 1.0)
    g8, _ = oracle.quantize_fp8(g, sg, fmt)
    w8, _ = oracle.quantize_fp8(w, sw, fmt)
    x8, _ = oracle.quantize_fp8(x, sx, fmt)
    tsg, tsw, tsx = (torch.tensor([v], device=DEV) for v in (sg, sw, sx))
    dX = sq.sq_gemm_fp8_scaled(to_dev(g8), to_dev(w8), tsg, tsw, fmt, sq.SQ_NN)
    rows = np.sort(np.random.default_rng(2).choice(T, 128, replace=False))
    check_fp8(dX, g8, w8, fmt, sq.SQ_NN, H, sg, sw, rows=rows)
    dW = sq.sq_gemm_fp8_scaled(to_dev(g8), to_dev(x8), tsg, tsx, fmt, sq.SQ_TN)
    assert dW.shape == (H, D)
    rows = np.sort(np.random.default_rng(3).choice(H, 128, replace=False))
    check_fp8(dW, g8, x8, fmt, sq.SQ_TN, T, sg, sx, rows=rows)


# ------------------------------------------------------------------ two GEMMs in one call
def fp8_operands(name, M, N, K, layout, fmt):
    """FP8 codes of A (M x K) and B (N x K) stored as `layout` wants them."""
    a8, b8, sa, sb = fp8_inputs(name, M, N, K, fmt)
    A = a8 if layout != sq.SQ_TN else np.ascontiguousarray(a8.T)
    B = b8 if layout == sq.SQ_NT else np.ascontiguousarray(b8.T)
    return A, B, sa, sb


def check_rows(C, A, B, fmt, layout, K, sa, sb, seed, n=64):
    M = C.shape[0]
    edges = np.concatenate([np.arange(0, M, 128), np.minimum(np.arange(127, M + 127, 128), M - 1)])
    rows = np.unique(np.concatenate([edges, np.random.default_rng(seed).choice(M, min(n, M),
                                                                               replace=False)]))
    check_fp8(C, A, B, fmt, layout, K, sa, sb, rows=rows)


# (problem 0, problem 1) as (M, N, K, layout); all small enough that one
# launch takes both, on 128- or 256-wide tiles as the estimate picks
FP8_PAIRS = [
    ("ragged NT + TN", (200, 176, 320, sq.SQ_NT), (272, 96, 512, sq.SQ_TN)),
    ("deep NN + short NT", (130, 144, 2048, sq.SQ_NN), (160, 96, 16, sq.SQ_NT)),
    ("one tile + wide", (128, 128, 128, sq.SQ_TN), (128, 1024, 256, sq.SQ_NN)),
    ("dX NN + dW TN ragged", (1016, 1008, 2048, sq.SQ_NN), (2032, 1008, 1024, sq.SQ_TN)),
    # 320 tiles of 128x128 on the 152 SMs: three rounds, the second dealt backwards
    ("three rounds NT + NN", (2048, 2048, 256, sq.SQ_NT), (1024, 1024, 128, sq.SQ_NN)),
]


@pytest.mark.parametrize("fmt", [sq.SQ_FMT_E4M3, sq.SQ_FMT_E5M2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("name,p0,p1", FP8_PAIRS, ids=[c[0] for c in FP8_PAIRS])
def test_fp8_gemm_pair(name, p0, p1, fmt):
    """Each problem of the pair matches the oracle as one GEMM does, and
    neither output's guard band is touched."""
    ops, outs = [], []
    for i, (M, N, K, layout) in enumerate((p0, p1)):
        A, B, sa, sb = fp8_operands(f"{name} {i}", M, N, K, layout, fmt)
        C, cbuf, n = guarded((M, N), torch.bfloat16, 3.0 + i)
        ops.append((A, B, sa, sb, layout, K))
        outs.append((C, cbuf, n))
    sq.sq_gemm_fp8_scaled_pair([to_dev(o[0]) for o in ops], [to_dev(o[1]) for o in ops],
                               [torch.tensor([o[2]], device=DEV) for o in ops],
                               [torch.tensor([o[3]], device=DEV) for o in ops], fmt,
                               [o[4] for o in ops], Cs=[o[0] for o in outs])
    assert sq.sq_get_last_device_error() == sq.SQ_OK
    for i, ((A, B, sa, sb, layout, K), (C, cbuf, n)) in enumerate(zip(ops, outs)):
        check_fp8(C, A, B, fmt, layout, K, sa, sb)
        assert guard_intact(cbuf, n, 3.0 + i)


def test_fp8_gemm_pair_backward_shapes_match_two_calls():
    """dX = G W (NN) and dW = G^T X (TN) of the MLP backward (dim 1024,
    hidden 4096, 2048 tokens) in one call: within the bound on sampled rows
    (every 128-row band's edges), and equal to two separate calls wherever
    both take the same tile width."""
    T, H, D = 2048, 4096, 1024
    fmt = sq.SQ_FMT_E4M3
    g = synth.normal(71, (T, H), std=1e-3, dtype=synth.BF16)
    w = synth.normal(72, (H, D), std=0.02, dtype=synth.BF16)
    x = synth.normal(73, (T, D), std=1.0, dtype=synth.BF16)

    def scale_of(seed, shape, std):
        p = synth.bf16_bits_to_f32(synth.normal(seed, shape, std=std, dtype=synth.BF16))
        return np.float32(np.abs(p).max()) / np.float32(448.0)

    sg, sw, sx = scale_of(74, (T, H), 1e-3), scale_of(75, (H, D), 0.02), scale_of(76, (T, D), 1.0)
    g8, _ = oracle.quantize_fp8(g, sg, fmt)
    w8, _ = oracle.quantize_fp8(w, sw, fmt)
    x8, _ = oracle.quantize_fp8(x, sx, fmt)
    tsg, tsw, tsx = (torch.tensor([v], device=DEV) for v in (sg, sw, sx))
    G8, W8, X8 = to_dev(g8), to_dev(w8), to_dev(x8)
    dX, dW = sq.sq_gemm_fp8_scaled_pair([G8, G8], [W8, X8], [tsg, tsg], [tsw, tsx], fmt,
                                        [sq.SQ_NN, sq.SQ_TN])
    assert dX.shape == (T, D) and dW.shape == (H, D)
    check_rows(dX, g8, w8, fmt, sq.SQ_NN, H, sg, sw, seed=77)
    check_rows(dW, g8, x8, fmt, sq.SQ_TN, T, sg, sx, seed=78)
    # the same products by the single-GEMM entry point: every element is one
    # tile's fp32 sum over the same K order, so the codes agree except where a
    # different tile width changes the tensor core's grouping of K
    dX1 = sq.sq_gemm_fp8_scaled(G8, W8, tsg, tsw, fmt, sq.SQ_NN)
    dW1 = sq.sq_gemm_fp8_scaled(G8, X8, tsg, tsx, fmt, sq.SQ_TN)
    for a, b in ((dX, dX1), (dW, dW1)):
        same = (a.view(torch.int16) == b.view(torch.int16)).float().mean().item()
        assert same > 0.99, same


def test_fp8_gemm_pair_in_a_cuda_graph():
    """The paired call captured in a CUDA graph on a side stream: its replays
    give the bits of the eager call."""
    fmt = sq.SQ_FMT_E4M3
    shapes = [(1016, 1008, 2048, sq.SQ_NN), (2032, 1008, 1024, sq.SQ_TN)]
    ops = [fp8_operands(f"graph pair {i}", *s_[:3], s_[3], fmt) for i, s_ in enumerate(shapes)]
    As, Bs = [to_dev(o[0]) for o in ops], [to_dev(o[1]) for o in ops]
    sas = [torch.tensor([o[2]], device=DEV) for o in ops]
    sbs = [torch.tensor([o[3]], device=DEV) for o in ops]
    layouts = [s_[3] for s_ in shapes]
    eager = sq.sq_gemm_fp8_scaled_pair(As, Bs, sas, sbs, fmt, layouts)
    Cs = [torch.full_like(c, 7.0) for c in eager]
    side = torch.cuda.Stream(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        sq.sq_gemm_fp8_scaled_pair(As, Bs, sas, sbs, fmt, layouts, Cs=Cs)
    for _ in range(2):
        for c in Cs:
            c.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(Cs, eager):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def test_fp8_gemm_pair_of_large_problems_runs_as_two_launches():
    """Problems with many rounds of tiles each are estimated faster as two
    ordinary launches; the results are the same GEMMs."""
    fmt = sq.SQ_FMT_E4M3
    shapes = [(4096, 8192, 1024, sq.SQ_NT), (4096, 8192, 1024, sq.SQ_NN)]
    ops = [fp8_operands(f"large pair {i}", *s[:3], s[3], fmt) for i, s in enumerate(shapes)]
    Cs = sq.sq_gemm_fp8_scaled_pair([to_dev(o[0]) for o in ops], [to_dev(o[1]) for o in ops],
                                    [torch.tensor([o[2]], device=DEV) for o in ops],
                                    [torch.tensor([o[3]], device=DEV) for o in ops], fmt,
                                    [s[3] for s in shapes])
    for i, (C, (A, B, sa, sb), s) in enumerate(zip(Cs, ops, shapes)):
        check_rows(C, A, B, fmt, s[3], s[2], sa, sb, seed=80 + i, n=32)
        single = sq.sq_gemm_fp8_scaled(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                                       torch.tensor([sb], device=DEV), fmt, s[3])
        assert torch.equal(C.view(torch.int16), single.view(torch.int16))


# ------------------------------------------------------------------ the pages' one-wave shapes
# The forward (NT 2048x1024x1024) and dX (NN) run on 128x128 tiles, dW (TN)
# on 128x256 tiles: one round of tiles each.  The ragged variants clip M, N
# and K against those tiles.
ONE_WAVE = [
    ("fwd NT 2048x1024x1024 e5m2", 2048, 1024, 1024, sq.SQ_NT, sq.SQ_FMT_E5M2),
    ("fwd NT ragged 2040x1000x1040", 2040, 1000, 1040, sq.SQ_NT, sq.SQ_FMT_E4M3),
    ("fwd NT ragged 1800x936x1024", 1800, 936, 1024, sq.SQ_NT, sq.SQ_FMT_E4M3),
    ("dX NN ragged 2040x1008x4096", 2040, 1008, 4096, sq.SQ_NN, sq.SQ_FMT_E4M3),
    ("dW TN ragged 4080x1008x2048", 4080, 1008, 2048, sq.SQ_TN, sq.SQ_FMT_E4M3),
    ("dW TN 4096x1024x2048 e5m2", 4096, 1024, 2048, sq.SQ_TN, sq.SQ_FMT_E5M2),
]


@pytest.mark.parametrize("name,M,N,K,layout,fmt", ONE_WAVE, ids=[c[0] for c in ONE_WAVE])
def test_fp8_gemm_one_wave_shapes(name, M, N, K, layout, fmt):
    a8, b8, sa, sb = fp8_inputs(name, M, N, K, fmt)
    A = a8 if layout != sq.SQ_TN else np.ascontiguousarray(a8.T)
    B = b8 if layout == sq.SQ_NT else np.ascontiguousarray(b8.T)
    C, cbuf, n = guarded((M, N), torch.bfloat16, 3.0)
    sq.sq_gemm_fp8_scaled(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), fmt, layout, C=C)
    # every tile row band of both CTAs of a pair: the first and last rows of
    # each 128-row block, plus seeded rows
    edges = np.concatenate([np.arange(0, M, 128), np.minimum(np.arange(127, M + 127, 128), M - 1)])
    rows = np.unique(np.concatenate([edges, np.random.default_rng(seed_of(name)).choice(M, 64,
                                                                                        replace=False)]))
    check_fp8(C, A, B, fmt, layout, K, sa, sb, rows=rows)
    assert guard_intact(cbuf, n, 3.0)


# ------------------------------------------------------------------ CTA-pair shapes
# Problems with several rounds of 256x256 tiles over the SM pairs and a long
# enough K run on the 2-SM (cta_group::2) kernel; these sizes select it and
# keep ragged tails in M and N (the last column of pair tiles is half empty).
PAIR_FP8 = [
    ("pair NT 4000x3968x4096", 4000, 3968, 4096, sq.SQ_NT),
    ("pair NN 4000x3968x4096", 4000, 3968, 4096, sq.SQ_NN),
    ("pair TN 4000x3968x4096", 4000, 3968, 4096, sq.SQ_TN),
]


@pytest.mark.parametrize("name,M,N,K,layout", PAIR_FP8, ids=[c[0] for c in PAIR_FP8])
def test_fp8_gemm_cta_pair(name, M, N, K, layout):
    a8, b8, sa, sb = fp8_inputs(name, M, N, K, sq.SQ_FMT_E4M3)
    A = a8 if layout != sq.SQ_TN else np.ascontiguousarray(a8.T)
    B = b8 if layout == sq.SQ_NT else np.ascontiguousarray(b8.T)
    C, cbuf, n = guarded((M, N), torch.bfloat16, 5.0)
    sq.sq_gemm_fp8_scaled(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), sq.SQ_FMT_E4M3, layout, C=C)
    rows = np.sort(np.concatenate([np.arange(0, 8), np.arange(M - 8, M),
                                   np.random.default_rng(4).choice(M, 240, replace=False)]))
    rows = np.unique(rows)
    check_fp8(C, A, B, sq.SQ_FMT_E4M3, layout, K, sa, sb, rows=rows)
    assert guard_intact(cbuf, n, 5.0)


def test_i8_gemm_cta_pair_ragged():
    s = seed_of("pair i8")
    a, b = synth.normal(s, (2200, 1040)), synth.normal(s + 1, (2300, 1040))
    qa, sa = oracle.quantize_rowwise_i8(a)
    qb, sb = oracle.quantize_rowwise_i8(b)
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(2196, 2200),
                                     np.random.default_rng(5).choice(2200, 120, replace=False)]))
    oacc, oC = oracle.gemm_i8(qa, qb, sa, sb, rows=rows)
    C, acc = run_i8(qa, sa, qb, sb)
    assert np.array_equal(acc[rows], oacc) and np.array_equal(C[rows], oC)


def test_i8_gemm_cta_pair_batched_heads():
    q = synth.normal(61, (24, 500, 64))
    k = synth.normal(62, (24, 520, 64))
    qq, sq_ = oracle.quantize_rowwise_i8(q)
    qk, sk = oracle.quantize_rowwise_i8(k)
    oacc, oC = oracle.gemm_i8(qq, qk, sq_, sk)
    C, acc = run_i8(qq, sq_, qk, sk)
    assert np.array_equal(acc, oacc) and np.array_equal(C, oC)


def test_i8_gemm_batched_staged_in_bulk():
    """Three heads of 600 x 2048 . (700 x 2048)^T: large enough that the codes
    are staged by the bulk pipeline (which also bounds their sums), with
    ragged 600- and 700-row heads; bit-exact against the oracle."""
    q = synth.student_t(63, (3, 600, 2048))
    k = synth.normal(64, (3, 700, 2048))
    qq, sq_ = oracle.quantize_rowwise_i8(q)
    qk, sk = oracle.quantize_rowwise_i8(k)
    oacc, oC = oracle.gemm_i8(qq, qk, sq_, sk)
    C, acc = run_i8(qq, sq_, qk, sk)
    assert np.array_equal(acc, oacc) and np.array_equal(C, oC)


# ------------------------------------------------------------------ E4M3 output
E4M3_OUT = [
    ("out8 NT 200x176x320", 200, 176, 320, sq.SQ_NT, sq.SQ_FMT_E4M3),
    ("out8 NN 256x384x512", 256, 384, 512, sq.SQ_NN, sq.SQ_FMT_E4M3),
    ("out8 TN 208x160x256", 208, 160, 256, sq.SQ_TN, sq.SQ_FMT_E5M2),
    ("out8 pair NT 4000x3968x4096", 4000, 3968, 4096, sq.SQ_NT, sq.SQ_FMT_E4M3),
    ("out8 one round NT 2040x1000x1024", 2040, 1000, 1024, sq.SQ_NT, sq.SQ_FMT_E4M3),
    ("out8 one round of 128x256 tiles NT 2048x2048x512", 2048, 2048, 512, sq.SQ_NT, sq.SQ_FMT_E4M3),
]


@pytest.mark.parametrize("name,M,N,K,layout,fmt", E4M3_OUT, ids=[c[0] for c in E4M3_OUT])
def test_fp8_gemm_e4m3_output(name, M, N, K, layout, fmt):
    """E4M3 codes of (acc*sa*sb)/out_scale: each code lies between the E4M3
    values bracketing the fp64 reference widened by the GEMM bound, and the
    output step is chosen so that some outputs saturate."""
    a8, b8, sa, sb = fp8_inputs(name, M, N, K, fmt)
    A = a8 if layout != sq.SQ_TN else np.ascontiguousarray(a8.T)
    B = b8 if layout == sq.SQ_NT else np.ascontiguousarray(b8.T)
    rows = None if M * N < 1_000_000 else np.unique(np.concatenate(
        [np.arange(4), np.arange(M - 4, M), np.random.default_rng(9).choice(M, 120, replace=False)]))
    ref, _ = oracle.gemm_fp8(A, B, fmt, layout, sa, sb, rows=rows, want_bf16=False)
    out_scale = np.float32(np.abs(ref).max() / 448.0 * 0.8)   # ~2% of outputs saturate
    t_ref, ocodes = oracle.gemm_fp8_e4m3(A, B, fmt, layout, sa, sb, out_scale, rows=rows)
    C, cbuf, n = guarded((M, N), torch.uint8, 0xA5)
    sq.sq_gemm_fp8_scaled_e4m3(to_dev(A), to_dev(B), torch.tensor([sa], device=DEV),
                               torch.tensor([sb], device=DEV), fmt, layout,
                               torch.tensor([out_scale], device=DEV), C=C)
    got = C.cpu().numpy()
    if rows is not None:
        got = got[rows]
    tab = oracle.fp8_decode_table(fmt)
    bound = oracle.fp8_gemm_bound(ref, K, sa, sb, np.abs(tab[A]).max(), np.abs(tab[B]).max())
    assert np.all(oracle.e4m3_acceptable(got, t_ref, bound / float(out_scale)))
    assert np.mean(got == ocodes) > 0.95
    assert np.any(np.abs(oracle.fp8_decode_table(0)[got]) == 448.0)
    assert guard_intact(cbuf, n, 0xA5)


# ------------------------------------------------------------------ row-group scales
GROUPED_GEMM = [
    ("per tensor both 128x512x1024", (128, 1024), (512, 1024), 128, 512),
    ("groups 8 x 30 ragged 200x300x160", (200, 160), (300, 160), 8, 30),
    ("pair per tensor A, per row B 2200x2300x256", (2200, 256), (2300, 256), 2200, 1),
]


@pytest.mark.parametrize("name,sa_shape,sb_shape,ga,gb", GROUPED_GEMM, ids=[c[0] for c in GROUPED_GEMM])
def test_i8_gemm_grouped_scales(name, sa_shape, sb_shape, ga, gb):
    s = seed_of(name)
    a, b = synth.normal(s, sa_shape), synth.normal(s + 1, sb_shape)
    qa, sa = oracle.quantize_grouped_i8(a, ga)
    qb, sb = oracle.quantize_grouped_i8(b, gb)
    M = sa_shape[0]
    rows = None if M < 1000 else np.unique(np.concatenate(
        [np.arange(4), np.arange(M - 4, M), np.random.default_rng(3).choice(M, 100, replace=False)]))
    oacc, oC = oracle.gemm_i8_grouped(qa, qb, sa, sb, ga, gb, rows=rows)
    ws = torch.empty(sq.gemm_i8_workspace_bytes(1, M, sb_shape[0], sa_shape[1]), dtype=torch.uint8,
                     device=DEV)
    C, acc = sq.sq_gemm_i8_grouped(to_dev(qa), to_dev(sa), ga, to_dev(qb), to_dev(sb), gb, ws,
                                   acc_out=True)
    C, acc = C.cpu().numpy(), acc.cpu().numpy()
    if rows is not None:
        C, acc = C[rows], acc[rows]
    assert np.array_equal(acc, oacc) and np.array_equal(C, oC)


def test_i8_gemm_grouped_batched_per_tensor_heads():
    """Per-head batched product with one scale per head (per_tensor within each
    head): group sizes equal to the head's row count."""
    q = synth.normal(81, (16, 196, 64))
    k = synth.normal(82, (16, 196, 64))
    qq, sqs = zip(*[oracle.quantize_grouped_i8(np.ascontiguousarray(q[h]), 196) for h in range(16)])
    qk, sks = zip(*[oracle.quantize_grouped_i8(np.ascontiguousarray(k[h]), 196) for h in range(16)])
    qq, qk = np.stack(qq), np.stack(qk)
    sqa, ska = np.concatenate(sqs), np.concatenate(sks)
    oacc, oC = oracle.gemm_i8_grouped(qq, qk, sqa, ska, 196, 196)
    ws = torch.empty(sq.gemm_i8_workspace_bytes(16, 196, 196, 64), dtype=torch.uint8, device=DEV)
    C, acc = sq.sq_gemm_i8_grouped(to_dev(qq), to_dev(sqa), 196, to_dev(qk), to_dev(ska), 196, ws,
                                   acc_out=True)
    assert np.array_equal(acc.cpu().numpy(), oacc) and np.array_equal(C.cpu().numpy(), oC)


# ------------------------------------------------------------------ clock records
def test_gemm_clock_probe_records_each_cta():
    """With record buffers set, a GEMM launch writes per CTA its start and end
    SM cycles and nanoseconds: the implied clocks are plausible, one record
    per CTA, and clearing the buffers stops the records."""
    rec8 = torch.zeros(256 * 4, dtype=torch.int64, device=DEV)
    rec_i8 = torch.zeros(256 * 4, dtype=torch.int64, device=DEV)
    sq.sq_set_clock_probe(rec8, rec_i8)
    try:
        a8, b8, sa, sb = fp8_inputs("clock probe", 1024, 1024, 2048, 0)
        C = sq.sq_gemm_fp8_scaled(to_dev(a8), to_dev(b8), torch.tensor([sa], device=DEV),
                                  torch.tensor([sb], device=DEV), 0, sq.SQ_NT)
        qa = torch.randint(-127, 128, (512, 1024), dtype=torch.int8, device=DEV)
        qb = torch.randint(-127, 128, (640, 1024), dtype=torch.int8, device=DEV)
        ws = torch.empty(sq.gemm_i8_workspace_bytes(1, 512, 640, 1024), dtype=torch.uint8,
                         device=DEV)
        sq.sq_gemm_i8_rowscaled(qa, torch.ones(512, device=DEV), qb, torch.ones(640, device=DEV),
                                ws)
        torch.cuda.synchronize()
    finally:
        sq.sq_set_clock_probe()
    # 8x8 tiles of 128 x 128; 4x20 tiles of 128 x 32
    for rec, ctas in ((rec8, 64), (rec_i8, 80)):
        r = rec.view(-1, 4)
        used = r[r[:, 3] > 0]
        assert used.shape[0] == ctas
        assert bool(torch.all(used[:, 1] > used[:, 0])) and bool(torch.all(used[:, 3] > used[:, 2]))
        mhz = sq.clock_probe_mhz(rec)
        assert 300.0 < mhz["min"] <= mhz["max"] < 3000.0, mhz
    check_fp8(C, a8, b8, 0, sq.SQ_NT, 2048, sa, sb)
    rec8.zero_()
    sq.sq_gemm_fp8_scaled(to_dev(a8), to_dev(b8), torch.tensor([sa], device=DEV),
                          torch.tensor([sb], device=DEV), 0, sq.SQ_NT)
    torch.cuda.synchronize()
    assert int(rec8.count_nonzero().item()) == 0
