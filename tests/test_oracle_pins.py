"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Every check here compares the oracle with something other than its own code:
the format value tables (tests/golden), exhaustive transition points derived
from the round-to-nearest-even rule, library routines (torch's float8/bf16
casts, numpy's float64 matmul), exact rational arithmetic, closed forms and
brute force on tiny inputs.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ E2M1

def test_e2m1_decode_matches_value_table(orc):
    for code, val in _read_table("e2m1_values.txt"):
        got = orc.e2m1_decode(int(code))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_encode_tie_and_saturation_cases(orc):
    for fmt, x, code in _read_table("encode_ties.txt"):
        x32 = float(np.float32(float(x)))
        got = orc.e2m1_encode(x32) if fmt == "e2m1" else orc.e4m3_encode(x32)
        assert got == int(code, 16), (fmt, x, hex(got), code)


def test_encode_decode_roundtrip(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_decode(c)) == c
    for c in range(0x7F):
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c


def _transitions(orc, enc_array, lo_bits, hi_bits, chunk=1 << 24):
    """Scan every fp32 bit pattern in [lo_bits, hi_bits) in increasing order and
    return [(first_bits_of_new_code, new_code)] plus the first code."""
    trans = []
    first = None
    prev = None
    for start in range(lo_bits, hi_bits, chunk):
        stop = min(start + chunk, hi_bits)
        bits = np.arange(start, stop, dtype=np.uint32)
        codes = enc_array(bits.view(np.float32))
        if first is None:
            first = int(codes[0])
        if prev is not None and codes[0] != prev:
            trans.append((start, int(codes[0])))
        d = np.nonzero(codes[1:] != codes[:-1])[0]
        for i in d:
            trans.append((start + int(i) + 1, int(codes[i + 1])))
        prev = codes[-1]
    return first, trans


def _bits(f):
    return int(np.array([f], np.float32).view(np.uint32)[0])


def _expected_transitions(values):
    """From a sorted list of (value, code) on a grid, the fp32 bit pattern where
    round-to-nearest-even first selects each next code: at the exact midpoint if
    the upper code is even, else just above it."""
    out = []
    for (v0, c0), (v1, c1) in zip(values[:-1], values[1:]):
        mid = (Fraction(v0) + Fraction(v1)) / 2
        mid32 = np.float32(float(mid))
        assert Fraction(float(mid32)) == mid  # midpoints are exact fp32 values
        b = _bits(mid32)
        out.append((b if c1 % 2 == 0 else b + 1, c1))
    return out


@pytest.mark.slow
def test_e2m1_encoder_exhaustive_positive(orc):
    """All 2^31 - 2^23 finite non-negative fp32 inputs: the encoder is the
    round-to-nearest-even step function of the E2M1 table (saturating at 6)."""
    first, trans = _transitions(orc, orc.e2m1_encode_array, 0, 0x7F800000)
    table = [(float(v), int(c)) for c, v in _read_table("e2m1_values.txt")[:8]]
    assert first == 0
    assert trans == _expected_transitions(table)


def test_e2m1_sign_copied(orc):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 0x7F800000, size=1 << 20, dtype=np.uint32)
    grid = np.array([0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 1e-45, 3e38], np.float32).view(np.uint32)
    near = (grid[:, None].astype(np.int64) + np.arange(-3, 4)[None, :]).clip(0, 0x7F7FFFFF).astype(np.uint32)
    bits = np.concatenate([bits, near.ravel()])
    pos = orc.e2m1_encode_array(bits.view(np.float32))
    neg = orc.e2m1_encode_array((bits | np.uint32(0x80000000)).view(np.float32))
    assert np.array_equal(neg, pos | 8)
    assert np.all(pos < 8)


# ------------------------------------------------------------------ E4M3

def test_e4m3_decode_points(orc):
    for code, val in _read_table("e4m3_points.txt"):
        got = orc.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_decode_matches_torch_float8(orc):
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert nan.sum() == 2  # 0x7F and 0xFF only
    finite_pos = got[:0x7F]
    assert np.all(np.diff(finite_pos) > 0) and finite_pos.max() == 448.0


@pytest.mark.slow
def test_e4m3_encoder_exhaustive_nonnegative(orc):
    """All finite non-negative fp32 inputs: round-to-nearest-even on the E4M3
    grid, saturating at 448 (0x7E)."""
    first, trans = _transitions(orc, orc.e4m3_encode_array, 0, 0x7F800000)
    table = [(orc.e4m3_decode(c), c) for c in range(0x7F)]
    assert first == 0
    assert trans == _expected_transitions(table)


def test_e4m3_encoder_matches_torch_cast(orc):
    """Inside the finite range torch's fp32 -> float8_e4m3fn cast (RNE) is a
    library implementation of the same rounding."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    lo, hi = 0, _bits(448.0)
    bits = np.concatenate([rng.integers(lo, hi + 1, size=1 << 21, dtype=np.uint32),
                           np.arange(_bits(2.0 ** -10) - 5, _bits(2.0 ** -5), 997, dtype=np.uint32)])
    x = bits.view(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode_array(x)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ bf16 / modulation / global scale

def test_bf16_rounding_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 0x7F7F0000, size=200000, dtype=np.uint32)
    bits[::2] |= np.uint32(0x80000000)
    bits[:64] = (np.arange(64, dtype=np.uint32) << 16) | np.uint32(0x8000)  # exact ties
    x = bits.view(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_float(float(v)) for v in x[:20000]], np.uint16)
    assert np.array_equal(got, ref[:20000])


def _round_f32_exact(q: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32, ties to even (brute force)."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda f: (abs(Fraction(float(f)) - q),
                                     int(np.array([f], np.float32).view(np.uint32)[0]) & 1))
    return np.float32(best)


def test_modulation_single_fma_rounding(orc):
    """m = bf16(fma(x, 1+scale, shift)): the fp32 value is the exactly rounded
    x*(1+scale)+shift (rational arithmetic), then bf16 (torch's cast)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    M, K = 8, 64
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * 3)
    shift = (rng.standard_normal((1, K), dtype=np.float32) * 0.1).astype(np.float32)
    scale = (rng.standard_normal((1, K), dtype=np.float32) * 0.1).astype(np.float32)
    got = orc.modulate(x, shift, scale, [0, M])
    xf = W.bf16_bits_to_f32(x)
    for r in range(M):
        for k in range(K):
            one_plus = _round_f32_exact(1 + Fraction(float(scale[0, k])))
            v = _round_f32_exact(Fraction(float(xf[r, k])) * Fraction(float(one_plus))
                                 + Fraction(float(shift[0, k])))
            want = torch.tensor([float(v)], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert got[r, k] == want, (r, k)


def test_modulation_special_cases(orc):
    rng = np.random.default_rng(4)
    M, K = 6, 32
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    z = np.zeros((1, K), np.float32)
    assert np.array_equal(orc.modulate(x, z, z, [0, M]), x)            # identity
    two = orc.modulate(x, z, np.ones((1, K), np.float32), [0, M])        # x*2 exactly
    assert np.array_equal(W.bf16_bits_to_f32(two), 2 * W.bf16_bits_to_f32(x))
    sh = np.full((1, K), 0.375, np.float32)
    killed = orc.modulate(x, sh, -np.ones((1, K), np.float32), [0, M])  # x*0 + shift
    assert np.all(W.bf16_bits_to_f32(killed) == 0.375)
    # two segments pick their own rows
    sh2 = np.stack([np.zeros(K, np.float32), np.full(K, 0.5, np.float32)])
    sc2 = np.zeros((2, K), np.float32)
    seg = orc.modulate(x, sh2, sc2, [0, 2, M])
    assert np.array_equal(seg[:2], x[:2])
    xf = W.bf16_bits_to_f32(x[2:]).astype(np.float64) + 0.5
    assert np.array_equal(seg[2:], W.to_bf16_bits(xf.astype(np.float32)))


def test_global_scale_closed_forms(orc):
    assert orc.global_scale(2688.0) == 1.0
    assert orc.global_scale(0.0) == 1.0                 # all-zero tensor reading
    assert orc.global_scale(6.0) == float(np.float32(6.0) / np.float32(2688.0))
    x = W.to_bf16_bits(np.array([[0.5, -7.25, 3.0, 0.0] * 4], np.float32))
    assert orc.amax(x) == 7.25


# ------------------------------------------------------------------ block quantiser invariants

def _deq_block(orc, S, q, s_g):
    return np.array([orc.e2m1_decode(int(c)) for c in q]) * orc.e4m3_decode(S) * s_g


def test_block_max_hits_six(orc):
    for Sv, s_g in [(1.0, 1.0), (0.75, 2.0 ** -3), (448.0, 1.0)]:
        m = np.linspace(-1, 1, 16).astype(np.float32) * np.float32(6 * Sv * s_g)
        m[3] = np.float32(6 * Sv * s_g)
        S, q = orc.quantize_block(m, s_g)
        assert orc.e4m3_decode(S) == Sv
        assert q[3] == 7 and q[0] == 15


def test_block_error_within_half_step(orc):
    rng = np.random.default_rng(9)
    for _ in range(300):
        s_g = float(np.float32(rng.uniform(1e-3, 1.0)))
        m = (rng.standard_normal(16) * rng.uniform(0.01, 3)).astype(np.float32)
        S, q = orc.quantize_block(m, s_g)
        eff = float(np.float32(orc.e4m3_decode(S) * s_g))
        deq = np.array([orc.e2m1_decode(int(c)) for c in q]) * eff
        for mi, di in zip(m.astype(np.float64), deq):
            u = abs(mi) / eff
            half = 0.25 if u < 2 else (0.5 if u < 4 else 1.0)
            excess = max(0.0, u - 6.0)  # saturation region
            assert abs(di - mi) <= (half + excess) * eff * (1 + 1e-6) + 1e-30


def test_block_sign_symmetry_and_idempotence(orc):
    rng = np.random.default_rng(10)
    for _ in range(300):
        m = (rng.standard_normal(16) * rng.uniform(0.2, 50)).astype(np.float32)
        m = W.bf16_bits_to_f32(W.to_bf16_bits(m))
        S, q = orc.quantize_block(m, 1.0)
        S2, q2 = orc.quantize_block(-m, 1.0)
        assert S == S2 and np.array_equal(q2, q ^ 8)
        deq = _deq_block(orc, S, q, 1.0).astype(np.float32)  # <= 6 significant bits: exact
        S3, q3 = orc.quantize_block(deq, 1.0)
        assert S3 == S and np.array_equal(q3 & 7, q & 7)


def test_block_special_cases(orc):
    S, q = orc.quantize_block(np.zeros(16, np.float32), 1.0)
    assert S == 0 and np.all(q == 0)
    S, q = orc.quantize_block(-np.zeros(16, np.float32), 0.5)
    assert S == 0 and np.all(q == 8)              # signed zero kept
    m = np.zeros(16, np.float32)
    m[7] = -5.0
    S, q = orc.quantize_block(m, 1.0)
    assert q[7] == 15 and np.all(np.delete(q, 7) == 0)
    # an all-zero tensor: global scale 1, zero scales, zero codes
    codes, sf, gs = orc.quantize(np.zeros((3, 64), np.uint16))
    assert gs == 1.0 and not codes.any() and not sf.any()


# ------------------------------------------------------------------ block-scale layout

@pytest.mark.parametrize("rows,K", [(1, 64), (127, 128), (128, 64), (129, 192), (300, 512), (5, 80)])
def test_sf_layout_is_tiled_reshape(orc, rows, K):
    """The offsets equal a 128x4 tiling built by numpy reshapes: tile rows
    (128 = 4 x 32) and tile columns (4 blocks) with rows-within-32 outermost
    inside a 512-byte tile, tiles in row-tile-major order; the map is a
    bijection onto [0, sf_bytes)."""
    cols = K // 16
    rt, kt = (rows + 127) // 128, (cols + 3) // 4
    ids = np.arange(rt * 128 * kt * 4).reshape(rt * 128, kt * 4)   # id = r*cols_pad + c
    tiled = ids.reshape(rt, 4, 32, kt, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    pos = np.empty_like(tiled)
    pos[tiled] = np.arange(tiled.size)
    assert orc.sf_bytes(rows, K) == tiled.size
    for r in range(rt * 128):
        for c in range(kt * 4):
            assert orc.sf_offset(r, c, K) == pos[r * kt * 4 + c]


def test_sf_roundtrip_and_padding_zero(orc):
    d = W.make_inputs("tiny", M=200)
    codes, sf, gs = orc.quantize(d["x"])
    K = d["K"]
    rows_pad = 256
    used = np.zeros(sf.size, bool)
    for r in range(200):
        for c in range(K // 16):
            used[orc.sf_offset(r, c, K)] = True
    assert not sf[~used].any()       # padding rows are zero bytes
    assert used.sum() == 200 * (K // 16) and sf.size == rows_pad * K // 16


# ------------------------------------------------------------------ GEMM and epilogue

def _py_dequant(orc, codes, sf, gs, rows, K):
    out = np.zeros((rows, K))
    for r in range(rows):
        for k in range(K):
            byte = int(codes[r, k // 2])
            q = byte & 15 if k % 2 == 0 else byte >> 4
            out[r, k] = orc.e2m1_decode(q) * orc.e4m3_decode(int(sf[orc.sf_offset(r, k // 16, K)])) * gs
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 3, 32), (4, 4, 64), (3, 2, 48)])
def test_linear_brute_force_tiny(orc, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = W.to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * 0.05)
    b = W.to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * 0.1)
    g = rng.uniform(0, 1, (1, N)).astype(np.float32)
    R = W.to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    a = orc.quantize(x)
    ww = orc.quantize(w)
    out, bound = orc.linear_full(a, ww, M, N, K, bias=b, gate=g, resid=R)
    da = _py_dequant(orc, a[0], a[1], a[2], M, K)
    dw = _py_dequant(orc, ww[0], ww[1], ww[2], N, K)
    bf, Rf = W.bf16_bits_to_f32(b), W.bf16_bits_to_f32(R)
    for m in range(M):
        for n in range(N):
            acc = sum(da[m, k] * dw[n, k] for k in range(K))
            want = float(Rf[m, n]) + float(g[0, n]) * (acc + float(bf[n]))
            assert abs(out[m, n] - want) <= 1e-12 * (abs(want) + 1)
            sabs = sum(abs(da[m, k] * dw[n, k]) for k in range(K))
            assert abs(bound[m, n] - (abs(out[m, n]) / 256 + 1e-5 * float(g[0, n]) * sabs)) <= 1e-12 * (bound[m, n] + 1e-30)


def test_gemm_matches_library_dgemm(orc):
    rng = np.random.default_rng(21)
    M, N, K = 70, 90, 256
    a = rng.standard_normal((M, K))
    w = rng.standard_normal((N, K))
    c = orc.gemm_f64(a, w)
    ref = a @ w.T
    assert np.max(np.abs(c - ref) / (np.abs(a) @ np.abs(w).T)) < 1e-12
    # the quantised linear without epilogue equals the library dgemm of the
    # exactly dequantised operands
    d = W.make_inputs("tiny", M=40)
    aq = orc.quantize(d["x"])
    wq = orc.quantize(d["w"][:50])
    out, _ = orc.linear_full(aq, wq, 40, 50, d["K"])
    da = orc.dequantize(aq[0], aq[1], aq[2], 40, d["K"])
    dw = orc.dequantize(wq[0], wq[1], wq[2], 50, d["K"])
    ref = da @ dw.T
    assert np.max(np.abs(out - ref) / (np.abs(da) @ np.abs(dw).T + 1e-300)) < 1e-12


def test_epilogue_closed_forms(orc):
    d = W.make_inputs("attn_out", M=64)
    K, N = d["K"], 48
    aq = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    wq = orc.quantize(d["w"][:N])
    R = d["resid"][:, :N].copy()
    y, _ = orc.linear_full(aq, wq, 64, N, K)
    zero_g = np.zeros((2, N), np.float32)
    out0, _ = orc.linear_full(aq, wq, 64, N, K, bias=d["bias"][:N], gate=zero_g, resid=R,
                              seg_off=d["seg_off"])
    assert np.array_equal(out0, W.bf16_bits_to_f32(R).astype(np.float64))   # g = 0 -> R
    one_g = np.ones((2, N), np.float32)
    out1, _ = orc.linear_full(aq, wq, 64, N, K, gate=one_g, resid=np.zeros_like(R),
                              seg_off=d["seg_off"])
    assert np.array_equal(out1, y)                                           # R=0,g=1,b=0 -> y
    # the points API agrees with the full one
    pts = np.array([[0, 0], [63, 47], [40, 3], [d["seg_off"][1], 5]])
    g = d["gate"][:, :N].copy()
    full, fb = orc.linear_full(aq, wq, 64, N, K, bias=d["bias"][:N], gate=g, resid=R, seg_off=d["seg_off"])
    pv, pb = orc.linear_points(aq, wq, 64, N, K, pts, bias=d["bias"][:N], gate=g, resid=R,
                               seg_off=d["seg_off"])
    assert np.array_equal(pv, full[pts[:, 0], pts[:, 1]]) and np.array_equal(pb, fb[pts[:, 0], pts[:, 1]])


def test_quantize_gscale_given_and_segments(orc):
    d = W.make_inputs("attn_out", M=96)
    c1, s1, g1 = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    c2, s2, g2 = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"], gscale=g1)
    assert g2 == g1 and np.array_equal(c1, c2) and np.array_equal(s1, s2)
    # one global amax spans both segments
    m = orc.modulate(d["x"], d["shift"], d["scale"], d["seg_off"])
    assert g1 == orc.global_scale(orc.amax(m))


# ------------------------------------------------------------------ SwiGLU producer

def _bf16_value(bits):
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def _nearest_bf16(v: Fraction) -> int:
    """Correctly rounded bf16 (ties to even) of an exact rational, by comparing
    exact distances to the two bf16 neighbours of its fp32 approximation."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    f32 = np.float32(float(a))
    lo = int(np.array([f32], np.float32).view(np.uint32)[0]) >> 16
    best = None
    for b in (lo - 1, lo, lo + 1, lo + 2):
        if b < 0 or b >= 0x7F80:
            continue
        dist = abs(_bf16_value(b) - a)
        key = (dist, b & 1)          # nearer first; on a tie the even code
        if best is None or key < best[0]:
            best = (key, b)
    return sign | best[1]


def _exact_swiglu(g_bits, u_bits, prec=60):
    """silu(g) * u with 60-digit decimal arithmetic (its own exp), as a Fraction."""
    from decimal import Decimal, localcontext
    g, u = _bf16_value(g_bits), _bf16_value(u_bits)
    with localcontext() as ctx:
        ctx.prec = prec
        gd = Decimal(g.numerator) / Decimal(g.denominator)
        ud = Decimal(u.numerator) / Decimal(u.denominator)
        val = gd / (1 + (-gd).exp()) * ud
    return Fraction(val)


def test_swiglu_matches_high_precision_rounding(orc):
    """bf16(silu(g) * u) against 60-digit decimal arithmetic and an exact
    nearest-bf16 search, over every bf16 g in [-24, 24] with a spread of u."""
    rng = np.random.default_rng(7)
    gs = [b for b in range(0x10000) if (b & 0x7F80) != 0x7F80 and abs(_bf16_value(b)) <= 24]
    gs = [gs[i] for i in rng.choice(len(gs), 3000, replace=False)] + [0x0000, 0x8000, 0x3F80, 0xBF80]
    gs += [0x0001, 0x8001, 0x00B9, 0x8093, 0x2570, 0xA570, 0x3000, 0xB000]   # tiny |g|: near-midpoints
    us = [0x3F80, 0xBF80, 0x4049, 0x3C23, 0xC2F7]
    bad = []
    for i, g in enumerate(gs):
        u = us[i % len(us)] if i % 3 else int(rng.integers(0x3000, 0x4300)) | (0x8000 if i % 2 else 0)
        want = _nearest_bf16(_exact_swiglu(g, u))
        got = orc.swiglu_bf16(g, u)
        if want & 0x7FFF == 0:       # an exact zero keeps the IEEE product sign
            want = (g ^ u) & 0x8000 if (g & 0x7FFF) == 0 else want
        if got != want:
            bad.append((hex(g), hex(u), hex(got), hex(want)))
    assert not bad, bad[:10]


def test_swiglu_closed_forms(orc):
    for u in (0x3F80, 0xBF80, 0x4120):
        h = orc.swiglu_bf16(0x0000, u)                 # silu(0) = 0
        assert h & 0x7FFF == 0
    # g >= 128: e^-g < 2^-184, so h = bf16(g * u), the rounded exact product
    for g in (0x4300, 0x4349, 0x4400):
        for u in (0x3F80, 0x3FC0, 0xC0A0):
            assert orc.swiglu_bf16(g, u) == _nearest_bf16(_bf16_value(g) * _bf16_value(u))
    # g <= -128: |silu(g) * u| < 1e-50, far below the smallest bf16: a signed zero
    assert orc.swiglu_bf16(0xC300, 0x3F80) == 0x8000
    assert orc.swiglu_bf16(0xC300, 0xBF80) == 0x0000


def test_swiglu_rows_pairing(orc):
    """Row layout: in each 256-column group the first 128 columns are gates and
    the next 128 the matching ups; h column 128 t + i pairs y columns
    256 t + i and 256 t + 128 + i."""
    rng = np.random.default_rng(3)
    y = W.to_bf16_bits(rng.standard_normal((5, 512)).astype(np.float32))
    h = orc.swiglu_rows(y)
    assert h.shape == (5, 256)
    for r in range(5):
        for j in range(256):
            t, i = divmod(j, 128)
            assert h[r, j] == orc.swiglu_bf16(int(y[r, 256 * t + i]), int(y[r, 256 * t + 128 + i]))


def _exact_silu_mul(g: float, u: float, prec=60):
    """silu(g) * u for float64 g, u with 60-digit decimal arithmetic (its own exp)."""
    from decimal import Decimal, localcontext
    with localcontext() as ctx:
        ctx.prec = prec
        gd, ud = Decimal(g), Decimal(u)      # exact conversions of the doubles
        return float(gd / (1 + (-gd).exp()) * ud)


def test_silu_mul_f64_matches_high_precision(orc):
    """The unrounded float64 silu(g) * u (the value the end-to-end SwiGLU bound
    is stated around) agrees with 60-digit decimal arithmetic to a few float64
    ulps, across large, moderate, tiny and zero g and both signs of u."""
    rng = np.random.default_rng(17)
    g = np.concatenate([rng.uniform(-40, 40, 2000), rng.standard_normal(500) * 1e-3,
                        np.array([0.0, -0.0, 1e-7, -1e-7, 3e-12, -2.5e-30, 1e-300, 20.0, -20.0, 2.4, -1.28])])
    u = rng.standard_normal(g.size) * np.exp(rng.uniform(-8, 8, g.size))
    got = orc.silu_mul_f64(g, u)
    for gi, ui, h in zip(g, u, got):
        want = _exact_silu_mul(float(gi), float(ui))
        if want == 0.0:
            assert h == 0.0
        else:
            assert abs(h - want) <= 1e-14 * abs(want), (gi, ui, h, want)
