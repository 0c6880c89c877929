"""Arithmetic identities the CUDA quantiser relies on, checked exhaustively on
the CPU over the inputs the kernel can see.

The block scale is S = e4m3(RN(RN(bmax / 6) / s_g)) (the encode order of the
"H3 Runtime Current State" quantiser, "Owned Performance Kernels").  bmax is the
maximum magnitude of bf16 values, hence itself a non-negative bf16 value, and
the kernel forms RN(bmax / 6) without a division: q = RN(bmax * RN(1/6)),
r = bmax - 6 q (exact in one fma), RN(q + r * RN(1/6)) (the correction step of
Markstein's FMA division).  These tests prove that this equals the IEEE quotient
for every non-negative finite bf16 value, and that the plain multiply alone
would not."""
import numpy as np


def _all_nonneg_bf16():
    return (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)


def _fma_div6(b):
    c = np.float32(1.0) / np.float32(6.0)
    assert c.view(np.uint32) == 0x3E2AAAAB
    q = (b * c).astype(np.float32)
    # q has 24 significant bits and |b - 6q| is tiny: both steps are exact in
    # float64, and the final conversion is the single fp32 rounding of the fma.
    r = b.astype(np.float64) - 6.0 * q.astype(np.float64)
    assert np.all((r.astype(np.float32).astype(np.float64)) == r), "remainder must be exact in fp32"
    return (q.astype(np.float64) + r * np.float64(c)).astype(np.float32)


def test_fma_corrected_div6_equals_ieee_division_on_every_bf16():
    b = _all_nonneg_bf16()
    ref = b / np.float32(6.0)
    got = _fma_div6(b)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_plain_reciprocal_multiply_is_not_enough():
    b = _all_nonneg_bf16()
    ref = b / np.float32(6.0)
    mul = b * (np.float32(1.0) / np.float32(6.0))
    assert np.count_nonzero(mul != ref) > 0
