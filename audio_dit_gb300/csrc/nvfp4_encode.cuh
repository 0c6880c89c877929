// NVFP4 block encoding shared by the activation quantiser and the GEMM's
// NVFP4-output epilogue, so that both produce the same bytes for the same
// bf16 values and global scale s:
//   S    = e4m3_rn_sat( RN( RN(bmax / 6) / s ) )      block scale code
//   eff  = RN(e4m3(S) * s),  r = (eff == 0) ? 0 : min(RN(1 / eff), FLT_MAX)
//   q_i  = e2m1_rn_sat( RN(m_i * r) ), sign kept, two codes per byte
// ("H3 Blackwell Runtime Plan", "Next Performance Plan: Blackwell NVFP4
// GEMMs": signed zero and tie-to-even FP4 rounding; the E4M3 block scale
// under an fp32 tensor scale amax / (6 * 448)).
#pragma once
#include <cfloat>
#include <cstdint>

#include "ptx_sm103.cuh"

namespace h3fp4 {

// Eight fp32 values -> eight E2M1 codes in one word, value 2i in bits 8i..8i+3
// and value 2i+1 in bits 8i+4..8i+7 (RN, saturating to +-6, sign kept).
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// E4M3 code (sign clear) -> fp32 through the hardware E4M3 -> f16 conversion
// (every E4M3 value is exact in f16, and f16 -> f32 is exact).
__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    float f;
    asm("{\n\t.reg .b16 c, lo, hi;\n\t.reg .b32 h2;\n\t"
        "cvt.u16.u32 c, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, c;\n\t"
        "mov.b32 {lo, hi}, h2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t}"
        : "=f"(f)
        : "r"(code));
    return f;
}

// RN(b / 6) for b >= 0 a bf16 value (a block maximum), without a division:
// q = RN(b * RN(1/6)), the remainder b - 6q is exact in one fma, and one more
// fma applies the correction step of Markstein's FMA-based division.  Equal to
// the IEEE quotient for every non-negative bf16 value, subnormal quotients
// included (checked exhaustively).
__device__ __forceinline__ float div6_bf16(float b)
{
    const float c = __uint_as_float(0x3E2AAAABu);  // RN(1/6)
    const float q = __fmul_rn(b, c);
    const float r = __fmaf_rn(-q, 6.0f, b);
    return __fmaf_rn(r, c, q);
}

// RN(1 / RN(e4m3(S) * s)) for block-scale code S (0 for a zero scale).
__device__ __forceinline__ float block_rcp(uint32_t S, float s)
{
    const float eff = __fmul_rn(e4m3_value(S), s);
    return (eff == 0.0f || S == 0x7Fu) ? 0.0f : fminf(__frcp_rn(eff), FLT_MAX);
}

// Block-scale code of a block whose largest magnitude is bmax (a bf16 value).
__device__ __forceinline__ uint32_t block_scale_code(float bmax, float s)
{
    return cvt_e4m3(__fdiv_rn(div6_bf16(bmax), s));
}

}  // namespace h3fp4
