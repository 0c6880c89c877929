// The AdaLN modulation prologue of an activation, shared by the quantiser's
// passes and the GEMM's in-kernel packer so that both produce the same bf16
// values m = bf16(x * (1 + scale[seg]) + shift[seg]) ("H3 Runtime Current
// State", "Owned Performance Kernels": modulation fused into the pack; the
// segment of a row selects its scale/shift vectors).
#pragma once
#include <cstdint>

#include <cuda_bf16.h>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"

namespace h3fp4 {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sixteen bf16 values (one 16-element block of a row) as eight words.
struct V16 {
    uint32_t w[8];
};

__device__ __forceinline__ void unpack16(const V16& v, float (&f)[16])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_lo(v.w[i]);
        f[2 * i + 1] = bf16_hi(v.w[i]);
    }
}

// Segment of row r: the i with off[i] <= r < off[i + 1].
__device__ __forceinline__ int segment_of(const Segments& s, long long r)
{
    int i = 0;
#pragma unroll 1
    while (i + 1 < s.nseg && r >= s.off[i + 1]) ++i;
    return i;
}

// Modulation constants of one 16-column block: (1 + scale, shift) of columns
// 2j, 2j + 1 as fp32 pairs, valid for rows [seg_begin, seg_end).
struct ModCols {
    uint64_t onep[8], sh[8];
    long long seg_begin, seg_end;
};

__device__ __forceinline__ void load_mod(const float* scale, const float* shift, long long K, const Segments& seg,
                                         int s, long long cb, ModCols& mc)
{
    const float4* sc = reinterpret_cast<const float4*>(scale + (long long)s * K + cb * 16);
    const float4* sh = reinterpret_cast<const float4*>(shift + (long long)s * K + cb * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 a = __ldg(sc + i);
        const float4 b = __ldg(sh + i);
        mc.onep[2 * i] = f2(__fadd_rn(1.0f, a.x), __fadd_rn(1.0f, a.y));
        mc.onep[2 * i + 1] = f2(__fadd_rn(1.0f, a.z), __fadd_rn(1.0f, a.w));
        mc.sh[2 * i] = f2(b.x, b.y);
        mc.sh[2 * i + 1] = f2(b.z, b.w);
    }
    mc.seg_begin = seg.off[s];
    mc.seg_end = seg.off[s + 1];
}

__device__ __forceinline__ void init_mod(ModCols& mc)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mc.onep[j] = f2(1.0f, 1.0f);
        mc.sh[j] = f2(0.0f, 0.0f);
    }
    mc.seg_begin = 0;
    mc.seg_end = -1;
}

// m = bf16(fma(x, 1 + scale, shift)) for 16 values: one fp32 fma each, then one
// packed round-to-nearest-even conversion per pair (cvt.rn.bf16x2.f32 rounds
// each half exactly like the scalar conversion, at half the conversion cost).
template <bool kMod>
__device__ __forceinline__ void modulate16(float (&f)[16], const ModCols& mc)
{
    if (kMod) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float a, b;
            unf2(fma2(f2(f[2 * j], f[2 * j + 1]), mc.onep[j], mc.sh[j]), a, b);
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
            f[2 * j] = bf16_lo(u);
            f[2 * j + 1] = bf16_hi(u);
        }
    }
}

}  // namespace h3fp4
