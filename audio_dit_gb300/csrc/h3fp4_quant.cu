// NVFP4 activation / weight quantisation for sm_103a.
//
// Two streaming passes over a bf16 [rows, K] tensor ("H3 Runtime Current
// State", "Owned Performance Kernels": scale discovery, then pack into qdata +
// swizzled block scales; "H3 Blackwell Runtime Plan", "Next Performance Plan":
// signed zero, tie-to-even FP4 rounding, cuBLAS tiled block-scale layout):
//
//   amax pass  m = prologue(x); per-CTA max|m| -> partials[]   (skipped when the
//              global scale is supplied by the caller)
//   pack pass  s = max(partials) / (6*448); per 16-element block: E4M3 scale,
//              E2M1 codes (two per byte), scale byte in the 128x4 tile layout.
//
// Thread mapping: a CTA of 128 threads owns 128 consecutive 8-element column
// vectors (1024 columns) and walks a contiguous range of rows; each thread
// issues one coalesced 16-byte load per row (a warp reads 512 contiguous
// bytes), keeps its column's (1 + scale, shift) in registers, and a pair of
// lanes forms one 16-element block (max by one shuffle).  Eight lanes (four
// blocks) form one 4-byte word of the scale tile.
#include <cfloat>
#include <cstdint>

#include <cuda_bf16.h>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"

namespace h3fp4 {
namespace {

constexpr int kThreads = 128;
constexpr int kRowUnroll = 4;

struct QuantParams {
    const uint16_t* x;
    long long rows, rows_pad, K;
    const float* shift;
    const float* scale;
    Segments seg;
    uint8_t* codes;
    uint8_t* sf;
    float* gscale;
    int gscale_given;
    float* partials;
    int nparts;
    int rows_per_cta;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 (round to nearest even) -> fp32: the exact BF16 modulated value.
__device__ __forceinline__ float round_bf16(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ int segment_of(const Segments& s, long long r)
{
    int i = 0;
#pragma unroll 1
    while (i + 1 < s.nseg && r >= s.off[i + 1]) ++i;
    return i;
}

// Per-thread modulation constants for the 8 columns it owns.
struct ModCols {
    float onep[8], sh[8];
    long long seg_end;
};

__device__ __forceinline__ void load_mod(const QuantParams& p, int seg, int cv, ModCols& mc)
{
    const float* sc = p.scale + (long long)seg * p.K + (long long)cv * 8;
    const float* sh = p.shift + (long long)seg * p.K + (long long)cv * 8;
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(sc));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(sc) + 1);
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(sh));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(sh) + 1);
    const float s8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float h8[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mc.onep[j] = __fadd_rn(1.0f, s8[j]);
        mc.sh[j] = h8[j];
    }
    mc.seg_end = p.seg.off[seg + 1];
}

__device__ __forceinline__ void init_mod(ModCols& mc)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mc.onep[j] = 1.0f;
        mc.sh[j] = 0.0f;
    }
    mc.seg_end = -1;
}

template <bool kMod>
__device__ __forceinline__ void modulate8(float (&f)[8], const ModCols& mc)
{
    if (kMod) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = round_bf16(__fmaf_rn(f[j], mc.onep[j], mc.sh[j]));
    }
}

__device__ __forceinline__ float block_reduce_max(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

// ------------------------------------------------------------------ pass 1: amax

template <bool kMod>
__global__ void __launch_bounds__(kThreads) amax_kernel(QuantParams p)
{
    __shared__ float red[kThreads / 32];
    const int cv = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = cv < p.K / 8;
    const long long r0 = (long long)blockIdx.y * p.rows_per_cta;
    const long long r1 = min(r0 + (long long)p.rows_per_cta, p.rows);
    const uint16_t* xc = p.x + (long long)cv * 8;

    ModCols mc;
    init_mod(mc);
    float mx = 0.0f;
    long long r = r0;
    for (; r < r1; r += kRowUnroll) {
        const int n = (int)min((long long)kRowUnroll, r1 - r);
        uint4 v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u)
            if (valid && u < n) v[u] = ld_stream_v4(xc + (r + u) * p.K);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            if (!(valid && u < n)) continue;
            if (kMod && r + u >= mc.seg_end) load_mod(p, segment_of(p.seg, r + u), cv, mc);
            float f[8];
            unpack8(v[u], f);
            modulate8<kMod>(f, mc);
#pragma unroll
            for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[j]));
        }
    }
    const float m = block_reduce_max(mx, red);
    if (threadIdx.x == 0) p.partials[blockIdx.y * gridDim.x + blockIdx.x] = m;
}

// ------------------------------------------------------------------ pass 2: pack

template <bool kMod>
__global__ void __launch_bounds__(kThreads) pack_kernel(QuantParams p)
{
    __shared__ float red[kThreads / 32];
    // Global scale: one full-activation amax over every partial of pass 1.
    float s_g;
    if (p.gscale_given) {
        s_g = *p.gscale;
    } else {
        float m = 0.0f;
        for (int i = threadIdx.x; i < p.nparts; i += kThreads) m = fmaxf(m, p.partials[i]);
        const float amax = block_reduce_max(m, red);
        s_g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.gscale = s_g;
    }

    const int lane = threadIdx.x & 31;
    const int cv = blockIdx.x * kThreads + threadIdx.x;
    const int K8 = (int)(p.K / 8);
    const bool valid = cv < K8;                 // uniform over each 8-lane group
    const long long kb4 = p.K / 64;             // scale tiles per 128 rows
    const long long r0 = (long long)blockIdx.y * p.rows_per_cta;
    const long long r1 = min(r0 + (long long)p.rows_per_cta, p.rows_pad);
    const uint16_t* xc = p.x + (long long)cv * 8;
    uint32_t* codes_c = reinterpret_cast<uint32_t*>(p.codes) + cv;  // 4 bytes per 8 elements
    const long long g = cv >> 3;                // 64-column group = scale word index

    ModCols mc;
    init_mod(mc);
    for (long long r = r0; r < r1; r += kRowUnroll) {
        uint4 v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (valid && r + u < p.rows) v[u] = ld_stream_v4(xc + (r + u) * p.K);
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            const long long rr = r + u;
            if (rr >= r1) break;                   // uniform over the CTA
            const bool real = rr < p.rows;
            float f[8];
            unpack8(v[u], f);
            if (kMod && real) {
                if (rr >= mc.seg_end && valid) load_mod(p, segment_of(p.seg, rr), cv, mc);
                modulate8<kMod>(f, mc);
            }
            float lmax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) lmax = fmaxf(lmax, fabsf(f[j]));
            const float bmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, 1));
            const uint32_t S = real ? cvt_e4m3(__fdiv_rn(__fdiv_rn(bmax, 6.0f), s_g)) : 0u;
            const float eff = __fmul_rn(e4m3_to_f32(S), s_g);
            const float rcp = (eff == 0.0f) ? 0.0f : fminf(__frcp_rn(eff), FLT_MAX);
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word |= cvt_e2m1x2(__fmul_rn(f[2 * j], rcp), __fmul_rn(f[2 * j + 1], rcp)) << (8 * j);
            if (valid && real) codes_c[rr * (p.K / 8)] = word;
            // gather the four block scales of this 64-column group into lane%8 == 0
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, S, 2);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, S, 4);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, S, 6);
            if (valid && (lane & 7) == 0) {
                const long long off = (((rr >> 7) * kb4 + g) << 9) + ((rr & 31) << 4) + (((rr >> 5) & 3) << 2);
                *reinterpret_cast<uint32_t*>(p.sf + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
            }
        }
    }
}

// One CTA: max over the amax partials of pass 1 -> *out (the tensor amax).
__global__ void __launch_bounds__(kThreads) reduce_partials_kernel(const float* partials, int nparts, float* out)
{
    __shared__ float red[kThreads / 32];
    float m = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += kThreads) m = fmaxf(m, partials[i]);
    const float amax = block_reduce_max(m, red);
    if (threadIdx.x == 0) *out = amax;
}

__global__ void gscale_from_amax_kernel(const float* amax, float* gscale)
{
    const float a = *amax;
    *gscale = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
}

QuantParams make_params(const QuantJob& job, dim3* grid)
{
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(job.x);
    p.rows = job.rows;
    p.rows_pad = (job.rows + 127) / 128 * 128;
    p.K = job.K;
    p.shift = job.shift;
    p.scale = job.scale;
    p.seg = job.seg;
    p.codes = job.codes;
    p.sf = job.sf;
    p.gscale = job.gscale;
    p.gscale_given = job.gscale_given ? 1 : 0;
    p.partials = job.partials;

    const int col_ctas = (int)((job.K / 8 + kThreads - 1) / kThreads);
    const int target = sm_count_current_device() * 8;
    int row_groups = (target + col_ctas - 1) / col_ctas;
    row_groups = max(1, min(row_groups, kMaxPartials / col_ctas));
    // rows per CTA covers the padded rows so the pack pass zeroes scale padding
    p.rows_per_cta = (int)((p.rows_pad + row_groups - 1) / row_groups);
    p.rows_per_cta = (p.rows_per_cta + kRowUnroll - 1) / kRowUnroll * kRowUnroll;
    row_groups = (int)((p.rows_pad + p.rows_per_cta - 1) / p.rows_per_cta);
    p.nparts = col_ctas * row_groups;
    *grid = dim3(col_ctas, row_groups);
    return p;
}

}  // namespace

cudaError_t launch_quantize(const QuantJob& job, cudaStream_t s)
{
    dim3 grid;
    const QuantParams p = make_params(job, &grid);
    const bool mod = job.shift != nullptr;

    if (!job.gscale_given) {
        if (mod) amax_kernel<true><<<grid, kThreads, 0, s>>>(p);
        else amax_kernel<false><<<grid, kThreads, 0, s>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (mod) pack_kernel<true><<<grid, kThreads, 0, s>>>(p);
    else pack_kernel<false><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_amax(const QuantJob& job, float* amax_out, cudaStream_t s)
{
    dim3 grid;
    const QuantParams p = make_params(job, &grid);
    if (job.shift != nullptr) amax_kernel<true><<<grid, kThreads, 0, s>>>(p);
    else amax_kernel<false><<<grid, kThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    reduce_partials_kernel<<<1, kThreads, 0, s>>>(p.partials, p.nparts, amax_out);
    return cudaGetLastError();
}

cudaError_t launch_gscale_from_amax(const float* amax, float* gscale, cudaStream_t s)
{
    gscale_from_amax_kernel<<<1, 1, 0, s>>>(amax, gscale);
    return cudaGetLastError();
}

}  // namespace h3fp4
