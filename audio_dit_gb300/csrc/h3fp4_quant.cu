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
#include "nvfp4_encode.cuh"
#include "act_prologue.cuh"

namespace h3fp4 {
namespace {

constexpr int kThreads = 64;     // one 16-element block per thread: 1024 columns per CTA
constexpr int kRowUnroll = 4;    // rows in flight per thread
// Rows in flight per thread in the pack pass: three with the prologue (its
// sixteen (1 + scale, shift) pairs take registers; measured faster than four
// or two on fc1 and attn_out), four without.
template <bool kMod>
__host__ __device__ constexpr int pack_unroll()
{
    return kMod ? 3 : 4;
}

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

// Sixteen bf16 values = 32 bytes: one 256-bit load when the row pointer is
// 32-byte aligned, two 128-bit loads otherwise.
template <bool kWide>
__device__ __forceinline__ V16 ld16(const uint16_t* p)
{
    V16 v;
    if (kWide) {
        asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                       "=r"(v.w[6]), "=r"(v.w[7])
                     : "l"(p));
    } else {
        const uint4 a = ld_stream_v4(p);
        const uint4 b = ld_stream_v4(p + 8);
        v.w[0] = a.x; v.w[1] = a.y; v.w[2] = a.z; v.w[3] = a.w;
        v.w[4] = b.x; v.w[5] = b.y; v.w[6] = b.z; v.w[7] = b.w;
    }
    return v;
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

template <bool kMod, bool kWide>
__global__ void __launch_bounds__(kThreads) amax_kernel(QuantParams p)
{
    __shared__ float red[kThreads / 32];
    griddep_launch_dependents();
    griddep_wait();  // X and the modulation vectors may come from the previous kernel
    const int cb = blockIdx.x * kThreads + threadIdx.x;  // 16-element block column
    const bool valid = cb < p.K / 16;
    const long long r0 = (long long)blockIdx.y * p.rows_per_cta;
    const long long r1 = min(r0 + (long long)p.rows_per_cta, p.rows);
    const uint16_t* xc = p.x + (long long)cb * 16;

    ModCols mc;
    init_mod(mc);
    float mx = 0.0f;
    for (long long r = r0; r < r1; r += kRowUnroll) {
        const int n = (int)min((long long)kRowUnroll, r1 - r);
        V16 v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u)
            if (valid && u < n) v[u] = ld16<kWide>(xc + (r + u) * p.K);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            if (!(valid && u < n)) continue;
            if (kMod && r + u >= mc.seg_end) load_mod(p.scale, p.shift, p.K, p.seg, segment_of(p.seg, r + u), cb, mc);
            float f[16];
            unpack16(v[u], f);
            if (kMod) {
                // The modulated values before their bf16 rounding: rounding to
                // nearest is monotone and odd, so the largest |bf16(m)| is the
                // bf16 rounding of the largest |m|, applied once below.
#pragma unroll
                for (int j = 0; j < 8; ++j) unf2(fma2(f2(f[2 * j], f[2 * j + 1]), mc.onep[j], mc.sh[j]), f[2 * j], f[2 * j + 1]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fabsf(f[j]));
        }
    }
    if (kMod) mx = __bfloat162float(__float2bfloat16_rn(mx));
    const float m = block_reduce_max(mx, red);
    if (threadIdx.x == 0) p.partials[blockIdx.y * gridDim.x + blockIdx.x] = m;
}

// ------------------------------------------------------------------ pass 2: pack

template <bool kMod, bool kWide>
__global__ void __launch_bounds__(kThreads, 10) pack_kernel(QuantParams p)
{
    __shared__ float red[kThreads / 32];
    __shared__ float rcp_tab[128];  // E4M3 code S -> RN(1 / RN(S * s)), 0 for S = 0
    griddep_launch_dependents();
    griddep_wait();  // the amax partials (or the given scale) come from the previous kernel
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
    // The effective scale eff = S * s and its reciprocal depend only on the
    // block's E4M3 code S (127 finite non-negative values; the saturating
    // conversion never yields the NaN code 0x7F): one table per CTA instead of
    // a multiply and an IEEE reciprocal per block.
    for (int c = threadIdx.x; c < 128; c += kThreads) {
        rcp_tab[c] = block_rcp((uint32_t)c, s_g);
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int cb = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = cb < p.K / 16;            // uniform over each group of 4 lanes
    const long long kb4 = p.K / 64;             // scale tiles per 128 rows
    const long long r0 = (long long)blockIdx.y * p.rows_per_cta;
    const long long r1 = min(r0 + (long long)p.rows_per_cta, p.rows_pad);
    const long long rend = min(r1, p.rows);      // real rows [r0, rend), padding rows [rend, r1)
    // Lanes past the last block column load column 0 (in bounds) and store nothing.
    const uint16_t* xc = p.x + (long long)(valid ? cb : 0) * 16;
    uint2* codes_c = reinterpret_cast<uint2*>(p.codes) + cb;  // 8 bytes per block
    const long long g = cb >> 2;                 // 64-column group = scale word index
    const bool sf_writer = valid && (lane & 3) == 0;

    ModCols mc;
    init_mod(mc);
    // Rows are walked from the end of the CTA's range back to its start: the
    // amax pass walked them forwards, so the rows it read last -- the ones most
    // likely still in L2 when X is larger than L2 -- are re-read first.
    constexpr int kPU = pack_unroll<kMod>();
    const long long last = rend > r0 ? r0 + (rend - r0 - 1) / kPU * kPU : r0 - kPU;
    for (long long r = last; r >= r0; r -= kPU) {
        V16 v[kPU];
#pragma unroll
        for (int u = 0; u < kPU; ++u)
            if (r + u < rend) v[u] = ld16<kWide>(xc + (r + u) * p.K);
#pragma unroll
        for (int u = 0; u < kPU; ++u) {
            const long long rr = r + u;
            if (rr >= rend) break;                 // uniform over the CTA
            float f[16];
            unpack16(v[u], f);
            if (kMod) {
                if ((rr >= mc.seg_end || rr < mc.seg_begin) && valid) load_mod(p.scale, p.shift, p.K, p.seg, segment_of(p.seg, rr), cb, mc);
                modulate16<kMod>(f, mc);
            }
            float bmax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(f[j]));
            const uint32_t S = block_scale_code(bmax, s_g);
            const float rcp = rcp_tab[S & 127u];
            const uint64_t rcp2 = f2(rcp, rcp);
            float q[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) unf2(mul2(f2(f[2 * j], f[2 * j + 1]), rcp2), q[2 * j], q[2 * j + 1]);
            const uint32_t w0 = e2m1x8(reinterpret_cast<const float(&)[8]>(q[0]));
            const uint32_t w1 = e2m1x8(reinterpret_cast<const float(&)[8]>(q[8]));
            if (valid) codes_c[rr * (p.K / 16)] = make_uint2(w0, w1);
            // gather the four block scales of this 64-column group into lane%4 == 0
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, S, 1);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, S, 2);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, S, 3);
            if (sf_writer) {
                const uint32_t r7 = (uint32_t)rr & 127u;
                const long long off = (((rr >> 7) * kb4 + g) << 9) + ((r7 & 31u) << 4) + ((r7 >> 5) << 2);
                *reinterpret_cast<uint32_t*>(p.sf + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
            }
        }
    }
    // Padding rows up to the next multiple of 128: zero scale words.
    if (sf_writer)
        for (long long rr = max(r0, rend); rr < r1; ++rr) {
            const uint32_t r7 = (uint32_t)rr & 127u;
            const long long off = (((rr >> 7) * kb4 + g) << 9) + ((r7 & 31u) << 4) + ((r7 >> 5) << 2);
            *reinterpret_cast<uint32_t*>(p.sf + off) = 0u;
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

// Resident CTAs per SM of each pass (occupancy of its slowest variant),
// cached once per process (every accepted device is sm_103).
int amax_ctas_per_sm()
{
    static const int n = [] {
        int a = 0, b = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, amax_kernel<true, true>, kThreads, 0);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, amax_kernel<true, false>, kThreads, 0);
        return max(1, min(a, b));
    }();
    return n;
}

int pack_ctas_per_sm()
{
    static const int n = [] {
        int a = 0, b = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, pack_kernel<true, true>, kThreads, 0);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, pack_kernel<true, false>, kThreads, 0);
        return max(1, min(a, b));
    }();
    return n;
}

// Parameters and grid of one pass: one full wave of `per_sm` resident CTAs
// per SM, each walking a contiguous range of rows (no half-empty second wave).
QuantParams make_params(const QuantJob& job, int per_sm, dim3* grid)
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

    const int col_ctas = (int)((job.K / 16 + kThreads - 1) / kThreads);
    const int target = sm_count_current_device() * per_sm;
    int row_groups = (target + col_ctas - 1) / col_ctas;
    row_groups = max(1, min(row_groups, kMaxPartials / col_ctas));
    // rows per CTA covers the padded rows so the pack pass zeroes scale padding
    // Rows per CTA are a multiple of the unroll depth unless that rounding would
    // leave more than 5 % of the wave's CTA slots empty (small activations).
    p.rows_per_cta = (int)((p.rows_pad + row_groups - 1) / row_groups);
    {
        const int rounded = (p.rows_per_cta + kRowUnroll - 1) / kRowUnroll * kRowUnroll;
        const long long groups = (p.rows_pad + rounded - 1) / rounded;
        if (groups * col_ctas * 100 >= (long long)target * 95) p.rows_per_cta = rounded;
    }
    row_groups = (int)((p.rows_pad + p.rows_per_cta - 1) / p.rows_per_cta);
    p.nparts = col_ctas * row_groups;
    *grid = dim3(col_ctas, row_groups);
    return p;
}

// Row starts are 32-byte aligned when the base is (K % 64 == 0).
bool wide_ok(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 31u) == 0; }

// Both passes launch with programmatic stream serialization: their CTAs may be
// scheduled while the previous kernel drains and wait for it in-kernel.
cudaError_t launch_pdl(void (*kernel)(QuantParams), const QuantParams& p, dim3 grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <bool kMod>
cudaError_t launch_amax_t(const QuantParams& p, dim3 grid, bool wide, cudaStream_t s)
{
    return launch_pdl(wide ? amax_kernel<kMod, true> : amax_kernel<kMod, false>, p, grid, s);
}

template <bool kMod>
cudaError_t launch_pack_t(const QuantParams& p, dim3 grid, bool wide, cudaStream_t s)
{
    return launch_pdl(wide ? pack_kernel<kMod, true> : pack_kernel<kMod, false>, p, grid, s);
}

}  // namespace

cudaError_t launch_quantize(const QuantJob& job, cudaStream_t s)
{
    // Each pass gets its own one-wave grid; the pack pass reduces the partials
    // of the amax pass's grid.
    dim3 agrid, pgrid;
    const QuantParams pa = make_params(job, amax_ctas_per_sm(), &agrid);
    QuantParams pp = make_params(job, pack_ctas_per_sm(), &pgrid);
    pp.nparts = pa.nparts;
    const bool mod = job.shift != nullptr;
    const bool wide = wide_ok(job.x);
    if (!job.gscale_given) {
        const cudaError_t e = mod ? launch_amax_t<true>(pa, agrid, wide, s) : launch_amax_t<false>(pa, agrid, wide, s);
        if (e != cudaSuccess) return e;
    }
    return mod ? launch_pack_t<true>(pp, pgrid, wide, s) : launch_pack_t<false>(pp, pgrid, wide, s);
}

cudaError_t launch_amax_partials(const QuantJob& job, int* nparts, cudaStream_t s)
{
    dim3 grid;
    const QuantParams p = make_params(job, amax_ctas_per_sm(), &grid);
    *nparts = p.nparts;
    return job.shift != nullptr ? launch_amax_t<true>(p, grid, wide_ok(job.x), s)
                                : launch_amax_t<false>(p, grid, wide_ok(job.x), s);
}

cudaError_t launch_amax(const QuantJob& job, float* amax_out, cudaStream_t s)
{
    dim3 grid;
    const QuantParams p = make_params(job, amax_ctas_per_sm(), &grid);
    const cudaError_t e = job.shift != nullptr ? launch_amax_t<true>(p, grid, wide_ok(job.x), s)
                                               : launch_amax_t<false>(p, grid, wide_ok(job.x), s);
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
