// Tensor-core ceilings of this device for block-scaled FP4, no global traffic,
// operands resident in shared memory (or TMEM) and block scales resident in
// TMEM: back-to-back tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X --
// the only tcgen05 kind that carries NVFP4 (16-element blocks, E4M3 scales) --
// in each of the forms the instruction offers:
//   kSingle       cta_group::1, M=128, N=256, K=64, A from shared memory
//   kPair         cta_group::2, M=256, N=256, K=64 (the GEMM's instruction)
//   kSingleTmemA  cta_group::1 with A from TMEM
//   kPairTmemA    cta_group::2 with A from TMEM
//   kSingleN128   cta_group::1, two N=128 MMAs per step sharing A
//   kSingleN128Collector  the same with .collector::a::fill / ::lastuse
//   kPairN128     cta_group::2, two N=128 MMAs per step sharing A
// Used as measured FP4 peaks next to the nominal one in roofline reports.
#include <cstdint>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"

namespace h3fp4 {
namespace {

constexpr int kPeakSmem = 120 * 1024;  // one CTA per SM (its TMEM allocation never waits)
constexpr int kFill = 65536;           // operand bytes filled with a fixed pattern

template <int F>
__host__ __device__ constexpr bool is_pair()
{
    return F == H3FP4_MMA_PAIR || F == H3FP4_MMA_PAIR_TMEM_A || F == H3FP4_MMA_PAIR_N128;
}

template <int F>
__host__ __device__ constexpr bool is_n128()
{
    return F == H3FP4_MMA_SINGLE_N128 || F == H3FP4_MMA_SINGLE_N128_COLLECTOR || F == H3FP4_MMA_PAIR_N128;
}

template <int F>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                    uint32_t acc, uint32_t a_tmem, int second)
{
#define H3_PRED "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
    if constexpr (F == H3FP4_MMA_SINGLE || F == H3FP4_MMA_SINGLE_N128) {
        asm volatile(H3_PRED "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                     ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    } else if constexpr (F == H3FP4_MMA_PAIR || F == H3FP4_MMA_PAIR_N128) {
        asm volatile(H3_PRED "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                     ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    } else if constexpr (F == H3FP4_MMA_SINGLE_TMEM_A) {
        asm volatile(H3_PRED "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%7], %2, %3, [%5], [%6], p;\n\t}"
                     ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb), "r"(a_tmem) : "memory");
    } else if constexpr (F == H3FP4_MMA_PAIR_TMEM_A) {
        asm volatile(H3_PRED "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%7], %2, %3, [%5], [%6], p;\n\t}"
                     ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb), "r"(a_tmem) : "memory");
    } else if constexpr (F == H3FP4_MMA_SINGLE_N128_COLLECTOR) {
        if (!second)
            asm volatile(H3_PRED "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X.collector::a::fill [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
        else
            asm volatile(H3_PRED "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X.collector::a::lastuse [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    }
#undef H3_PRED
}

// Per CTA, per iteration (one K = 64 step): 2 * 128 * 256 * 64 flops in every form.
template <int F>
__global__ void __launch_bounds__(128, 1) mma_form_kernel(int iters, unsigned int* status)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int warp = threadIdx.x >> 5;
    if ((smem_u32(sm) & 1023u) != 0) return;  // same layout in every CTA: a pair leaves together
    for (int i = threadIdx.x; i < kFill; i += blockDim.x) sm[i] = (uint8_t)((i * 7 + 3) & 0x77);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    if (warp == 0) {
        if constexpr (is_pair<F>()) {
            tmem_alloc_pair(&tbase, 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tbase, 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {  // columns 256..511 (A operand for the TMEM forms, block scales): every byte 0x38 (E4M3 1.0)
        uint32_t v[32];
        for (int i = 0; i < 32; ++i) v[i] = 0x38383838u;
        const uint32_t t = tbase + ((uint32_t)(32 * warp) << 16);
        for (int c = 256; c < 512; c += 32) tc_st_32x32b_x32(t + c, v);
        tc_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if constexpr (is_pair<F>()) cluster_sync();  // the partner's operands and scales are in place
    tc_fence_after();
    const bool issuer = threadIdx.x == 0 && (!is_pair<F>() || cluster_ctarank() == 0);
    if (issuer) {
        const uint32_t s = smem_u32(sm);
        const uint32_t m4 = is_pair<F>() ? 16u : 8u;                 // M >> 4
        const uint32_t n8 = is_n128<F>() ? 16u : 32u;                // N >> 3
        const uint32_t idesc = (1u << 7) | (1u << 10) | (n8 << 17) | (m4 << 24);  // E2M1 x E2M1, UE4M3 scales
        for (int i = 0; i < iters; ++i) {
            const uint32_t j = (uint32_t)(i & 3);
            const uint64_t a = smem_desc(s + 32 * j, 16, 1024, 2);
            const uint64_t b = smem_desc(s + 16384 + 32 * j, 16, 1024, 2);
            const uint32_t acc = i > 0 ? 1u : 0u;
            if constexpr (is_n128<F>()) {
                // B rows [0, 128) and [128, 256) (per CTA [0, 64) / [64, 128) for the pair) into
                // the two halves of the accumulator, both with the same A
                const uint64_t b2 = b + ((is_pair<F>() ? 8192u : 16384u) >> 4);
                mma<F>(tbase, a, b, idesc, tbase + 256 + 4 * j, tbase + 320 + 8 * j, acc, 0, 0);
                mma<F>(tbase + 128, a, b2, idesc, tbase + 256 + 4 * j, tbase + 324 + 8 * j, acc, 0, 1);
            } else {
                mma<F>(tbase, a, b, idesc, tbase + 288 + 4 * j, tbase + 320 + 8 * j, acc, tbase + 256 + 8 * j, 0);
            }
        }
        if constexpr (is_pair<F>()) tc_commit_pair(&bar); else tc_commit(&bar);
        (void)mbar_wait(&bar, 0u, 2000000000ull, status, kStatusTimeoutMma);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (is_pair<F>()) cluster_sync();  // no CTA releases TMEM while the leader's MMAs may still use it
    if (warp == 0) {
        tc_fence_after();
        if constexpr (is_pair<F>()) tmem_dealloc_pair(tbase, 512); else tmem_dealloc(tbase, 512);
    }
    if constexpr (is_pair<F>()) cluster_sync();
}

template <int F>
cudaError_t measure_form(int iters, unsigned int* status, float* tflops)
{
    auto kern = mma_form_kernel<F>;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), kPeakSmem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count_current_device();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = is_pair<F>() ? 2 : 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(is_pair<F>() ? 2 * (unsigned)(sms / 2) : (unsigned)sms);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kPeakSmem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (is_pair<F>()) {
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters <= 0) return cudaErrorInvalidConfiguration;
        if (2 * clusters < (int)cfg.gridDim.x) cfg.gridDim = dim3(2 * (unsigned)clusters);
    }
    cudaEvent_t e0, e1;
    e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) {
        cudaEventDestroy(e0);
        return e;
    }
    e = cudaLaunchKernelEx(&cfg, kern, 100, status);  // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(e0);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, kern, iters, status);
    if (e == cudaSuccess) e = cudaEventRecord(e1);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    *tflops = (float)(2.0 * 128 * 256 * 64 * (double)iters * cfg.gridDim.x / (ms * 1e-3) / 1e12);
    return cudaGetLastError();
}

}  // namespace

cudaError_t measure_fp4_form(int form, int iters, unsigned int* status, float* tflops)
{
    switch (form) {
    case H3FP4_MMA_SINGLE: return measure_form<H3FP4_MMA_SINGLE>(iters, status, tflops);
    case H3FP4_MMA_PAIR: return measure_form<H3FP4_MMA_PAIR>(iters, status, tflops);
    case H3FP4_MMA_SINGLE_TMEM_A: return measure_form<H3FP4_MMA_SINGLE_TMEM_A>(iters, status, tflops);
    case H3FP4_MMA_PAIR_TMEM_A: return measure_form<H3FP4_MMA_PAIR_TMEM_A>(iters, status, tflops);
    case H3FP4_MMA_SINGLE_N128: return measure_form<H3FP4_MMA_SINGLE_N128>(iters, status, tflops);
    case H3FP4_MMA_SINGLE_N128_COLLECTOR: return measure_form<H3FP4_MMA_SINGLE_N128_COLLECTOR>(iters, status, tflops);
    case H3FP4_MMA_PAIR_N128: return measure_form<H3FP4_MMA_PAIR_N128>(iters, status, tflops);
    }
    return cudaErrorInvalidValue;
}

cudaError_t measure_fp4_peak(int iters, unsigned int* status, float* tflops)
{
    return measure_form<H3FP4_MMA_SINGLE>(iters, status, tflops);
}

cudaError_t measure_fp4_pair_peak(int iters, unsigned int* status, float* tflops)
{
    return measure_form<H3FP4_MMA_PAIR>(iters, status, tflops);
}

}  // namespace h3fp4
