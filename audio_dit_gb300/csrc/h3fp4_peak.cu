// Tensor-core ceilings of this device for block-scaled FP4, no global traffic,
// operands resident in shared memory and block scales resident in TMEM:
//   single CTA: back-to-back tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale
//               .scale_vec::4X (M=128, N=256, K=64) on every SM;
//   CTA pair:   the same with .cta_group::2 (M=256, N=256, K=64) issued by the
//               leader of every 2-CTA cluster -- the instruction the GEMM uses.
// Used as measured FP4 peaks next to the nominal one in roofline reports.
#include <cstdint>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"

namespace h3fp4 {
namespace {

constexpr int kPeakSmem = 49152;  // A 16 KB + B 32 KB

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, unsigned int* status)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int warp = threadIdx.x >> 5;
    if ((smem_u32(sm) & 1023u) != 0) return;
    for (int i = threadIdx.x; i < kPeakSmem; i += blockDim.x) sm[i] = (uint8_t)((i * 7 + 3) & 0x77);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tbase, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {  // every block scale = 1.0 (E4M3 0x38) in columns 256..511
        uint32_t v[32];
        for (int i = 0; i < 32; ++i) v[i] = 0x38383838u;
        const uint32_t t = tbase + ((uint32_t)(32 * warp) << 16);
        for (int c = 256; c < 512; c += 32) tc_st_32x32b_x32(t + c, v);
        tc_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t s = smem_u32(sm);
        const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (8u << 24);  // N=256, M=128
        for (int i = 0; i < iters; ++i) {
            const uint32_t j = (uint32_t)(i & 3);
            mma_mxf4nvf4(tbase, smem_desc(s + 32 * j, 16, 1024, 2), smem_desc(s + 16384 + 32 * j, 16, 1024, 2), idesc,
                         tbase + 256 + 4 * j, tbase + 320 + 8 * j, i > 0 ? 1u : 0u);
        }
        tc_commit(&bar);
        (void)mbar_wait(&bar, 0u, 2000000000ull, status, kStatusTimeoutMma);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// One CTA per SM (the large dynamic allocation keeps a second CTA off the SM,
// whose TMEM allocation would otherwise wait for the first).
constexpr int kPairSmem = 120 * 1024;

__global__ void __launch_bounds__(128, 1) mma_pair_peak_kernel(int iters, unsigned int* status)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int warp = threadIdx.x >> 5;
    if ((smem_u32(sm) & 1023u) != 0) return;  // same layout in both CTAs: both return
    for (int i = threadIdx.x; i < 32768; i += blockDim.x) sm[i] = (uint8_t)((i * 7 + 3) & 0x77);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(&tbase, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {  // every block scale = 1.0 (E4M3 0x38) in columns 256..511 of both CTAs
        uint32_t v[32];
        for (int i = 0; i < 32; ++i) v[i] = 0x38383838u;
        const uint32_t t = tbase + ((uint32_t)(32 * warp) << 16);
        for (int c = 256; c < 512; c += 32) tc_st_32x32b_x32(t + c, v);
        tc_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the partner's operands and scales are in place
    tc_fence_after();
    if (cluster_ctarank() == 0 && threadIdx.x == 0) {
        const uint32_t s = smem_u32(sm);
        const uint32_t idesc = (1u << 7) | (1u << 10) | (32u << 17) | (16u << 24);  // N=256, M=256
        for (int i = 0; i < iters; ++i) {
            const uint32_t j = (uint32_t)(i & 3);
            mma_pair_mxf4nvf4(tbase, smem_desc(s + 32 * j, 16, 1024, 2), smem_desc(s + 16384 + 32 * j, 16, 1024, 2),
                              idesc, tbase + 256 + 4 * j, tbase + 320 + 8 * j, i > 0 ? 1u : 0u);
        }
        tc_commit_pair(&bar);
        (void)mbar_wait(&bar, 0u, 2000000000ull, status, kStatusTimeoutMma);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA releases TMEM while the leader's MMAs may still use it
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, 512);
    }
    cluster_sync();
}

}  // namespace

cudaError_t measure_fp4_pair_peak(int iters, unsigned int* status, float* tflops)
{
    {
        const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(mma_pair_peak_kernel), kPairSmem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (unsigned)(sm_count_current_device() / 2));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int clusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, mma_pair_peak_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    if (2 * clusters < (int)cfg.gridDim.x) cfg.gridDim = dim3(2 * (unsigned)clusters);
    cudaEvent_t e0, e1;
    e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) return e;
    int warm = 100;
    e = cudaLaunchKernelEx(&cfg, mma_pair_peak_kernel, warm, status);  // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(e0);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, mma_pair_peak_kernel, iters, status);
    if (e == cudaSuccess) e = cudaEventRecord(e1);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    const double pairs = cfg.gridDim.x / 2;
    *tflops = (float)(2.0 * 256 * 256 * 64 * (double)iters * pairs / (ms * 1e-3) / 1e12);
    return cudaGetLastError();
}

cudaError_t measure_fp4_peak(int iters, unsigned int* status, float* tflops)
{
    {
        const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(mma_peak_kernel), kPeakSmem);
        if (e != cudaSuccess) return e;
    }
    const int sms = sm_count_current_device();
    cudaEvent_t e0, e1;
    cudaError_t e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) return e;
    mma_peak_kernel<<<sms, 128, kPeakSmem>>>(100, status);  // warm-up
    cudaEventRecord(e0);
    mma_peak_kernel<<<sms, 128, kPeakSmem>>>(iters, status);
    cudaEventRecord(e1);
    e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    *tflops = (float)(2.0 * 128 * 256 * 64 * (double)iters * sms / (ms * 1e-3) / 1e12);
    return cudaGetLastError();
}

}  // namespace h3fp4
