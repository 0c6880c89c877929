// Block-scaled NVFP4 GEMM with fused bias + residual-gate epilogue, sm_103a.
//
//   out[m][n] = bf16( R[m][n] + g[seg(m)][n] * (alpha * acc[m][n] + b[n]) )
//   acc[m][n] = sum_k e2m1(A[m][k]) * SA[m][k/16] * e2m1(W[n][k]) * SW[n][k/16]
//   alpha     = s_a * s_w, applied to the fp32 accumulator before the BF16 cast
//               ("H3 Runtime Current State", "Owned Performance Kernels":
//               alpha-before-BF16 epilogue; "Implemented And Validated": fused
//               residual gates).
//
// Structure (one persistent CTA per SM, 352 threads, warp-specialised):
//   warp 0      TMA producer: A/W code tiles (128-byte swizzle) and the 512-byte
//               block-scale tiles (plain bulk copies) into a 3-stage ring.
//   warp 10     block-scale copier: per landed stage, twelve tcgen05.cp
//               32x128b.warpx4 of the scale tiles into that stage's TMEM slot,
//               then a tcgen05.commit on the stage's "scales ready" barrier.
//               Each copy occupies the tensor pipe for ~60 cycles whatever its
//               size; issuing them from their own thread lets them overlap the
//               MMAs instead of serialising behind them on one issuer.
//   warp 1      TMEM owner + MMA issuer: per stage four
//               tcgen05.mma.kind::mxf4nvf4.block_scale (M=128, N=256, K=64)
//               once the stage's scales are in TMEM.
//   warps 2-9   epilogue: tcgen05.ld the 128x256 fp32 accumulator (each warp 32
//               rows x 128 columns), release TMEM, then alpha/bias/gate/residual
//               in fp32, bf16 into a 64-byte-swizzled staging tile and TMA store;
//               the residual tile is TMA-loaded into the same staging buffer
//               ahead of time.
//
// Tile 128 x 256 x 256 (K in elements).  TMEM: accumulator in columns
// [0, 256); stage s scale slots at 256 + 48 s (16 columns for A's four 64-K
// groups, 32 for W's two 128-row halves).  Every mbarrier wait is bounded.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"

namespace h3fp4 {
namespace {

constexpr int BM = 128, BN = 256, BK = 256;
constexpr int kStages = 3;
constexpr int kThreads = 352;
constexpr int kCopyWarp = 10;
constexpr int kEpiWarps = 8;
constexpr uint32_t kABytes = BM * BK / 2;            // 16384
constexpr uint32_t kBBytes = BN * BK / 2;            // 32768
constexpr uint32_t kSFABytes = BM * (BK / 16);       // 2048: four 512-byte tiles
constexpr uint32_t kSFBBytes = BN * (BK / 16);       // 4096: two rows of four tiles
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;
constexpr uint32_t kChunkBytes = 32 * 32 * 2;        // 32 rows x 32 bf16
constexpr uint32_t kEpiWarpBytes = 4 * kChunkBytes;  // 8192
constexpr uint32_t kEpiOff = kStages * kStageBytes;
constexpr uint32_t kBarOff = kEpiOff + kEpiWarps * kEpiWarpBytes;
constexpr uint32_t kSmemBytes = kBarOff + 256;  // barriers, TMEM address, abort flag
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmem = 256;
constexpr uint32_t kSfTmemPerStage = 48;
static_assert(kSfTmem + kStages * kSfTmemPerStage <= kTmemCols, "TMEM budget");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Instruction descriptor, kind::mxf4nvf4: A/B E2M1 (1) in bits 7-9 / 10-12,
// K-major A and B, N >> 3 in bits 17-22, UE4M3 scales (bit 23 = 0),
// M >> 4 in bits 24-28, scale-factor ids 0, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct GemmParams {
    const uint8_t* a_sf;
    const uint8_t* w_sf;
    const float* a_gscale;
    const float* w_gscale;
    const __nv_bfloat16* bias;
    const float* gate;
    int M, N, K;
    int m_tiles, n_tiles, k_stages, kb4, n_sf_tiles;
    int has_resid;
    Segments seg;
    unsigned int* status;
    unsigned long long wait_ns;
    int stall;  // self-test: the producer issues nothing, so every consumer wait must time out
};

__device__ __forceinline__ int segment_of_row(const Segments& s, int r)
{
    int i = 0;
#pragma unroll 1
    while (i + 1 < s.nseg && r >= s.off[i + 1]) ++i;
    return i;
}

// Byte offset of 16-byte chunk j of row r inside a 32-row x 64-byte tile stored
// with the TMA 64-byte swizzle (chunk bits 4-5 XOR address bits 7-8).
__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t j)
{
    const uint32_t lin = r * 64u + j * 16u;
    return lin ^ (((lin >> 7) & 3u) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmR,
                      const GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Swizzled TMA tiles need 1024-byte alignment; refuse to run otherwise.
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSmemAlign);
        return;
    }

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* rbar = acc_empty + 1;  // one per epilogue warp
    uint64_t* done_bar = rbar + kEpiWarps;
    uint64_t* sfready = done_bar + 1;  // [kStages]: the stage's scales are in TMEM
    uint64_t* cp_done = sfready + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cp_done + 1);
    volatile int& s_abort = *reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kEpiWarps);
        for (int e = 0; e < kEpiWarps; ++e) mbar_init(&rbar[e], 1);
        mbar_init(done_bar, 1);
        for (int s = 0; s < kStages; ++s) mbar_init(&sfready[s], 1);
        mbar_init(cp_done, 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmOut);
        if (p.has_resid) prefetch_tensormap(&tmR);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int num_tiles = p.m_tiles * p.n_tiles;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t fills[kStages] = {};
            for (int tile = blockIdx.x; tile < num_tiles && !s_abort && !p.stall; tile += gridDim.x) {
                const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
                const int sfb_tiles = (2 * nt + 1 < p.n_sf_tiles) ? 2 : 1;
                for (int kb = 0; kb < p.k_stages; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns, p.status, kStatusTimeoutProducer)) {
                        s_abort = 1;
                        break;
                    }
                    const int nk = min(4, p.kb4 - kb * 4);
                    uint8_t* st = smem + stage * kStageBytes;
                    const uint32_t bytes = kABytes + kBBytes + (uint32_t)(nk * 512) * (1 + sfb_tiles);
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    tma_load_2d(st, &tmA, &full[stage], kb * (BK / 2), mt * BM);
                    tma_load_2d(st + kABytes, &tmB, &full[stage], kb * (BK / 2), nt * BN);
                    bulk_load(st + kABytes + kBBytes, p.a_sf + ((size_t)mt * p.kb4 + kb * 4) * 512, nk * 512,
                              &full[stage]);
                    for (int j = 0; j < sfb_tiles; ++j)
                        bulk_load(st + kABytes + kBBytes + kSFABytes + j * 2048,
                                  p.w_sf + ((size_t)(2 * nt + j) * p.kb4 + kb * 4) * 512, nk * 512, &full[stage]);
                    ++fills[stage];
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: every issued copy must land before the CTA may exit.  The last
            // fill of stage s completes phase fills[s] - 1 of full[s].
            for (int s = 0; s < kStages; ++s)
                if (fills[s] > 0)
                    (void)mbar_wait(&full[s], (fills[s] - 1u) & 1u, p.wait_ns, p.status, kStatusTimeoutProducer);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles && !s_abort; tile += gridDim.x) {
                if (!mbar_wait(acc_empty, acc_phase ^ 1u, p.wait_ns, p.status, kStatusTimeoutMma)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < p.k_stages; ++kb) {
                    if (!mbar_wait(&sfready[stage], phase, p.wait_ns, p.status, kStatusTimeoutMma) ||
                        !mbar_wait(&full[stage], phase, p.wait_ns, p.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, p.kb4 - kb * 4);
                    const uint32_t st = smem_u32(smem + stage * kStageBytes);
                    const uint32_t sfa_t = tmem + kSfTmem + stage * kSfTmemPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    for (int j = 0; j < nk; ++j) {
                        const uint64_t adesc = smem_desc(st + 32 * j, 16, 1024, 2);
                        const uint64_t bdesc = smem_desc(st + kABytes + 32 * j, 16, 1024, 2);
                        mma_mxf4nvf4(tmem, adesc, bdesc, kIdesc, sfa_t + 4 * j, sfb_t + 8 * j,
                                     (kb > 0 || j > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    s_abort = 1;
                    break;
                }
                tc_commit(acc_full);
                acc_phase ^= 1u;
            }
            // Every issued MMA / copy must finish before TMEM is released.
            tc_commit(done_bar);
            (void)mbar_wait(done_bar, 0u, p.wait_ns, p.status, kStatusTimeoutMma);
        }
    } else if (warp == kCopyWarp) {
        // ---------------------------------------------------------------- block-scale copier
        // The TMEM slot of a stage is rewritten only after the stage was refilled,
        // i.e. after the MMAs that read the previous contents committed.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles && !s_abort; tile += gridDim.x) {
                bool ok = true;
                for (int kb = 0; kb < p.k_stages; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, p.kb4 - kb * 4);
                    const uint32_t st = smem_u32(smem + stage * kStageBytes);
                    const uint32_t sfa_s = st + kABytes + kBBytes, sfb_s = sfa_s + kSFABytes;
                    const uint32_t sfa_t = tmem + kSfTmem + stage * kSfTmemPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    for (int j = 0; j < nk; ++j) {
                        tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc(sfa_s + 512 * j, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sfb_t + 8 * j, smem_desc(sfb_s + 512 * j, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sfb_t + 8 * j + 4, smem_desc(sfb_s + 2048 + 512 * j, 0, 128, 0));
                    }
                    tc_commit(&sfready[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    s_abort = 1;
                    break;
                }
            }
            // every copy must finish before TMEM is released
            tc_commit(cp_done);
            (void)mbar_wait(cp_done, 0u, p.wait_ns, p.status, kStatusTimeoutMma);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int e = warp - 2;            // 0..7
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int h = e >> 2;              // column half of the 256-wide tile
        uint8_t* stg = smem + kEpiOff + e * kEpiWarpBytes;
        const float alpha = __fmul_rn(__ldg(p.a_gscale), __ldg(p.w_gscale));
        uint32_t acc_phase = 0, r_phase = 0;
        bool r_pending = false;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            if (__any_sync(0xffffffffu, s_abort != 0)) break;  // warp-uniform exit
            const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
            const int m0 = mt * BM + 32 * q;      // first row of this warp
            const int nc0 = nt * BN + 128 * h;    // first column of this warp
            if (lane == 0) bulk_wait_read_all();  // staging buffer free again
            __syncwarp();
            if (p.has_resid && lane == 0) {
                mbar_arrive_expect_tx(&rbar[e], 4 * kChunkBytes);
                for (int c = 0; c < 4; ++c) tma_load_2d(stg + c * kChunkBytes, &tmR, &rbar[e], nc0 + 32 * c, m0);
            }
            r_pending = p.has_resid != 0;
            bool ok = mbar_wait(acc_full, acc_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) {
                s_abort = 1;
                break;
            }
            acc_phase ^= 1u;
            tc_fence_after();
            uint32_t acc[4][32];
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + 128u * h;
#pragma unroll
            for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(tbase + 32u * c, acc[c]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);   // accumulator may be overwritten now

            if (p.has_resid) {
                ok = mbar_wait(&rbar[e], r_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
                if (!__all_sync(0xffffffffu, ok)) {
                    s_abort = 1;
                    break;
                }
                r_phase ^= 1u;
                r_pending = false;
            }
            const int row = m0 + lane;
            const float* grow = nullptr;
            if (p.gate != nullptr && row < p.M) grow = p.gate + (size_t)segment_of_row(p.seg, row) * p.N;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint8_t* buf = stg + c * kChunkBytes;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n8 = nc0 + 32 * c + 8 * j;
                    float b[8], g[8], r[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        b[i] = 0.0f;
                        g[i] = 1.0f;
                        r[i] = 0.0f;
                    }
                    if (n8 < p.N) {
                        if (p.bias != nullptr) {
                            const uint4 bv = __ldg(reinterpret_cast<const uint4*>(p.bias + n8));
                            const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                b[2 * i] = __uint_as_float(bw[i] << 16);
                                b[2 * i + 1] = __uint_as_float(bw[i] & 0xFFFF0000u);
                            }
                        }
                        if (grow != nullptr) {
                            const float4 g0 = __ldg(reinterpret_cast<const float4*>(grow + n8));
                            const float4 g1 = __ldg(reinterpret_cast<const float4*>(grow + n8) + 1);
                            g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
                            g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
                        }
                    }
                    uint4* slot = reinterpret_cast<uint4*>(buf + swz64(lane, j));
                    if (p.has_resid) {
                        const uint4 rv = *slot;
                        const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            r[2 * i] = __uint_as_float(rw[i] << 16);
                            r[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
                        }
                    }
                    float o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float y = __fmul_rn(__uint_as_float(acc[c][8 * j + i]), alpha);
                        const float v = __fadd_rn(y, b[i]);
                        o[i] = (grow != nullptr) ? __fmaf_rn(g[i], v, r[i]) : __fadd_rn(v, r[i]);
                    }
                    *slot = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                       pack_bf16x2(o[6], o[7]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tma_store_2d(&tmOut, buf, nc0 + 32 * c, m0);
            }
            if (lane == 0) bulk_commit();
        }
        if (r_pending) (void)mbar_wait(&rbar[e], r_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

static cudaError_t launch_gemm_impl(const GemmJob& job, int stall, cudaStream_t s);

cudaError_t launch_gemm(const GemmJob& job, cudaStream_t s) { return launch_gemm_impl(job, 0, s); }

cudaError_t launch_gemm_stall_selftest(const GemmJob& job, cudaStream_t s) { return launch_gemm_impl(job, 1, s); }

static cudaError_t launch_gemm_impl(const GemmJob& job, int stall, cudaStream_t s)
{
    CUtensorMap tmA, tmB, tmOut, tmR;
    const uint64_t kbytes = (uint64_t)job.K / 2;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.a_codes, kbytes, (uint64_t)job.M, kbytes, BK / 2, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.w_codes, kbytes, (uint64_t)job.N, kbytes, BK / 2, BN,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, job.out, (uint64_t)job.N, (uint64_t)job.M,
                     (uint64_t)job.N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_2d(&tmR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, job.resid ? job.resid : job.out, (uint64_t)job.N,
                     (uint64_t)job.M, (uint64_t)job.N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;

    GemmParams p{};
    p.a_sf = job.a_sf;
    p.w_sf = job.w_sf;
    p.a_gscale = job.a_gscale;
    p.w_gscale = job.w_gscale;
    p.bias = static_cast<const __nv_bfloat16*>(job.bias);
    p.gate = job.gate;
    p.M = (int)job.M;
    p.N = (int)job.N;
    p.K = (int)job.K;
    p.m_tiles = (int)((job.M + BM - 1) / BM);
    p.n_tiles = (int)((job.N + BN - 1) / BN);
    p.k_stages = (int)((job.K + BK - 1) / BK);
    p.kb4 = (int)(job.K / 64);
    p.n_sf_tiles = (int)((job.N + 127) / 128);
    p.has_resid = job.resid != nullptr ? 1 : 0;
    p.seg = job.seg;
    p.status = job.status;
    p.wait_ns = job.wait_limit_ns;
    p.stall = stall;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;

    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = tiles < sm_count_current_device() ? tiles : sm_count_current_device();
    nvfp4_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, tmOut, tmR, p);
    return cudaGetLastError();
}

}  // namespace h3fp4
