// Block-scaled NVFP4 GEMM with fused bias + residual-gate epilogue, sm_103a.
//
//   out[m][n] = bf16( R[m][n] + g[seg(m)][n] * (alpha * acc[m][n] + b[n]) )
//   acc[m][n] = sum_k e2m1(A[m][k]) * SA[m][k/16] * e2m1(W[n][k]) * SW[n][k/16]
//   alpha     = s_a * s_w, applied to the fp32 accumulator before the BF16 cast
//               ("H3 Runtime Current State", "Owned Performance Kernels":
//               alpha-before-BF16 epilogue; "Implemented And Validated": fused
//               residual gates).
// or, for FC1 feeding FC2 (kSwiglu; the same section's exact SwiGLU-to-FC2
// producer fusion, which keeps the two BF16 boundaries):
//   out[m][128 t + i] = bf16( silu(g) * u ),  g, u = bf16(alpha * acc + b) of the
//               gate column 256 t + i and the up column 256 t + 128 + i,
// and optionally (kAmax) max |out| over the call, for FC2's one-pass quantisation.
//
// CTA pairs.  The kernel runs as clusters of two CTAs on two SMs; a pair owns
// a 256 x 256 output tile.  CTA r of the pair loads the 128 rows
// [m0 + 128 r, +128) of A and the 128 rows [n0 + 128 r, +128) of W, and the
// leader CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 64): each
// SM's tensor core multiplies its own 128 rows of A by all 256 rows of W,
// fetching the other half of W from its partner.  Compared with one CTA per
// 128 x 256 tile this cuts the bytes each SM pulls from L2 per MMA by 30 %
// (A 4 KB + W 4 KB + scales 1.5 KB instead of 4 + 8 + 1.5 KB).
//
// Block scales reach TMEM through registers.  The MMA reads the scales of
// every row of W from all four TMEM lane quarters, so each quarter holds its
// own copy.  tcgen05.cp (one copy per instruction, ~one instruction per MMA
// duration while MMAs run) cannot keep up with three scale tiles per MMA;
// tcgen05.st from registers writes TMEM at ~190 B/clk without slowing the MMAs.
// So four "scale warps", one per lane quarter, load each stage's 512-byte
// scale tiles from shared memory and store them into their quarter.
//
// Roles (512 threads per CTA in four warpgroups, persistent over pair tiles).
// The producer and the MMA issuer run as whole warps -- every lane takes the
// barrier waits, one elected lane issues -- because a single-lane loop around
// bounded waits measured about 2.2x slower MMA issue (the tensor pipe idles):
//   warp 0      TMA producer (both CTAs): per stage first this CTA's
//               block-scale tiles (on its own "scales landed" barrier), then
//               the A / W code tiles (128-byte swizzle), whose bytes complete
//               on the LEADER's "full" barrier (5-stage ring; 4 with the wide
//               and pack plans).
//   warp 1      TMEM owner (both) + MMA issuer (leader): per stage, one wait
//               on the leader's "full", four paired MMAs, then a commit
//               multicast to both CTAs' "empty" barrier.
//   warps 2-3   (kPack only) packer (both): quantise 128 x 256 units of X
//               into the codes / scales the producer loads, each published by
//               a ready flag the producer acquires before its A loads.
//   warps 4-7   scale warps (both), warp 4 + q serving lane quarter q: per
//               stage, as soon as the CTA's scale tiles landed, twelve 16-byte
//               shared loads per lane, tcgen05.st of 48 columns, then an
//               arrival on the leader's "full" -- overlapping the code tiles'
//               transfer.  "full" therefore completes when both CTAs' code
//               tiles landed (transaction bytes) and all eight scale warps
//               arrived: a single wait per stage in the issuing warp.
//   warps 8-15  epilogue (both): tcgen05.ld the CTA's 128 x 256 fp32
//               accumulator (each warp 32 rows x 128 columns), release it to
//               the leader, then alpha/bias/gate/residual on paired fp32
//               instructions (fma.rn.f32x2, cvt.rn.bf16x2.f32: the epilogue
//               shares issue slots with the producer, MMA and scale warps) and
//               bf16 stores in two passes of two 32x32 chunks, each through two
//               64-byte-swizzled staging buffers and TMA stores; a pass's
//               residual chunks are TMA-loaded into those buffers first (the
//               wide plan stages all four chunks, and the gate and bias, ahead
//               of the accumulator).  SwiGLU: gate and up columns of 32 rows x
//               64 hidden units per warp, one pass.
// Each kernel launch may start while the previous kernel of the stream drains
// (programmatic dependent launch); it reads no input before griddepcontrol.wait.
// Registers per thread (setmaxnreg): warpgroup 0: 40, scale warps: 96,
// epilogue: 184 (with the in-kernel packer 104 / 72 / 168).  Per 128-thread
// warpgroup that is 40 + 96 + 2 x 184 = 504 (104 + 72 + 2 x 168 = 512)
// registers per thread-slot, within the 4 x 128 the CTA is launched with.
//
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>

#include "h3fp4_internal.h"
#include "ptx_sm103.cuh"
#include "nvfp4_encode.cuh"
#include "act_prologue.cuh"

namespace h3fp4 {
namespace {

constexpr int BM = 128;                               // rows of A per CTA (256 per pair)
constexpr int BN = 256;                               // rows of W per pair tile
constexpr int BK = 256;                               // K elements per stage
constexpr int kThreads = 512;
constexpr int kScaleWarp0 = 4;   // warps 4..7: scale warps, lane quarter = warp & 3
constexpr int kEpiWarp0 = 8;     // warps 8..15: epilogue
constexpr int kEpiWarps = 8;
// Registers per thread of each warpgroup (setmaxnreg): control (producer, MMA
// issuer; with the in-kernel packer also the two packer warps), scale warps,
// epilogue.  Each split sums to at most the 4 x 128 registers per thread-slot
// the CTA is launched with.
template <bool kPack>
struct Regs {
    static constexpr uint32_t kCtl = kPack ? 104 : 40;
    static constexpr uint32_t kScale = kPack ? 72 : 96;
    static constexpr uint32_t kEpi = kPack ? 168 : 184;
    static_assert(128 * (kCtl + kScale + 2 * kEpi) <= 65536, "setmaxnreg shares exceed the launch budget");
};
constexpr uint32_t kABytes = BM * BK / 2;             // 16384
constexpr uint32_t kBBytes = (BN / 2) * BK / 2;       // 16384: this CTA's half of W
constexpr uint32_t kSFABytes = BM * (BK / 16);        // 2048: four 512-byte tiles
constexpr uint32_t kSFBBytes = BN * (BK / 16);        // 4096: both halves, four tiles each
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;  // 38912
constexpr uint32_t kPairTxBytes = 2 * (kABytes + kBBytes);  // both CTAs' code tiles complete on the leader
constexpr uint32_t kSfBox = 2048;                     // scale-tile TMA box: 8 rows x 256 bytes
constexpr uint32_t kChunkBytes = 32 * 32 * 2;         // 32 rows x 32 bf16
constexpr uint32_t kXTileBytes = 32 * BK * 2;         // packer: 32 rows x 256 bf16 of X per TMA box
constexpr uint32_t kPackThreads = 64;                 // packer: warps 2 and 3
constexpr uint32_t kPackBar = 2;                      // packer: named barrier id
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmem = 256;
constexpr uint32_t kSfTmemPerStage = 48;
static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");

// Ring depth and epilogue staging.  The default plan keeps five stages in
// flight and two 32x32 staging chunks per epilogue warp, so a gated epilogue
// loads its second pass's residual only after the first pass's stores have
// read the chunks.  The wide plan (gated residual epilogue over a short K
// loop, where that epilogue is longer than a tile's mainloop) gives up one
// stage for four chunks per warp: the whole tile's residual is loaded ahead
// of the accumulator, and the epilogue runs in one pass.  The pack plan (the
// GEMM quantises its own activation) gives up one stage for two 16 KB X tiles
// of the packer.
// K stages per tile below which a gated residual epilogue takes the wide plan.
constexpr int kWideMaxKStages = 24;
static_assert(kXTileBytes % 1024 == 0, "X tiles keep the 1024-byte alignment");

template <bool kWide, bool kPack>
struct Plan {
    static_assert(!(kWide && kPack), "one plan at a time");
    static constexpr int kStages = (kWide || kPack) ? 4 : 5;
    static constexpr int kChunks = kWide ? 4 : 2;               // staging chunks per epilogue warp
    static constexpr uint32_t kEpiWarpBytes = kChunks * kChunkBytes;
    static constexpr uint32_t kEpiOff = kStages * kStageBytes;
    static constexpr uint32_t kXOff = kEpiOff + kEpiWarps * kEpiWarpBytes;  // kPack: two X tiles
    static constexpr uint32_t kBarOff = kXOff + (kPack ? 2 * kXTileBytes : 0);
    // barriers (full, empty, sf_full per stage; acc_full, acc_empty, done, one
    // per epilogue warp; x_full x 2, sg_ready), TMEM address, abort flag,
    // global scale of the packed activation, packer reduction slots
    static constexpr uint32_t kBarBytes = 8 * (3 * kStages + 3 + kEpiWarps + 3) + 8 + 16;
    static constexpr uint32_t kRcpOff = kBarOff + 512;          // kNvfp4: 128 fp32 block reciprocals of h;
                                                                // kPack: of the packed activation
    // kWide: per epilogue warp the gate of its 128 columns for two segments
    // (fp32, 1 KB) and their bias (bf16, 256 B), staged before the accumulator
    // wait so that the epilogue -- the wide plan's critical path -- reads them
    // from shared memory instead of waiting on global loads
    static constexpr uint32_t kGateOff = kRcpOff + 512;
    static constexpr uint32_t kBiasOff = kGateOff + (kWide ? kEpiWarps * 1024 : 0);
    static constexpr uint32_t kSmemBytes = kBiasOff + (kWide ? kEpiWarps * 256 : 0);
    static_assert(kBarBytes <= 512, "barrier block");
    static_assert(kSfTmem + kStages * kSfTmemPerStage <= kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};
static_assert(kSFABytes == kSfBox && kSFBBytes == 2 * kSfBox, "scale tiles move in 2 KB boxes");

// Instruction descriptor, kind::mxf4nvf4: A/B E2M1 (1) in bits 7-9 / 10-12,
// K-major A and B, N >> 3 in bits 17-22, UE4M3 scales (bit 23 = 0),
// M >> 4 in bits 24-28 (M = 256: the pair), scale-factor ids 0, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(2 * BM >> 4) << 24);

struct GemmParams {
    const float* a_gscale;
    const float* w_gscale;
    const __nv_bfloat16* bias;
    const float* gate;
    int M, N, K;
    int m_tiles, n_tiles, pair_m_tiles, k_stages, kb4;
    int has_resid;
    Segments seg;
    unsigned int* status;
    unsigned long long wait_ns;
    int stall;  // self-test: 1 = the producer issues nothing, so every consumer wait must time out;
                //            2 = (kPack) the packer publishes no tile, so the producer's flag waits time out
    float* amax_out;  // kAmax: atomic max of |out| (bf16 values, as fp32 bits) over the call
    // kNvfp4: h written as NVFP4 under the caller's global scale of h
    uint8_t* h_codes;      // [M][N/4] bytes
    uint8_t* h_sf;         // block scales of h, 128x4-tiled, sf_bytes(M, N/2)
    const float* h_gscale; // device fp32
    int h_kb4;             // N/2/64 scale groups per row of h
    // kPack: the activation quantised in-kernel (X bf16 [M][K] through tmX)
    const float* pk_shift;    // [nseg][K] or null: the modulation prologue
    const float* pk_scale;
    uint8_t* pk_codes;        // out: [M][K/2] (what tmA reads)
    uint8_t* pk_sf;           // out: block scales, 128x4-tiled (what tmSFA reads)
    float* pk_gscale;         // in if pk_given, else out (written by CTA 0)
    const float* pk_partials; // amax partials of the preceding amax pass
    int pk_nparts;
    int pk_given;
    uint32_t* pk_flags;       // [m_tiles][k_stages] ready flags
    uint32_t pk_epoch;        // the value a ready flag holds in this launch
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

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// kPack: waits (bounded by limit_ns, or until the pair aborts) until *flag holds
// v; acquire, so the tile the flag publishes is visible afterwards.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t v, uint64_t limit_ns, unsigned int* err,
                                          volatile int& abort)
{
    if (ld_acquire_gpu_u32(flag) == v) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(128);
        if (ld_acquire_gpu_u32(flag) == v) return true;
        if (abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, kStatusTimeoutPackFlag);
            return false;
        }
    }
}

// silu(g) = g * sigmoid(g) in fp32.  With t = 2^(-|g| log2 e) in (0, 1],
// sigmoid(g) = 1 / (1 + t) for g >= 0 and t / (1 + t) for g < 0, so no step
// overflows for any g (e^-g itself overflows fp32 below g = -88.7).  Over every
// finite bf16 g the result is within 3.4e-6 relative of the exact silu for
// |g| < 88, and bf16(result) within one bf16 step of the correctly rounded value.
__device__ __forceinline__ float silu_f32(float g)
{
    const float t = ex2_approx(-fabsf(g) * 1.4426950408889634f);
    const float r = rcp_approx(1.0f + t);
    return g * (g >= 0.0f ? r : t * r);
}

// kSwiglu: SwiGLU epilogue (out [M][N/2]); kAmax: track max |out| into p.amax_out;
// kNvfp4 (with kSwiglu): h is not stored in bf16 but quantised to NVFP4 under the
// given global scale of h, with the quantiser's arithmetic (nvfp4_encode.cuh).
// Compile-time, so that the plain epilogue carries none of them.  kWide: the
// wide plan (Plan above; gated residual epilogue only).  kPack: the kernel
// quantises its activation itself (packer warps, below) instead of reading
// codes a separate quantiser wrote.
template <bool kSwiglu, bool kAmax, bool kNvfp4, bool kWide, bool kPack>
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                      const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmR,
                      const __grid_constant__ CUtensorMap tmX, const GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    static_assert(!kWide || !kSwiglu, "the wide plan is for the gated residual epilogue");
    static_assert(!kPack || (!kSwiglu && !kNvfp4), "the in-kernel packer serves the plain and gated epilogues");
    using P = Plan<kWide, kPack>;
    using R = Regs<kPack>;
    constexpr int kStages = P::kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Swizzled TMA tiles need 1024-byte alignment; refuse to run otherwise.  Both
    // CTAs of a pair have the same layout, so both leave here together.
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSmemAlign);
        return;
    }

    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs)
    const bool leader = rank == 0;
    // Leader's "full": both CTAs' code tiles landed (tx bytes) AND the eight
    // scale warps of the pair stored the stage's scales in TMEM (arrivals), so
    // one wait clears a stage for the MMAs.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::kBarOff);
    uint64_t* empty = full + kStages;                                // both: the MMAs released the stage
    uint64_t* sf_full = empty + kStages;                             // both: this CTA's scale tiles landed
    uint64_t* acc_full = sf_full + kStages;                          // both: accumulator complete
    uint64_t* acc_empty = acc_full + 1;                              // leader's: both epilogues drained
    uint64_t* rbar = acc_empty + 1;                                  // one per epilogue warp
    uint64_t* done_bar = rbar + kEpiWarps;
    uint64_t* x_full = done_bar + 1;                                 // kPack: the packer's two X tiles landed
    uint64_t* sg_ready = x_full + 2;                                 // kPack: s_gscale holds the activation scale
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sg_ready + 1);
    volatile int& s_abort = *reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* s_gscale = reinterpret_cast<float*>(tmem_slot + 2);
    float* s_red = s_gscale + 1;                                     // kPack: the packer warps' partial maxima

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1 + 2 * 4);  // the producer's expect_tx + four scale warps per CTA
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kEpiWarps);
        for (int e = 0; e < kEpiWarps; ++e) mbar_init(&rbar[e], 1);
        mbar_init(done_bar, 1);
        if (kPack) {
            mbar_init(&x_full[0], 1);
            mbar_init(&x_full[1], 1);
            mbar_init(sg_ready, 1);
        }
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmSFA);
        prefetch_tensormap(&tmSFB);
        prefetch_tensormap(&tmOut);
        if (p.has_resid) prefetch_tensormap(&tmR);
        if (kPack) prefetch_tensormap(&tmX);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc_fence_after();
    // Everything above overlaps the previous kernel's tail (programmatic
    // dependent launch); the operands, scales and global scales it may have
    // produced are read only after this.
    griddep_wait();
    const uint32_t tmem = *tmem_slot;
    const int num_tiles = p.pair_m_tiles * p.n_tiles;
    // A timeout anywhere stops both CTAs of the pair.
    auto set_abort = [&]() {
        s_abort = 1;
        st_shared_cluster_u32(mapa_shared(smem_u32((const void*)&s_abort), cluster_ctarank() ^ 1u), 1u);
    };

    if (warp < kScaleWarp0) {
        setmaxnreg_dec<R::kCtl>();
        // The producer and the MMA issuer run as whole warps: every lane takes
        // the barrier waits (decided warp-wide), one elected lane issues the
        // copies / MMAs.  A single-lane loop around bounded waits measured far
        // slower MMA issue (the tensor pipe then idles between MMAs).
        if (warp == 0) {
            // ------------------------------------------------------------ producer (both CTAs)
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t fills[kStages] = {};
            for (int tile = blockIdx.x >> 1; tile < num_tiles && p.stall != 1; tile += gridDim.x >> 1) {
                if (__any_sync(0xffffffffu, s_abort != 0)) break;  // warp-uniform exit
                const int mp = tile / p.n_tiles, nt = tile - mp * p.n_tiles;
                const int mt = 2 * mp + (int)rank;  // this CTA's 128-row tile of A
                bool ok = true;
                // kPack: bit kb set once the packer published unit (mt, kb) (k_stages <= 64).
                uint64_t rdy = ~0ull;
                const uint32_t* flags = kPack ? p.pk_flags + (size_t)mt * (size_t)p.k_stages : nullptr;
                auto poll = [&]() {
                    uint64_t m = 0;
                    for (int base = 0; base < p.k_stages; base += 32) {
                        const int k = base + lane;
                        const bool r = k < p.k_stages && ld_acquire_gpu_u32(flags + k) == p.pk_epoch;
                        m |= (uint64_t)__ballot_sync(0xffffffffu, r) << base;
                    }
                    return m;
                };
                if (kPack && mt < p.m_tiles) rdy = poll();
                for (int kb = 0; kb < p.k_stages; ++kb) {
                    ok = mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns, p.status, kStatusTimeoutProducer);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kPack) {
                        if (!((rdy >> kb) & 1ull)) {
                            int r = 1;
                            if (lane == 0) r = wait_flag(flags + kb, p.pk_epoch, p.wait_ns, p.status, s_abort) ? 1 : 0;
                            if (!__shfl_sync(0xffffffffu, r, 0)) {
                                ok = false;
                                break;
                            }
                            rdy = poll() | (1ull << kb);
                        }
                        fence_proxy_async_global();  // the published codes and scales, before the TMA reads them
                    }
                    if (elect_one()) {
                        uint8_t* st = smem + stage * kStageBytes;
                        // Scale tiles first (as rows of 256 bytes; a 512-byte tile is
                        // two rows): the scale warps move them into TMEM while the
                        // code tiles are still arriving.
                        mbar_arrive_expect_tx(&sf_full[stage], kSFABytes + kSFBBytes);
                        uint8_t* sf = st + kABytes + kBBytes;
                        tma_load_2d(sf, &tmSFA, &sf_full[stage], 0, (mt * p.kb4 + kb * 4) * 2);
                        tma_load_2d(sf + kSFABytes, &tmSFB, &sf_full[stage], 0, ((2 * nt) * p.kb4 + kb * 4) * 2);
                        tma_load_2d(sf + kSFABytes + kSfBox, &tmSFB, &sf_full[stage], 0,
                                    ((2 * nt + 1) * p.kb4 + kb * 4) * 2);
                        const uint32_t bar = full_leader + 8u * (uint32_t)stage;
                        if (leader) mbar_arrive_expect_tx(&full[stage], kPairTxBytes);
                        tma_load_2d_pair(st, &tmA, bar, kb * (BK / 2), mt * BM);
                        tma_load_2d_pair(st + kABytes, &tmB, bar, kb * (BK / 2), nt * BN + (int)rank * (BN / 2));
                    }
                    __syncwarp();
                    ++fills[stage];
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    if (lane == 0) set_abort();
                    break;
                }
            }
            // Drain: every copy into either CTA must land before the pair may exit.
            // The leader's "full" phase of a fill completes only when both CTAs'
            // code tiles arrived; the last fill of stage s completes phase fills[s] - 1.
            for (int s = 0; s < kStages; ++s)
                if (fills[s] > 0) {
                    if (leader)
                        (void)mbar_wait(&full[s], (fills[s] - 1u) & 1u, p.wait_ns, p.status, kStatusTimeoutProducer);
                    (void)mbar_wait(&sf_full[s], (fills[s] - 1u) & 1u, p.wait_ns, p.status, kStatusTimeoutProducer);
                }
            __syncwarp();
        } else if (warp == 1 && leader) {
            // ------------------------------------------------------------ MMA issuer (leader)
            const uint32_t smem_base = smem_u32(smem);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x >> 1; tile < num_tiles; tile += gridDim.x >> 1) {
                if (__any_sync(0xffffffffu, s_abort != 0)) break;  // warp-uniform exit
                bool ok = mbar_wait(acc_empty, acc_phase ^ 1u, p.wait_ns, p.status, kStatusTimeoutMma);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) set_abort();
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < p.k_stages; ++kb) {
                    // Both CTAs' code tiles in shared memory, both CTAs' scales in TMEM.
                    ok = mbar_wait(&full[stage], phase, p.wait_ns, p.status, kStatusTimeoutMma);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, p.kb4 - kb * 4);
                    const uint32_t st = smem_base + (uint32_t)stage * kStageBytes;
                    // K group j of the stage starts 32 bytes further into each
                    // 128-byte swizzled row: +2 in the descriptors' address field.
                    const uint64_t adesc = smem_desc(st, 16, 1024, 2);
                    const uint64_t bdesc = smem_desc(st + kABytes, 16, 1024, 2);
                    const uint32_t sfa_t = tmem + kSfTmem + (uint32_t)stage * kSfTmemPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    if (elect_one()) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j < nk)
                                mma_pair_mxf4nvf4(tmem, adesc + 2u * j, bdesc + 2u * j, kIdesc, sfa_t + 4u * j,
                                                  sfb_t + 8u * j, (kb > 0 || j > 0) ? 1u : 0u);
                        tc_commit_pair_mc(&empty[stage], 3);
                    }
                    __syncwarp();
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    if (lane == 0) set_abort();
                    break;
                }
                if (elect_one()) tc_commit_pair_mc(acc_full, 3);
                __syncwarp();
                acc_phase ^= 1u;
            }
            // Every issued MMA must finish before TMEM is released.
            if (elect_one()) tc_commit_pair(done_bar);
            __syncwarp();
            (void)mbar_wait(done_bar, 0u, p.wait_ns, p.status, kStatusTimeoutMma);
            __syncwarp();
        } else if (kPack && warp >= 2) {
            // ------------------------------------------------------------ packer (both CTAs, kPack)
            // Quantises the activation once, in units of one 128-row m-tile x one
            // 256-column k-stage, with the quantiser's arithmetic (act_prologue.cuh,
            // nvfp4_encode.cuh): same codes, block scales and global scale.  Each
            // unit is published by a release store of its ready flag, which the
            // producers of every CTA consuming that m-tile acquire before their
            // TMA loads.  Units go to CTAs round-robin in the order the persistent
            // schedule first needs them.  X comes in 32-row TMA tiles, two in flight.
            const int pt = (int)threadIdx.x - 64;  // 0..63
            float* a_rcp = reinterpret_cast<float*>(smem + P::kRcpOff);
            float s_g;
            if (p.pk_given) {
                s_g = *p.pk_gscale;
            } else {
                // one full-activation amax over the amax pass's partials
                float m = 0.0f;
                for (int i = pt; i < p.pk_nparts; i += (int)kPackThreads) m = fmaxf(m, p.pk_partials[i]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if (lane == 0) s_red[warp - 2] = m;
                named_bar_sync(kPackBar, kPackThreads);
                const float amax = fmaxf(s_red[0], s_red[1]);
                s_g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
                if (blockIdx.x == 0 && pt == 0) *p.pk_gscale = s_g;
            }
            for (int c = pt; c < 128; c += (int)kPackThreads) a_rcp[c] = block_rcp((uint32_t)c, s_g);
            named_bar_sync(kPackBar, kPackThreads);
            if (pt == 0) {
                *s_gscale = s_g;
                mbar_arrive(sg_ready);  // the epilogue's alpha
            }

            const int ks = p.k_stages, mtiles = p.m_tiles;
            const long long nunits = (long long)mtiles * ks;
            const long long pairs = gridDim.x >> 1;
            const long long K = p.K;
            const bool mod = p.pk_shift != nullptr;
            // First m-tile of group g: pair mp first appears in tile mp * n_tiles,
            // i.e. in round mp * n_tiles / pairs of the persistent schedule.
            auto group_first = [&](long long g) -> long long {
                const long long mp = (g * pairs + p.n_tiles - 1) / p.n_tiles;
                return min(2 * mp, (long long)mtiles);
            };
            long long grp = 0;
            auto coords = [&](long long o, int& mt, int& kb) {
                while (o >= group_first(grp + 1) * ks) ++grp;
                const long long f = group_first(grp);
                const long long nm = group_first(grp + 1) - f;
                const long long rel = o - f * ks;
                kb = (int)(rel / nm);
                mt = (int)(f + rel % nm);
            };
            const long long my_units =
                (long long)blockIdx.x < nunits ? (nunits - 1 - (long long)blockIdx.x) / gridDim.x + 1 : 0;
            const long long T = 4 * my_units;  // jobs: 32-row X tiles
            const int bc = pt & 15;            // this thread's 16-column block of a unit
            const int rq = pt >> 4;            // its first row in an X tile (then every fourth)
            ModCols mc;
            init_mod(mc);
            long long mc_cb = -1;
            int cur_mt = 0, cur_kb = 0, nxt_mt = 0, nxt_kb = 0;
            auto issue = [&](long long t, int mt, int kb) {
                const int b = (int)(t & 1);
                mbar_arrive_expect_tx(&x_full[b], kXTileBytes);
                tma_load_2d(smem + P::kXOff + b * kXTileBytes, &tmX, &x_full[b], kb * BK,
                            mt * BM + 32 * (int)(t & 3));
            };
            long long issued = 0, landed = 0;
            if (T > 0) {
                coords((long long)blockIdx.x, cur_mt, cur_kb);
                if (pt == 0) issue(0, cur_mt, cur_kb);
                issued = 1;
            }
            bool ok = true;
            for (long long t = 0; t < T; ++t) {
                // the next tile into the other buffer (its readers passed the barrier
                // that ended the previous job)
                if (t + 1 < T) {
                    if (((t + 1) & 3) == 0)
                        coords((long long)blockIdx.x + ((t + 1) >> 2) * gridDim.x, nxt_mt, nxt_kb);
                    else {
                        nxt_mt = cur_mt;
                        nxt_kb = cur_kb;
                    }
                    if (pt == 0) issue(t + 1, nxt_mt, nxt_kb);
                    ++issued;
                }
                const int b = (int)(t & 1);
                bool got = mbar_wait(&x_full[b], (uint32_t)(t >> 1) & 1u, p.wait_ns, p.status, kStatusTimeoutPacker);
                // one decision for all 64 packer threads (they share named barriers)
                if (!named_bar_and(kPackBar, kPackThreads, got && s_abort == 0)) {
                    ok = false;
                    landed = got ? t + 1 : t;
                    break;
                }
                landed = t + 1;
                const uint8_t* xt = smem + P::kXOff + b * kXTileBytes;
                const long long row0 = (long long)cur_mt * BM + 32 * (t & 3);
                const long long cb = (long long)cur_kb * 16 + bc;  // 16-column block index in the row
                const bool colv = cb < K / 16;
                if (mod && colv && cb != mc_cb) {
                    mc_cb = cb;
                    mc.seg_end = -1;  // reload the constants of the new column block
                }
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    const int rl = rq + 4 * j;
                    const long long row = row0 + rl;
                    const bool real = row < p.M;
                    const uint32_t xa = smem_u32(xt) + (uint32_t)rl * (BK * 2) + (uint32_t)bc * 32u;
                    const uint4 v0 = ld_shared_v4(xa), v1 = ld_shared_v4(xa + 16u);
                    V16 v;
                    v.w[0] = v0.x; v.w[1] = v0.y; v.w[2] = v0.z; v.w[3] = v0.w;
                    v.w[4] = v1.x; v.w[5] = v1.y; v.w[6] = v1.z; v.w[7] = v1.w;
                    float f[16];
                    unpack16(v, f);
                    if (mod && real && colv) {
                        if (row >= mc.seg_end || row < mc.seg_begin)
                            load_mod(p.pk_scale, p.pk_shift, K, p.seg, segment_of(p.seg, row), cb, mc);
                        modulate16<true>(f, mc);
                    }
                    float bmax = 0.0f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(f[i]));
                    const uint32_t S = real ? block_scale_code(bmax, s_g) : 0u;  // padding rows: zero scales
                    const float rcp = a_rcp[S & 127u];
                    const uint64_t rcp2 = f2(rcp, rcp);
                    float q[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) unf2(mul2(f2(f[2 * i], f[2 * i + 1]), rcp2), q[2 * i], q[2 * i + 1]);
                    const uint32_t w0 = e2m1x8(reinterpret_cast<const float(&)[8]>(q[0]));
                    const uint32_t w1 = e2m1x8(reinterpret_cast<const float(&)[8]>(q[8]));
                    if (real && colv)
                        *reinterpret_cast<uint2*>(p.pk_codes + row * (K / 2) + cb * 8) = make_uint2(w0, w1);
                    // the four block scales of a 64-column group into its first lane
                    const uint32_t s1 = __shfl_down_sync(0xffffffffu, S, 1);
                    const uint32_t s2 = __shfl_down_sync(0xffffffffu, S, 2);
                    const uint32_t s3 = __shfl_down_sync(0xffffffffu, S, 3);
                    if (colv && (bc & 3) == 0) {
                        const long long g = cb >> 2;
                        const uint32_t r7 = (uint32_t)row & 127u;
                        const long long off = (((row >> 7) * p.kb4 + g) << 9) + ((r7 & 31u) << 4) + ((r7 >> 5) << 2);
                        *reinterpret_cast<uint32_t*>(p.pk_sf + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
                    }
                }
                const bool last = (t & 3) == 3;
                fence_proxy_async_smem();  // this job's reads of the X tile, before its refill
                if (last) {
                    fence_proxy_async_global();  // the unit's codes and scales, for TMA readers
                    __threadfence();
                }
                named_bar_sync(kPackBar, kPackThreads);
                if (last && pt == 0 && p.stall != 2)
                    st_release_gpu_u32(p.pk_flags + (size_t)cur_mt * (size_t)ks + cur_kb, p.pk_epoch);
                cur_mt = nxt_mt;
                cur_kb = nxt_kb;
            }
            if (!ok) {
                if (pt == 0) set_abort();
                // tiles still in flight must land before the CTA may exit
                for (long long t = landed; t < issued; ++t)
                    (void)mbar_wait(&x_full[t & 1], (uint32_t)(t >> 1) & 1u, p.wait_ns, p.status, kStatusTimeoutPacker);
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------------------- scale warps (both CTAs)
        // Lane i of the warp for quarter q writes TMEM lane 32 q + i: columns
        // [sfa_t + 4 j, +4) <- bytes [16 i, 16 i + 16) of A's scale tile for K group j,
        // columns [sfb_t + 8 j + 4 h, +4) <- the same bytes of W's tile (half h, group j)
        // -- the TMEM image the MMA reads (each quarter a full copy).
        // The TMEM slot of a stage is rewritten only after the stage was refilled,
        // i.e. after the MMAs that read the previous contents committed.
        setmaxnreg_dec<R::kScale>();
        const uint32_t q = (uint32_t)(warp & 3);
        const uint32_t ready_leader = mapa_shared(smem_u32(full), 0);
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x >> 1; tile < num_tiles; tile += gridDim.x >> 1) {
            bool ok = true;
            for (int kb = 0; kb < p.k_stages; ++kb) {
                if (__any_sync(0xffffffffu, s_abort != 0)) {
                    ok = false;
                    break;
                }
                ok = mbar_wait(&sf_full[stage], phase, p.wait_ns, p.status, kStatusTimeoutMma);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const uint32_t sfa_s = smem_u32(smem + stage * kStageBytes + kABytes + kBBytes) + 16u * (uint32_t)lane;
                const uint32_t sfb_s = sfa_s + kSFABytes;
                uint32_t va[16], vb[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = ld_shared_v4(sfa_s + 512u * j);
                    va[4 * j] = a.x;
                    va[4 * j + 1] = a.y;
                    va[4 * j + 2] = a.z;
                    va[4 * j + 3] = a.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 b = ld_shared_v4(sfb_s + kSfBox * h + 512u * j);
                        vb[8 * j + 4 * h] = b.x;
                        vb[8 * j + 4 * h + 1] = b.y;
                        vb[8 * j + 4 * h + 2] = b.z;
                        vb[8 * j + 4 * h + 3] = b.w;
                    }
                }
                const uint32_t sfa_t = tmem + ((32u * q) << 16) + kSfTmem + stage * kSfTmemPerStage;
                tc_st_32x32b_x16(sfa_t, va);
                tc_st_32x32b_x32(sfa_t + 16, vb);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(ready_leader + 8u * (uint32_t)stage);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                if (lane == 0) set_abort();
                break;
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        setmaxnreg_inc<R::kEpi>();
        const int e = warp - kEpiWarp0;    // 0..7
        float* rcp_tab = reinterpret_cast<float*>(smem + P::kRcpOff);
        if constexpr (kNvfp4) {
            // The reciprocal of every possible block scale of h (the same values
            // the quantiser uses), shared by the eight epilogue warps.
            const float s_h = __ldg(p.h_gscale);
            const int t = (int)threadIdx.x - kEpiWarp0 * 32;
            if (t < 128) rcp_tab[t] = block_rcp((uint32_t)t, s_h);
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        }
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int h = e >> 2;              // column half of the 256-wide tile
        uint8_t* stg = smem + P::kEpiOff + e * P::kEpiWarpBytes;
        float a_s;
        if constexpr (kPack) {
            // the packer's global scale of the activation (it may be computing it in this launch)
            a_s = mbar_wait(sg_ready, 0u, p.wait_ns, p.status, kStatusTimeoutEpilogue) ? *s_gscale : 0.0f;
        } else {
            a_s = __ldg(p.a_gscale);
        }
        const float alpha = __fmul_rn(a_s, __ldg(p.w_gscale));
        const uint64_t alpha2 = f2(alpha, alpha);
        uint32_t acc_phase = 0, r_phase = 0;
        bool r_pending = false;
        float omax = 0.0f;  // max |out| over this lane's rows < M (before the bf16 rounding)
        for (int tile = blockIdx.x >> 1; tile < num_tiles; tile += gridDim.x >> 1) {
            if (__any_sync(0xffffffffu, s_abort != 0)) break;  // warp-uniform exit
            const int mp = tile / p.n_tiles, nt = tile - mp * p.n_tiles;
            // (blockIdx.x & 1 is the CTA's rank in its pair)
            const int m0 = (2 * mp + (int)(blockIdx.x & 1u)) * BM + 32 * q;  // first row of this warp
            const int nc0 = nt * BN + 128 * h;                                 // first column of this warp
            // Two passes of two 32x32 chunks through the warp's staging chunks;
            // the residual chunks of a pass are TMA-loaded into them first (pass 0
            // ahead of the accumulator; with the wide plan all four chunks).
            if (lane == 0) bulk_wait_read_all();  // staging buffers free again
            __syncwarp();
            if (p.has_resid && lane == 0) {
                mbar_arrive_expect_tx(&rbar[e], P::kChunks * kChunkBytes);
                for (int c = 0; c < P::kChunks; ++c)
                    tma_load_2d(stg + c * kChunkBytes, &tmR, &rbar[e], nc0 + 32 * c, m0);
            }
            r_pending = p.has_resid != 0;
            // kWide: the gate of this warp's 128 columns for the segments of its
            // first and last rows, staged in shared memory before the accumulator
            // wait (lanes in a third segment read it from global memory)
            int seg_a = 0, seg_b = 0;
            float* gst = reinterpret_cast<float*>(smem + P::kGateOff + 1024u * (uint32_t)e);
            if (kWide && p.gate != nullptr) {
                seg_a = segment_of_row(p.seg, min(m0, p.M - 1));
                seg_b = segment_of_row(p.seg, min(m0 + 31, p.M - 1));
                const int col = nc0 + 4 * lane;
                float4 ga = make_float4(1.0f, 1.0f, 1.0f, 1.0f), gb = ga;
                if (col < p.N) {
                    ga = __ldg(reinterpret_cast<const float4*>(p.gate + (size_t)seg_a * p.N + col));
                    gb = __ldg(reinterpret_cast<const float4*>(p.gate + (size_t)seg_b * p.N + col));
                }
                reinterpret_cast<float4*>(gst)[lane] = ga;
                reinterpret_cast<float4*>(gst + 128)[lane] = gb;
                __syncwarp();
            }
            uint8_t* bst = smem + P::kBiasOff + 256u * (uint32_t)e;  // kWide: the bias of the warp's 128 columns
            if (kWide && p.bias != nullptr) {
                const int col = nc0 + 4 * lane;
                uint2 bv = make_uint2(0u, 0u);
                if (col < p.N) bv = __ldg(reinterpret_cast<const uint2*>(p.bias + col));
                reinterpret_cast<uint2*>(bst)[lane] = bv;
                __syncwarp();
            }
            bool ok = mbar_wait(acc_full, acc_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) set_abort();
                break;
            }
            acc_phase ^= 1u;
            tc_fence_after();
            uint32_t acc[4][32];
            // Plain: this warp's columns [128 h, +128) in acc[0..3].  SwiGLU: the
            // gate columns [64 h, +64) in acc[0..1] and the matching up columns
            // [128 + 64 h, +64) in acc[2..3].
            const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t col = kSwiglu ? 64u * h + 128u * (c >> 1) + 32u * (c & 1) : 128u * h + 32u * c;
                tc_ld_32x32b_x32(tq + col, acc[c]);
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty), 0));  // accumulator free

            const int row = m0 + lane;
            const float* grow = nullptr;
            const float* gsm = nullptr;  // kWide: this lane's staged gate row
            if (p.gate != nullptr && row < p.M) {
                const int sg = segment_of_row(p.seg, row);
                grow = p.gate + (size_t)sg * p.N;
                if (kWide) gsm = sg == seg_a ? gst : (sg == seg_b ? gst + 128 : nullptr);
            }
            bool failed = false;
            uint32_t hcode[8];       // kNvfp4: this row's 64 values of h as 32 bytes of codes
            uint32_t hscale = 0u;    // kNvfp4: its four block-scale codes
            const float s_h_reg = kNvfp4 ? __ldg(p.h_gscale) : 0.0f;
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                if (pass == 1 && kSwiglu) break;  // 64 output columns per warp: one pass
                if (pass == 1 && !kWide) {
                    if (lane == 0) bulk_wait_read_all();  // pass 0's stores have read the buffers
                    __syncwarp();
                    if (p.has_resid && lane == 0) {
                        mbar_arrive_expect_tx(&rbar[e], 2 * kChunkBytes);
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d(stg + c * kChunkBytes, &tmR, &rbar[e], nc0 + 64 + 32 * c, m0);
                    }
                    r_pending = p.has_resid != 0;
                }
                if (p.has_resid && (pass == 0 || !kWide)) {
                    ok = mbar_wait(&rbar[e], r_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
                    if (!__all_sync(0xffffffffu, ok)) {
                        failed = true;
                        break;
                    }
                    r_phase ^= 1u;
                    r_pending = false;
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * pass + cc;
                    uint8_t* buf = stg + (kWide ? c : cc) * kChunkBytes;
                    if constexpr (kSwiglu) {
                        // g, u = the plain epilogue's values rounded to bf16 (the FC1
                        // output boundary); h = bf16(silu(g) * u) in fp32.
                        const int ng = nt * BN + 64 * h + 32 * cc;  // gate column of the chunk (up: + 128)
                        float hv[32];  // kNvfp4: the chunk's 32 values of h, bf16-rounded
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float bg[8], bu[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                bg[i] = 0.0f;
                                bu[i] = 0.0f;
                            }
                            if (p.bias != nullptr) {
                                const uint4 gv = __ldg(reinterpret_cast<const uint4*>(p.bias + ng + 8 * j));
                                const uint4 uv = __ldg(reinterpret_cast<const uint4*>(p.bias + ng + 128 + 8 * j));
                                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    bg[2 * i] = __uint_as_float(gw[i] << 16);
                                    bg[2 * i + 1] = __uint_as_float(gw[i] & 0xFFFF0000u);
                                    bu[2 * i] = __uint_as_float(uw[i] << 16);
                                    bu[2 * i + 1] = __uint_as_float(uw[i] & 0xFFFF0000u);
                                }
                            }
                            float o[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                // g, u exactly as the plain epilogue stores them (alpha*acc + b, one rounding, then bf16)
                                const uint32_t gw = cvt_bf16x2(fma2(
                                    f2(__uint_as_float(acc[cc][8 * j + 2 * i]), __uint_as_float(acc[cc][8 * j + 2 * i + 1])),
                                    alpha2, f2(bg[2 * i], bg[2 * i + 1])));
                                const uint32_t uw = cvt_bf16x2(fma2(
                                    f2(__uint_as_float(acc[2 + cc][8 * j + 2 * i]),
                                       __uint_as_float(acc[2 + cc][8 * j + 2 * i + 1])),
                                    alpha2, f2(bu[2 * i], bu[2 * i + 1])));
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    const float g = k ? __uint_as_float(gw & 0xFFFF0000u) : __uint_as_float(gw << 16);
                                    const float u = k ? __uint_as_float(uw & 0xFFFF0000u) : __uint_as_float(uw << 16);
                                    o[2 * i + k] = __fmul_rn(silu_f32(g), u);
                                    if (kAmax && row < p.M) omax = fmaxf(omax, fabsf(o[2 * i + k]));
                                }
                            }
                            const uint32_t hw[4] = {cvt_bf16x2(f2(o[0], o[1])), cvt_bf16x2(f2(o[2], o[3])),
                                                    cvt_bf16x2(f2(o[4], o[5])), cvt_bf16x2(f2(o[6], o[7]))};
                            if constexpr (kNvfp4) {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    hv[8 * j + 2 * i] = __uint_as_float(hw[i] << 16);
                                    hv[8 * j + 2 * i + 1] = __uint_as_float(hw[i] & 0xFFFF0000u);
                                }
                            } else {
                                *reinterpret_cast<uint4*>(buf + swz64(lane, j)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            }
                        }
                        if constexpr (kNvfp4) {
                            // Two 16-value blocks of this row: block scale, codes.
#pragma unroll
                            for (int b = 0; b < 2; ++b) {
                                float bmax = 0.0f;
#pragma unroll
                                for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(hv[16 * b + i]));
                                const uint32_t S = block_scale_code(bmax, s_h_reg);
                                const uint64_t r2 = f2(rcp_tab[S & 127u], rcp_tab[S & 127u]);
                                float qv[16];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    unf2(mul2(f2(hv[16 * b + 2 * i], hv[16 * b + 2 * i + 1]), r2), qv[2 * i], qv[2 * i + 1]);
                                hcode[4 * cc + 2 * b] = e2m1x8(reinterpret_cast<const float(&)[8]>(qv[0]));
                                hcode[4 * cc + 2 * b + 1] = e2m1x8(reinterpret_cast<const float(&)[8]>(qv[8]));
                                hscale |= S << (8 * (2 * cc + b));
                            }
                            continue;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tma_store_2d(&tmOut, buf, nt * (BN / 2) + 64 * h + 32 * cc, m0);
                        continue;
                    } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int n8 = nc0 + 32 * c + 8 * j;
                        // Lane pairs through the paired fp32 instructions (each lane
                        // rounds like the scalar op): y = alpha*acc + b in one fma, then
                        // out = g*y + R in one fma with the residual gate.
                        uint64_t y2[4];
                        {
                            uint32_t bw[4] = {0u, 0u, 0u, 0u};
                            if (kWide && p.bias != nullptr) {
                                const uint4 bv = reinterpret_cast<const uint4*>(bst)[4 * c + j];
                                bw[0] = bv.x; bw[1] = bv.y; bw[2] = bv.z; bw[3] = bv.w;
                            } else if (n8 < p.N && p.bias != nullptr) {
                                const uint4 bv = __ldg(reinterpret_cast<const uint4*>(p.bias + n8));
                                bw[0] = bv.x; bw[1] = bv.y; bw[2] = bv.z; bw[3] = bv.w;
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                y2[i] = fma2(f2(__uint_as_float(acc[c][8 * j + 2 * i]),
                                                __uint_as_float(acc[c][8 * j + 2 * i + 1])),
                                             alpha2, f2(__uint_as_float(bw[i] << 16), __uint_as_float(bw[i] & 0xFFFF0000u)));
                        }
                        uint4* slot = reinterpret_cast<uint4*>(buf + swz64(lane, j));
                        if (p.has_resid) {
                            const uint4 rv = *slot;
                            const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
                            float4 g0 = make_float4(1.0f, 1.0f, 1.0f, 1.0f), g1 = g0;
                            if (kWide && gsm != nullptr) {
                                g0 = reinterpret_cast<const float4*>(gsm + 32 * c + 8 * j)[0];
                                g1 = reinterpret_cast<const float4*>(gsm + 32 * c + 8 * j)[1];
                            } else if (grow != nullptr && n8 < p.N) {
                                g0 = __ldg(reinterpret_cast<const float4*>(grow + n8));
                                g1 = __ldg(reinterpret_cast<const float4*>(grow + n8) + 1);
                            }
                            const uint64_t g2[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                y2[i] = fma2(g2[i], y2[i],
                                             f2(__uint_as_float(rw[i] << 16), __uint_as_float(rw[i] & 0xFFFF0000u)));
                        }
                        if (kAmax && row < p.M && n8 < p.N) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float lo, hi;
                                unf2(y2[i], lo, hi);
                                omax = fmaxf(omax, fmaxf(fabsf(lo), fabsf(hi)));
                            }
                        }
                        *slot = make_uint4(cvt_bf16x2(y2[0]), cvt_bf16x2(y2[1]), cvt_bf16x2(y2[2]), cvt_bf16x2(y2[3]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tma_store_2d(&tmOut, buf, nc0 + 32 * c, m0);
                    }
                }
                if (lane == 0) bulk_commit();
            }
            if constexpr (kNvfp4) {
                // Row `row` of h, columns [128 nt + 64 h, +64): 32 bytes of codes and
                // one 4-byte word of block scales (scale group 2 nt + h) in the
                // 128x4-tiled layout; rows past M (up to the 128-row padding the
                // scale layout has) get zero scales and no codes.
                const int hcol = nt * (BN / 2) + 64 * h;
                if (row < p.M) {
                    uint8_t* dst = p.h_codes + (size_t)row * (size_t)(p.N / 4) + hcol / 2;
                    asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst),
                                 "r"(hcode[0]), "r"(hcode[1]), "r"(hcode[2]), "r"(hcode[3]), "r"(hcode[4]),
                                 "r"(hcode[5]), "r"(hcode[6]), "r"(hcode[7])
                                 : "memory");
                }
                if (row < p.m_tiles * BM) {  // the odd CTA of a last pair has no rows in the layout
                    const size_t soff = ((size_t)(row >> 7) * (size_t)p.h_kb4 + (size_t)(hcol >> 6)) * 512u +
                                        (size_t)((row & 31) << 4) + (size_t)(((row >> 5) & 3) << 2);
                    *reinterpret_cast<uint32_t*>(p.h_sf + soff) = row < p.M ? hscale : 0u;
                }
            }
            if (failed) {
                if (lane == 0) set_abort();
                break;
            }
        }
        if (r_pending) (void)mbar_wait(&rbar[e], r_phase, p.wait_ns, p.status, kStatusTimeoutEpilogue);
        if constexpr (kAmax) {
            // bf16 rounding is monotone and odd, so the largest stored |out| is
            // the rounded largest |out|; non-negative floats order like their bits.
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) omax = fmaxf(omax, __shfl_xor_sync(0xffffffffu, omax, off));
            if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(bf16_round(omax)));
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    // No CTA of the pair may release TMEM or exit while the leader's MMAs and
    // copies can still touch its shared memory or TMEM, or while its partner may
    // still arrive on its barriers.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
    cluster_sync();
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

cudaError_t launch_gemm_pack_stall_selftest(const GemmJob& job, cudaStream_t s) { return launch_gemm_impl(job, 2, s); }

// Largest number of CTA pairs that can be resident at once on the current
// device (GPCs with an odd number of free SMs leave one SM idle), cached per device.
static int max_pairs_current_device()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (unsigned)sm_count_current_device());
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Plan<false, false>::kSmemBytes;  // one CTA per SM with every plan
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        const void* probe = reinterpret_cast<const void*>(nvfp4_gemm_kernel<false, false, false, false, false>);
        if (ensure_dynamic_smem(probe, (int)Plan<false, false>::kSmemBytes) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_kernel<false, false, false, false, false>, &cfg) !=
                cudaSuccess ||
            n <= 0)
            n = sm_count_current_device() / 2;
        cache[dev] = n;
    }
    return cache[dev];
}

static cudaError_t launch_gemm_impl(const GemmJob& job, int stall, cudaStream_t s)
{
    CUtensorMap tmA, tmB, tmSFA, tmSFB, tmOut, tmR, tmX;
    const bool pack = job.pk_x != nullptr;
    if (pack && (job.swiglu || job.h_codes != nullptr || (job.K + BK - 1) / BK > kPackMaxKStages))
        return cudaErrorInvalidValue;
    const uint64_t kbytes = (uint64_t)job.K / 2;
    const int64_t m_tiles = (job.M + BM - 1) / BM;
    const int64_t n_sf_tiles = (job.N + 127) / 128;
    const int64_t kb4 = job.K / 64;
    // Block scales as rows of 256 bytes: one 512-byte tile is two rows.
    const uint64_t sfa_rows = (uint64_t)(m_tiles * kb4 * 2), sfb_rows = (uint64_t)(n_sf_tiles * kb4 * 2);
    const uint64_t out_cols = job.swiglu ? (uint64_t)job.N / 2 : (uint64_t)job.N;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.a_codes, kbytes, (uint64_t)job.M, kbytes, BK / 2, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.w_codes, kbytes, (uint64_t)job.N, kbytes, BK / 2,
                     BN / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.a_sf, 256, sfa_rows, 256, 256, kSfBox / 256,
                     CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, job.w_sf, 256, sfb_rows, 256, 256, kSfBox / 256,
                     CU_TENSOR_MAP_SWIZZLE_NONE) ||
        // (NVFP4 output of h: no bf16 output is stored; the map spans the codes
        // buffer only to be valid)
        !make_map_2d(&tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, job.h_codes ? (const void*)job.h_codes : job.out,
                     job.h_codes ? (uint64_t)job.N / 8 : out_cols, (uint64_t)job.M,
                     job.h_codes ? (uint64_t)job.N / 4 : out_cols * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_2d(&tmR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     job.resid ? job.resid : (job.out ? job.out : (const void*)job.h_codes), (uint64_t)job.N,
                     (uint64_t)job.M, (uint64_t)job.N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        // the packer's X tiles: 32 rows x 256 columns (without the packer a valid stand-in)
        !make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pack ? job.pk_x : (const void*)job.a_codes,
                     pack ? (uint64_t)job.K : kbytes / 2, (uint64_t)job.M, pack ? (uint64_t)job.K * 2 : kbytes,
                     BK, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    GemmParams p{};
    p.a_gscale = job.a_gscale;
    p.w_gscale = job.w_gscale;
    p.bias = static_cast<const __nv_bfloat16*>(job.bias);
    p.gate = job.gate;
    p.M = (int)job.M;
    p.N = (int)job.N;
    p.K = (int)job.K;
    p.m_tiles = (int)m_tiles;
    p.pair_m_tiles = (int)((m_tiles + 1) / 2);
    p.n_tiles = (int)((job.N + BN - 1) / BN);
    p.k_stages = (int)((job.K + BK - 1) / BK);
    p.kb4 = (int)kb4;
    p.has_resid = job.resid != nullptr ? 1 : 0;
    p.seg = job.seg;
    p.status = job.status;
    p.wait_ns = job.wait_limit_ns;
    p.stall = stall;
    p.amax_out = job.amax_out;
    p.h_codes = job.h_codes;
    p.h_sf = job.h_sf;
    p.h_gscale = job.h_gscale;
    p.h_kb4 = (int)(job.N / 128);
    if (pack) {
        // Call numbers: a fixed odd stride walks all 2^32 values before it
        // repeats, so flags left by earlier calls never hold this call's
        // number; 0 (a zeroed workspace) is skipped.
        static std::atomic<uint32_t> calls{0};
        uint32_t e = 0;
        while (e == 0) e = (calls.fetch_add(1) + 1) * 0x9E3779B1u;
        p.pk_shift = job.pk_shift;
        p.pk_scale = job.pk_scale;
        p.pk_codes = const_cast<uint8_t*>(job.a_codes);
        p.pk_sf = const_cast<uint8_t*>(job.a_sf);
        p.pk_gscale = const_cast<float*>(job.a_gscale);
        p.pk_partials = job.pk_partials;
        p.pk_nparts = job.pk_nparts;
        p.pk_given = job.pk_given ? 1 : 0;
        p.pk_flags = job.pk_flags;
        p.pk_epoch = e;
    }

    // The wide plan where a tile's gated epilogue outlasts its mainloop (short
    // K); the pack plan when the kernel quantises its own activation.
    const bool wide = !pack && p.has_resid && !job.swiglu && job.h_codes == nullptr && p.k_stages < kWideMaxKStages;
    auto kernel = pack ? (job.amax_out ? nvfp4_gemm_kernel<false, true, false, false, true>
                                       : nvfp4_gemm_kernel<false, false, false, false, true>)
                  : job.h_codes != nullptr ? nvfp4_gemm_kernel<true, false, true, false, false>
                  : job.swiglu ? (job.amax_out ? nvfp4_gemm_kernel<true, true, false, false, false>
                                               : nvfp4_gemm_kernel<true, false, false, false, false>)
                  : wide ? (job.amax_out ? nvfp4_gemm_kernel<false, true, false, true, false>
                                         : nvfp4_gemm_kernel<false, false, false, true, false>)
                         : (job.amax_out ? nvfp4_gemm_kernel<false, true, false, false, false>
                                         : nvfp4_gemm_kernel<false, false, false, false, false>);
    const uint32_t smem_bytes = pack   ? Plan<false, true>::kSmemBytes
                                : wide ? Plan<true, false>::kSmemBytes
                                       : Plan<false, false>::kSmemBytes;
    const cudaError_t attr_err = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), (int)smem_bytes);
    if (attr_err != cudaSuccess) return attr_err;

    const int tiles = p.pair_m_tiles * p.n_tiles;
    const int max_pairs = max_pairs_current_device();
    const int pairs = tiles < max_pairs ? tiles : max_pairs;
    if (pairs <= 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * (unsigned)pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmSFA, tmSFB, tmOut, tmR, tmX, p);
}

}  // namespace h3fp4
