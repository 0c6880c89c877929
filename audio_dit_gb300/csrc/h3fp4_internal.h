// Internal declarations shared by the h3fp4 translation units (not part of the ABI).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/h3fp4.h"

namespace h3fp4 {

// Workspace layout (bytes from the workspace base, each region 256-aligned).
constexpr size_t kWsStatus = 0;         // uint32 device status word (+ padding)
constexpr size_t kWsPartials = 256;     // fp32 amax partial maxima
constexpr int kMaxPartials = 4096;
constexpr size_t kWsActGscale = kWsPartials + 4 * kMaxPartials;  // fp32 activation global scale
constexpr size_t kWsOutAmax = kWsActGscale + 16;                  // fp32 max |out| of the last EPI_AMAX call
constexpr size_t kWsActCodes = kWsActGscale + 256;                // activation codes, then block scales

// Device status bits (workspace status word).
constexpr unsigned int kStatusTimeoutProducer = 1u;
constexpr unsigned int kStatusTimeoutMma = 2u;
constexpr unsigned int kStatusTimeoutEpilogue = 4u;
constexpr unsigned int kStatusBadSmemAlign = 8u;
constexpr unsigned int kStatusTimeoutPackFlag = 16u;  // GEMM producer: an activation tile never published
constexpr unsigned int kStatusTimeoutPacker = 32u;    // in-kernel packer: an X tile never landed

struct Segments {
    int nseg;
    long long off[H3FP4_MAX_SEGMENTS + 1];
};

struct QuantJob {
    const void* x;          // bf16 [rows][K]
    int64_t rows, K;
    const float* shift;     // [nseg][K] or null (no prologue)
    const float* scale;
    Segments seg;
    uint8_t* codes;         // [rows][K/2]
    uint8_t* sf;            // sf_bytes(rows, K)
    float* gscale;          // device fp32 (in if given, else out)
    bool gscale_given;
    float* partials;        // kMaxPartials floats
};

// Launches the amax pass (unless gscale_given) and the pack pass.
cudaError_t launch_quantize(const QuantJob& job, cudaStream_t s);

struct GemmJob {
    const uint8_t* a_codes;  // [M][K/2]
    const uint8_t* a_sf;
    const float* a_gscale;
    const uint8_t* w_codes;  // [N][K/2]
    const uint8_t* w_sf;
    const float* w_gscale;
    int64_t M, N, K;
    const void* bias;        // bf16 [N] or null
    const float* gate;       // fp32 [nseg][N] or null
    const void* resid;       // bf16 [M][N] or null
    void* out;               // bf16 [M][N], or [M][N/2] with swiglu
    Segments seg;
    unsigned int* status;    // device status word
    uint64_t wait_limit_ns;
    bool swiglu;             // SwiGLU epilogue (N % 256 == 0, no gate/residual)
    float* amax_out;         // zeroed by the caller; receives max |out| (or null)
    // SwiGLU with h written as NVFP4 (codes [M][N/4], block scales of h) under
    // the given global scale of h; null for a bf16 output
    uint8_t* h_codes;
    uint8_t* h_sf;
    const float* h_gscale;
    // In-kernel quantisation of the activation (plain or gated epilogue): the
    // kernel's packer warps write a_codes / a_sf from X (and, unless
    // pk_given, the global scale into a_gscale from the amax pass's partials)
    // while its GEMM consumes them.  Null pk_x: a_codes / a_sf are inputs.
    const void* pk_x;         // bf16 [M][K]
    const float* pk_shift;    // [nseg][K] or null
    const float* pk_scale;
    const float* pk_partials;
    int pk_nparts;
    bool pk_given;
    uint32_t* pk_flags;       // pack_flag_words(M, K) words, owned by the call
};

// Ready-flag words the in-kernel quantisation needs: one per (128-row tile,
// 256-column stage) of the activation.
inline size_t pack_flag_words(int64_t M, int64_t K) { return (size_t)((M + 127) / 128) * (size_t)((K + 255) / 256); }

// K stages per tile the in-kernel quantisation supports (K <= 16384).
constexpr int kPackMaxKStages = 64;

// Launches only the amax pass; *nparts receives the number of partials it writes.
cudaError_t launch_amax_partials(const QuantJob& job, int* nparts, cudaStream_t s);

cudaError_t launch_gemm(const GemmJob& job, cudaStream_t s);

// The same GEMM kernel with its producer disabled: every consumer wait runs out,
// the kernel records a timeout in the status word and returns (self-test).
cudaError_t launch_gemm_stall_selftest(const GemmJob& job, cudaStream_t s);

// The in-kernel quantisation with its packer publishing no tile: every wait of
// the producer for a tile runs out (self-test).
cudaError_t launch_gemm_pack_stall_selftest(const GemmJob& job, cudaStream_t s);

// Global amax of the (modulated) activation into amax_out (device fp32).
cudaError_t launch_amax(const QuantJob& job, float* amax_out, cudaStream_t s);

// gscale = (amax == 0) ? 1 : amax / (6 * 448), one thread.
cudaError_t launch_gscale_from_amax(const float* amax, float* gscale, cudaStream_t s);

int sm_count_current_device();

// Host-side validation shared by every entry point (defined in h3fp4_api.cu).
bool aligned16(const void* p);
// H3FP4_OK on an sm_103 current device, else ERR_UNSUPPORTED_DEVICE / ERR_CUDA.
h3fp4_status check_device();
// Copies and validates the host segment table (nseg <= 0 is read as 1).
h3fp4_status make_segments(const int64_t* seg_off, int nseg, int64_t rows, Segments* out);
// rows >= 1, K a positive multiple of 64 within the amax-partials budget.
h3fp4_status check_shape(int64_t rows, int64_t K);

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize of `func` on the current
// device the first time it is asked for that (function, device) pair; the
// attribute belongs to each device's context.
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

// Synchronous: FP4 MMA loop on every SM, returns TFLOP/s (status word for its bounded wait).
cudaError_t measure_fp4_peak(int iters, unsigned int* status, float* tflops);

// The same for the paired (cta_group::2) MMA on every 2-CTA cluster.
cudaError_t measure_fp4_pair_peak(int iters, unsigned int* status, float* tflops);

// The same for any h3fp4_mma_form.
cudaError_t measure_fp4_form(int form, int iters, unsigned int* status, float* tflops);

}  // namespace h3fp4
