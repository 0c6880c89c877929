// h3fp4_quantize_act_noalloc: the activation quantiser for callers that are
// handed only their input and output buffers and may not allocate device
// memory -- for example a plugin whose host application owns all device memory
// and offers it no workspace, or a serving loop that forbids device allocation
// once it is running, because cudaMalloc/cudaFree can synchronise the device
// and fragment a pool that another allocator manages.
//
// The only scratch the quantiser needs is the list of per-CTA amax partial
// maxima of its first pass.  Here it lives in a file-scope __device__ array
// (kNoAllocPartials floats = 16 KiB, held by every GPU that loads the library
// until the process exits) instead of a caller workspace.  Host code cannot
// pass the array's name to a kernel -- on the host that name is only a
// stand-in, not a device address -- so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current, and every
// later call on that device reuses it.
//
// Nothing in this file allocates: no cudaMalloc, cudaFree or allocating
// library routine.  All calls share the one array, which keeps what the last
// call wrote; every call writes each partial it later reads, so nothing needs
// clearing, but calls that can overlap on the GPU (different streams, or
// several host threads) race on the array and must be serialised by the caller.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "h3fp4_internal.h"

namespace h3fp4 {
namespace {

constexpr int kNoAllocPartials = kMaxPartials;  // 4096 fp32 partial maxima
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::once_flag g_addr_once[kNoAllocMaxDevices];
float* g_addr[kNoAllocMaxDevices];
cudaError_t g_addr_err[kNoAllocMaxDevices];

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace h3fp4

using namespace h3fp4;

extern "C" h3fp4_status h3fp4_quantize_act_noalloc(const void* x_bf16, int64_t M, int64_t K, const float* shift,
                                                   const float* scale, const int64_t* seg_off, int nseg, void* codes,
                                                   void* sf, float* gscale, int flags, cudaStream_t stream)
{
    // Shapes: every 1024-column slab of a row needs at least one partial, so K
    // is capped at kNoAllocPartials * 1024 columns; rows are unbounded by the
    // scratch (the grid is sized to the partial count).
    if (M < 1 || K < 64 || K % 64 != 0 || M > (int64_t)INT32_MAX) return H3FP4_ERR_SHAPE;
    if (K > (int64_t)kNoAllocPartials * 1024) return H3FP4_ERR_SHAPE;
    if (M * (K / 8) > (int64_t)INT32_MAX * 8) return H3FP4_ERR_SHAPE;
    if (!x_bf16 || !codes || !sf || !gscale) return H3FP4_ERR_INVALID;
    if (flags & ~(H3FP4_PROLOGUE_MOD | H3FP4_GSCALE_GIVEN)) return H3FP4_ERR_INVALID;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (!is_aligned16(x_bf16) || !is_aligned16(codes) || !is_aligned16(sf) ||
        (reinterpret_cast<uintptr_t>(gscale) & 3u) || (mod && (!is_aligned16(shift) || !is_aligned16(scale))))
        return H3FP4_ERR_ALIGN;

    QuantJob job{};
    std::memset(&job.seg, 0, sizeof(job.seg));
    if (seg_off == nullptr) {
        if (nseg > 1) return H3FP4_ERR_INVALID;
        job.seg.nseg = 1;
        job.seg.off[1] = M;
    } else {
        if (nseg < 1 || nseg > H3FP4_MAX_SEGMENTS) return H3FP4_ERR_SHAPE;
        if (seg_off[0] != 0 || seg_off[nseg] != M) return H3FP4_ERR_INVALID;
        for (int i = 0; i < nseg; ++i)
            if (seg_off[i + 1] < seg_off[i]) return H3FP4_ERR_INVALID;
        job.seg.nseg = nseg;
        for (int i = 0; i <= nseg; ++i) job.seg.off[i] = seg_off[i];
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return H3FP4_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    if (major != 10 || minor != 3) return H3FP4_ERR_UNSUPPORTED_DEVICE;

    // One-time set-up per device, with that device current: the device address
    // of the scratch array.
    std::call_once(g_addr_once[dev], [dev] {
        void* p = nullptr;
        g_addr_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_partials);
        g_addr[dev] = static_cast<float*>(p);
    });
    if (g_addr_err[dev] != cudaSuccess || g_addr[dev] == nullptr) return H3FP4_ERR_CUDA;

    job.x = x_bf16;
    job.rows = M;
    job.K = K;
    job.shift = mod ? shift : nullptr;
    job.scale = mod ? scale : nullptr;
    job.codes = static_cast<uint8_t*>(codes);
    job.sf = static_cast<uint8_t*>(sf);
    job.gscale = gscale;
    job.gscale_given = (flags & H3FP4_GSCALE_GIVEN) != 0;
    job.partials = g_addr[dev];
    return launch_quantize(job, stream) == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}
