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
#include <mutex>

#include "h3fp4_internal.h"

namespace h3fp4 {
namespace {

constexpr int kNoAllocPartials = kMaxPartials;  // 4096 fp32 partial maxima
constexpr int kNoAllocMaxDevices = 64;
static_assert(kNoAllocPartials >= kMaxPartials, "the amax pass may write kMaxPartials partials");

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

// Device address of the array per device; a failed look-up is not cached, so
// a later call retries it.
std::mutex g_addr_mu;
float* g_addr[kNoAllocMaxDevices];

}  // namespace
}  // namespace h3fp4

using namespace h3fp4;

extern "C" h3fp4_status h3fp4_quantize_act_noalloc(const void* x_bf16, int64_t M, int64_t K, const float* shift,
                                                   const float* scale, const int64_t* seg_off, int nseg, void* codes,
                                                   void* sf, float* gscale, int flags, cudaStream_t stream)
{
    // Validation is shared with h3fp4_quantize_act, so both entries accept and
    // reject the same arguments.  check_shape caps K at kMaxPartials * 1024
    // columns: every 1024-column slab of a row needs one partial, and the grid
    // is sized to at most kNoAllocPartials partials, so rows are unbounded by
    // the scratch.
    h3fp4_status st = check_shape(M, K);
    if (st != H3FP4_OK) return st;
    if (K > (int64_t)kNoAllocPartials * 1024) return H3FP4_ERR_SHAPE;
    if (!x_bf16 || !codes || !sf || !gscale) return H3FP4_ERR_INVALID;
    if (flags & ~(H3FP4_PROLOGUE_MOD | H3FP4_GSCALE_GIVEN)) return H3FP4_ERR_INVALID;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(sf) || (reinterpret_cast<uintptr_t>(gscale) & 3u) ||
        (mod && (!aligned16(shift) || !aligned16(scale))))
        return H3FP4_ERR_ALIGN;
    QuantJob job{};
    st = make_segments(seg_off, nseg <= 0 ? 1 : nseg, M, &job.seg);
    if (st != H3FP4_OK) return st;
    if ((st = check_device()) != H3FP4_OK) return st;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return H3FP4_ERR_CUDA;
    // One-time set-up per device, with that device current: the device address
    // of the scratch array (cached for the life of the process; see the header
    // for cudaDeviceReset).
    float* partials = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_addr_mu);
        if (g_addr[dev] == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) return H3FP4_ERR_CUDA;
            g_addr[dev] = static_cast<float*>(p);
        }
        partials = g_addr[dev];
    }

    job.x = x_bf16;
    job.rows = M;
    job.K = K;
    job.shift = mod ? shift : nullptr;
    job.scale = mod ? scale : nullptr;
    job.codes = static_cast<uint8_t*>(codes);
    job.sf = static_cast<uint8_t*>(sf);
    job.gscale = gscale;
    job.gscale_given = (flags & H3FP4_GSCALE_GIVEN) != 0;
    job.partials = partials;
    return launch_quantize(job, stream) == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}
