// C ABI of the h3fp4 library: argument validation, workspace layout, device
// check and kernel dispatch.  No entry point allocates device memory or
// synchronises a stream (h3fp4_check excepted, which exists to do so).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "h3fp4_internal.h"

namespace h3fp4 {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
int g_dev_ok[kMaxDevices];
int g_dev_sms[kMaxDevices];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

h3fp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA; }

}  // namespace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

h3fp4_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return H3FP4_ERR_CUDA;
    std::call_once(g_dev_once[dev], [dev] {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
        g_dev_sms[dev] = sms;
    });
    return g_dev_ok[dev] ? H3FP4_OK : H3FP4_ERR_UNSUPPORTED_DEVICE;
}

// Copies and validates the host segment table.
h3fp4_status make_segments(const int64_t* seg_off, int nseg, int64_t rows, Segments* out)
{
    std::memset(out, 0, sizeof(*out));
    if (seg_off == nullptr) {
        if (nseg > 1) return H3FP4_ERR_INVALID;
        out->nseg = 1;
        out->off[0] = 0;
        out->off[1] = rows;
        return H3FP4_OK;
    }
    if (nseg < 1 || nseg > H3FP4_MAX_SEGMENTS) return H3FP4_ERR_SHAPE;
    if (seg_off[0] != 0 || seg_off[nseg] != rows) return H3FP4_ERR_INVALID;
    for (int i = 0; i < nseg; ++i)
        if (seg_off[i + 1] < seg_off[i]) return H3FP4_ERR_INVALID;
    out->nseg = nseg;
    for (int i = 0; i <= nseg; ++i) out->off[i] = seg_off[i];
    return H3FP4_OK;
}

h3fp4_status check_shape(int64_t rows, int64_t K)
{
    if (rows < 1 || K < 64 || K % 64 != 0 || K > (int64_t)kMaxPartials * 1024) return H3FP4_ERR_SHAPE;
    if (rows > (int64_t)INT32_MAX || K > (int64_t)INT32_MAX / 2) return H3FP4_ERR_SHAPE;
    if (rows * (K / 8) > (int64_t)INT32_MAX * 8) return H3FP4_ERR_SHAPE;
    return H3FP4_OK;
}

cudaError_t ensure_dynamic_smem(const void* func, int bytes)
{
    struct Entry {
        const void* func;
        int dev;
    };
    static std::mutex mu;
    static Entry done[16 * kMaxDevices];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i].func == func && done[i].dev == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && ndone < 16 * kMaxDevices) done[ndone++] = Entry{func, dev};
    return e;
}

int sm_count_current_device()
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && g_dev_sms[dev] > 0) return g_dev_sms[dev];
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace h3fp4

using namespace h3fp4;

extern "C" {

size_t h3fp4_codes_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0) return 0;
    return (size_t)rows * (size_t)K / 2;
}

size_t h3fp4_sf_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0) return 0;
    return (size_t)((rows + 127) / 128) * 128 * (size_t)((K / 16 + 3) / 4) * 4;
}

size_t h3fp4_workspace_bytes(int64_t M, int64_t N, int64_t K, int flags)
{
    (void)N;
    size_t bytes = kWsActCodes;
    if (!(flags & H3FP4_A_PREQUANT))
        bytes += round256(h3fp4_codes_bytes(M, K)) + round256(h3fp4_sf_bytes(M, K)) +
                 round256(4 * pack_flag_words(M, K));
    return bytes;
}

void h3fp4_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

const char* h3fp4_status_string(h3fp4_status s)
{
    switch (s) {
    case H3FP4_OK: return "ok";
    case H3FP4_ERR_INVALID: return "invalid argument";
    case H3FP4_ERR_SHAPE: return "unsupported shape (K % 64, N % 8, rows >= 1, segments)";
    case H3FP4_ERR_ALIGN: return "pointer not 16-byte aligned";
    case H3FP4_ERR_CUDA: return "CUDA error";
    case H3FP4_ERR_TIMEOUT: return "device wait timed out";
    case H3FP4_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    }
    return "unknown status";
}

h3fp4_status h3fp4_quantize_act(const void* x_bf16, int64_t M, int64_t K, const float* shift, const float* scale,
                                const int64_t* seg_off, int nseg, void* codes, void* sf, float* gscale, int flags,
                                void* ws, cudaStream_t stream)
{
    h3fp4_status st = check_shape(M, K);
    if (st != H3FP4_OK) return st;
    if (!x_bf16 || !codes || !sf || !gscale || !ws) return H3FP4_ERR_INVALID;
    if (flags & ~(H3FP4_PROLOGUE_MOD | H3FP4_GSCALE_GIVEN)) return H3FP4_ERR_INVALID;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(sf) || !aligned16(ws) ||
        (reinterpret_cast<uintptr_t>(gscale) & 3u) || (mod && (!aligned16(shift) || !aligned16(scale))))
        return H3FP4_ERR_ALIGN;
    QuantJob job{};
    st = make_segments(seg_off, nseg <= 0 ? 1 : nseg, M, &job.seg);
    if (st != H3FP4_OK) return st;
    if ((st = check_device()) != H3FP4_OK) return st;
    job.x = x_bf16;
    job.rows = M;
    job.K = K;
    job.shift = mod ? shift : nullptr;
    job.scale = mod ? scale : nullptr;
    job.codes = static_cast<uint8_t*>(codes);
    job.sf = static_cast<uint8_t*>(sf);
    job.gscale = gscale;
    job.gscale_given = (flags & H3FP4_GSCALE_GIVEN) != 0;
    job.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsPartials);
    return from_cuda(launch_quantize(job, stream));
}

h3fp4_status h3fp4_quantize_weight(const void* w_bf16, int64_t N, int64_t K, void* codes, void* sf,
                                   float* w_gscale, void* ws, cudaStream_t stream)
{
    if (N % 8 != 0) return H3FP4_ERR_SHAPE;
    return h3fp4_quantize_act(w_bf16, N, K, nullptr, nullptr, nullptr, 1, codes, sf, w_gscale, 0, ws, stream);
}

h3fp4_status h3fp4_linear(const void* x, const void* a_sf, const float* a_gscale, int64_t M, int64_t N, int64_t K,
                          const void* w_codes, const void* w_sf, const float* w_gscale, const float* shift,
                          const float* scale, const float* gate, const int64_t* seg_off, int nseg,
                          const void* bias_bf16, const void* resid_bf16, void* out_bf16, int flags, void* ws,
                          cudaStream_t stream)
{
    h3fp4_status st = check_shape(M, K);
    if (st != H3FP4_OK) return st;
    if (N < 8 || N % 8 != 0 || N > (int64_t)INT32_MAX) return H3FP4_ERR_SHAPE;
    const int known = H3FP4_PROLOGUE_MOD | H3FP4_EPI_BIAS | H3FP4_EPI_GATE_RESID | H3FP4_GSCALE_GIVEN |
                      H3FP4_A_PREQUANT | H3FP4_EPI_SWIGLU | H3FP4_EPI_AMAX | H3FP4_FUSED_QUANT;
    if (flags & ~known) return H3FP4_ERR_INVALID;
    const bool prequant = (flags & H3FP4_A_PREQUANT) != 0;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    const bool bias = (flags & H3FP4_EPI_BIAS) != 0;
    const bool gated = (flags & H3FP4_EPI_GATE_RESID) != 0;
    const bool given = (flags & H3FP4_GSCALE_GIVEN) != 0;
    const bool swiglu = (flags & H3FP4_EPI_SWIGLU) != 0;
    const bool want_amax = (flags & H3FP4_EPI_AMAX) != 0;
    const bool fused = (flags & H3FP4_FUSED_QUANT) != 0;
    if (swiglu && N % 256 != 0) return H3FP4_ERR_SHAPE;
    if (fused && (prequant || swiglu)) return H3FP4_ERR_INVALID;
    if (fused && (K + 255) / 256 > kPackMaxKStages) return H3FP4_ERR_SHAPE;
    if (swiglu && gated) return H3FP4_ERR_INVALID;
    if (!x || !w_codes || !w_sf || !w_gscale || !out_bf16 || !ws) return H3FP4_ERR_INVALID;
    if (prequant && (mod || !a_sf || !a_gscale)) return H3FP4_ERR_INVALID;
    if (given && !a_gscale) return H3FP4_ERR_INVALID;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (bias && !bias_bf16) return H3FP4_ERR_INVALID;
    if (gated && (!gate || !resid_bf16)) return H3FP4_ERR_INVALID;
    if (out_bf16 == x || (gated && out_bf16 == resid_bf16)) return H3FP4_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_codes) || !aligned16(w_sf) || !aligned16(out_bf16) || !aligned16(ws) ||
        (prequant && !aligned16(a_sf)) || (bias && !aligned16(bias_bf16)) ||
        (gated && (!aligned16(gate) || !aligned16(resid_bf16))) || (mod && (!aligned16(shift) || !aligned16(scale))))
        return H3FP4_ERR_ALIGN;
    Segments seg;
    st = make_segments(seg_off, nseg <= 0 ? 1 : nseg, M, &seg);
    if (st != H3FP4_OK) return st;
    if ((st = check_device()) != H3FP4_OK) return st;
    if (fused) {
        // The ready flags carry this call's number, fixed at launch: a captured
        // launch replayed from a graph would find the flags of its own previous
        // replay already set.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return H3FP4_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return H3FP4_ERR_INVALID;
    }

    uint8_t* wsb = static_cast<uint8_t*>(ws);
    // Zeroed ahead of the quantiser so that the quantiser -> GEMM launch pair
    // stays adjacent (programmatic dependent launch).
    if (want_amax && (st = from_cuda(cudaMemsetAsync(wsb + kWsOutAmax, 0, sizeof(float), stream))) != H3FP4_OK)
        return st;
    GemmJob g{};
    if (prequant) {
        g.a_codes = static_cast<const uint8_t*>(x);
        g.a_sf = static_cast<const uint8_t*>(a_sf);
        g.a_gscale = a_gscale;
    } else {
        QuantJob q{};
        q.x = x;
        q.rows = M;
        q.K = K;
        q.shift = mod ? shift : nullptr;
        q.scale = mod ? scale : nullptr;
        q.seg = seg;
        q.codes = wsb + kWsActCodes;
        q.sf = q.codes + round256(h3fp4_codes_bytes(M, K));
        q.gscale = given ? const_cast<float*>(a_gscale) : reinterpret_cast<float*>(wsb + kWsActGscale);
        q.gscale_given = given;
        q.partials = reinterpret_cast<float*>(wsb + kWsPartials);
        if (fused) {
            // amax pass (unless given); the GEMM kernel packs and consumes the tiles
            int nparts = 0;
            if (!given && (st = from_cuda(launch_amax_partials(q, &nparts, stream))) != H3FP4_OK) return st;
            g.pk_x = x;
            g.pk_shift = q.shift;
            g.pk_scale = q.scale;
            g.pk_partials = q.partials;
            g.pk_nparts = nparts;
            g.pk_given = given;
            g.pk_flags = reinterpret_cast<uint32_t*>(q.sf + round256(h3fp4_sf_bytes(M, K)));
        } else if ((st = from_cuda(launch_quantize(q, stream))) != H3FP4_OK) {
            return st;
        }
        g.a_codes = q.codes;
        g.a_sf = q.sf;
        g.a_gscale = q.gscale;
    }
    g.w_codes = static_cast<const uint8_t*>(w_codes);
    g.w_sf = static_cast<const uint8_t*>(w_sf);
    g.w_gscale = w_gscale;
    g.M = M;
    g.N = N;
    g.K = K;
    g.bias = bias ? bias_bf16 : nullptr;
    g.gate = gated ? gate : nullptr;
    g.resid = gated ? resid_bf16 : nullptr;
    g.out = out_bf16;
    g.seg = seg;
    g.status = reinterpret_cast<unsigned int*>(wsb + kWsStatus);
    g.wait_limit_ns = g_wait_limit_ns.load();
    g.swiglu = swiglu;
    g.amax_out = want_amax ? reinterpret_cast<float*>(wsb + kWsOutAmax) : nullptr;
    return from_cuda(launch_gemm(g, stream));
}

h3fp4_status h3fp4_linear_swiglu_nvfp4(const void* x, const void* a_sf, const float* a_gscale, int64_t M, int64_t N,
                                       int64_t K, const void* w_codes, const void* w_sf, const float* w_gscale,
                                       const float* shift, const float* scale, const int64_t* seg_off, int nseg,
                                       const void* bias_bf16, const float* h_gscale, void* h_codes, void* h_sf,
                                       int flags, void* ws, cudaStream_t stream)
{
    h3fp4_status st = check_shape(M, K);
    if (st != H3FP4_OK) return st;
    if (N < 256 || N % 256 != 0 || N > (int64_t)INT32_MAX) return H3FP4_ERR_SHAPE;
    const int known = H3FP4_PROLOGUE_MOD | H3FP4_EPI_BIAS | H3FP4_GSCALE_GIVEN | H3FP4_A_PREQUANT;
    if (flags & ~known) return H3FP4_ERR_INVALID;
    const bool prequant = (flags & H3FP4_A_PREQUANT) != 0;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    const bool bias = (flags & H3FP4_EPI_BIAS) != 0;
    const bool given = (flags & H3FP4_GSCALE_GIVEN) != 0;
    if (!x || !w_codes || !w_sf || !w_gscale || !h_gscale || !h_codes || !h_sf || !ws) return H3FP4_ERR_INVALID;
    if (prequant && (mod || !a_sf || !a_gscale)) return H3FP4_ERR_INVALID;
    if (given && !a_gscale) return H3FP4_ERR_INVALID;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (bias && !bias_bf16) return H3FP4_ERR_INVALID;
    if (h_codes == x || h_codes == w_codes || h_sf == w_sf) return H3FP4_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_codes) || !aligned16(w_sf) || !aligned16(h_codes) || !aligned16(h_sf) ||
        !aligned16(ws) || (reinterpret_cast<uintptr_t>(h_gscale) & 3u) || (prequant && !aligned16(a_sf)) ||
        (bias && !aligned16(bias_bf16)) || (mod && (!aligned16(shift) || !aligned16(scale))))
        return H3FP4_ERR_ALIGN;
    Segments seg;
    st = make_segments(seg_off, nseg <= 0 ? 1 : nseg, M, &seg);
    if (st != H3FP4_OK) return st;
    if ((st = check_device()) != H3FP4_OK) return st;

    uint8_t* wsb = static_cast<uint8_t*>(ws);
    GemmJob g{};
    if (prequant) {
        g.a_codes = static_cast<const uint8_t*>(x);
        g.a_sf = static_cast<const uint8_t*>(a_sf);
        g.a_gscale = a_gscale;
    } else {
        QuantJob q{};
        q.x = x;
        q.rows = M;
        q.K = K;
        q.shift = mod ? shift : nullptr;
        q.scale = mod ? scale : nullptr;
        q.seg = seg;
        q.codes = wsb + kWsActCodes;
        q.sf = q.codes + round256(h3fp4_codes_bytes(M, K));
        q.gscale = given ? const_cast<float*>(a_gscale) : reinterpret_cast<float*>(wsb + kWsActGscale);
        q.gscale_given = given;
        q.partials = reinterpret_cast<float*>(wsb + kWsPartials);
        if ((st = from_cuda(launch_quantize(q, stream))) != H3FP4_OK) return st;
        g.a_codes = q.codes;
        g.a_sf = q.sf;
        g.a_gscale = q.gscale;
    }
    g.w_codes = static_cast<const uint8_t*>(w_codes);
    g.w_sf = static_cast<const uint8_t*>(w_sf);
    g.w_gscale = w_gscale;
    g.M = M;
    g.N = N;
    g.K = K;
    g.bias = bias ? bias_bf16 : nullptr;
    g.seg = seg;
    g.status = reinterpret_cast<unsigned int*>(wsb + kWsStatus);
    g.wait_limit_ns = g_wait_limit_ns.load();
    g.swiglu = true;
    g.h_codes = static_cast<uint8_t*>(h_codes);
    g.h_sf = static_cast<uint8_t*>(h_sf);
    g.h_gscale = h_gscale;
    return from_cuda(launch_gemm(g, stream));
}

float* h3fp4_ws_out_amax(void* ws)
{
    return ws ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsOutAmax) : nullptr;
}

h3fp4_status h3fp4_act_amax(const void* x_bf16, int64_t M, int64_t K, const float* shift, const float* scale,
                            const int64_t* seg_off, int nseg, float* amax, int flags, void* ws, cudaStream_t stream)
{
    h3fp4_status st = check_shape(M, K);
    if (st != H3FP4_OK) return st;
    if (!x_bf16 || !amax || !ws) return H3FP4_ERR_INVALID;
    if (flags & ~H3FP4_PROLOGUE_MOD) return H3FP4_ERR_INVALID;
    const bool mod = (flags & H3FP4_PROLOGUE_MOD) != 0;
    if (mod && (!shift || !scale)) return H3FP4_ERR_INVALID;
    if (!aligned16(x_bf16) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(amax) & 3u) ||
        (mod && (!aligned16(shift) || !aligned16(scale))))
        return H3FP4_ERR_ALIGN;
    QuantJob job{};
    st = make_segments(seg_off, nseg <= 0 ? 1 : nseg, M, &job.seg);
    if (st != H3FP4_OK) return st;
    if ((st = check_device()) != H3FP4_OK) return st;
    job.x = x_bf16;
    job.rows = M;
    job.K = K;
    job.shift = mod ? shift : nullptr;
    job.scale = mod ? scale : nullptr;
    job.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsPartials);
    return from_cuda(launch_amax(job, amax, stream));
}

h3fp4_status h3fp4_gscale_from_amax(const float* amax, float* gscale, cudaStream_t stream)
{
    if (!amax || !gscale) return H3FP4_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(gscale) & 3u))
        return H3FP4_ERR_ALIGN;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    return from_cuda(launch_gscale_from_amax(amax, gscale, stream));
}

h3fp4_status h3fp4_selftest_timeout(void* ws, uint64_t limit_ns, cudaStream_t stream)
{
    if (!ws) return H3FP4_ERR_INVALID;
    if (!aligned16(ws)) return H3FP4_ERR_ALIGN;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    GemmJob g{};
    // Dummy operands: the tensor maps need valid, aligned addresses but the
    // disabled producer never issues a copy and no output is ever stored.
    g.a_codes = wsb + kWsActCodes;
    g.a_sf = wsb + kWsActCodes;
    g.a_gscale = reinterpret_cast<const float*>(wsb + kWsActGscale);
    g.w_codes = wsb + kWsActCodes;
    g.w_sf = wsb + kWsActCodes;
    g.w_gscale = reinterpret_cast<const float*>(wsb + kWsActGscale);
    g.M = 128;
    g.N = 256;
    g.K = 256;
    g.out = wsb + kWsActCodes;
    g.seg.nseg = 1;
    g.seg.off[1] = 128;
    g.status = reinterpret_cast<unsigned int*>(wsb + kWsStatus);
    g.wait_limit_ns = limit_ns ? limit_ns : 1;
    return from_cuda(launch_gemm_stall_selftest(g, stream));
}

h3fp4_status h3fp4_selftest_pack_timeout(const void* x_bf16, const float* a_gscale, void* ws, uint64_t limit_ns,
                                         cudaStream_t stream)
{
    if (!x_bf16 || !a_gscale || !ws) return H3FP4_ERR_INVALID;
    if (!aligned16(x_bf16) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(a_gscale) & 3u)) return H3FP4_ERR_ALIGN;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const int64_t M = 128, N = 256, K = 256;
    GemmJob g{};
    // The packer writes the workspace's codes, scales and flags; the GEMM
    // issues no copy (it never sees a published tile) and stores no output.
    g.a_codes = wsb + kWsActCodes;
    g.a_sf = wsb + kWsActCodes + round256(h3fp4_codes_bytes(M, K));
    g.a_gscale = a_gscale;
    g.w_codes = g.a_codes;
    g.w_sf = g.a_sf;
    g.w_gscale = a_gscale;
    g.M = M;
    g.N = N;
    g.K = K;
    g.out = wsb + kWsActCodes;
    g.seg.nseg = 1;
    g.seg.off[1] = M;
    g.status = reinterpret_cast<unsigned int*>(wsb + kWsStatus);
    g.wait_limit_ns = limit_ns ? limit_ns : 1;
    g.pk_x = x_bf16;
    g.pk_given = true;
    g.pk_flags = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(g.a_sf) + round256(h3fp4_sf_bytes(M, K)));
    return from_cuda(launch_gemm_pack_stall_selftest(g, stream));
}

h3fp4_status h3fp4_measure_fp4_peak(int iters, float* tflops, void* ws)
{
    if (!tflops || !ws || iters < 1) return H3FP4_ERR_INVALID;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    return from_cuda(measure_fp4_peak(iters, reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kWsStatus),
                                      tflops));
}

h3fp4_status h3fp4_measure_fp4_pair_peak(int iters, float* tflops, void* ws)
{
    if (!tflops || !ws || iters < 1) return H3FP4_ERR_INVALID;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    return from_cuda(
        measure_fp4_pair_peak(iters, reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kWsStatus), tflops));
}

h3fp4_status h3fp4_measure_fp4_form(int form, int iters, float* tflops, void* ws)
{
    if (!tflops || !ws || iters < 1 || form < H3FP4_MMA_SINGLE || form > H3FP4_MMA_PAIR_N128)
        return H3FP4_ERR_INVALID;
    h3fp4_status st = check_device();
    if (st != H3FP4_OK) return st;
    return from_cuda(measure_fp4_form(form, iters,
                                      reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kWsStatus), tflops));
}

h3fp4_status h3fp4_check(void* ws, cudaStream_t stream)
{
    if (!ws) return H3FP4_ERR_INVALID;
    unsigned int word = 0;
    unsigned int* dev = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + kWsStatus);
    if (cudaMemcpyAsync(&word, dev, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return H3FP4_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(dev, 0, sizeof(word), stream) != cudaSuccess) return H3FP4_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return H3FP4_ERR_CUDA;
        return H3FP4_ERR_TIMEOUT;
    }
    return H3FP4_OK;
}

}  // extern "C"
