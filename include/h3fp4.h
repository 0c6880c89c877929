/*
 * h3fp4 -- NVFP4 linear path for GB300 (sm_103a), C ABI.
 *
 * One linear layer of a joint video/audio diffusion transformer (QKV,
 * attention output, MLP FC1, MLP FC2) computed as
 *
 *     m   = bf16(x * (1 + scale[seg]) + shift[seg])        (optional AdaLN prologue)
 *     A   = NVFP4(m)    W = NVFP4(w)                      (16-element E4M3 blocks,
 *                                                          fp32 global scales)
 *     y   = (s_a * s_w) * (A_q . W_q^T)                   (fp32 accumulation)
 *     out = bf16(R + g[seg] * (y + b))  or  bf16(y + b)   (bias + residual gate)
 *
 * Sources (page title / section):
 *   "H3 Runtime Current State", "Owned Performance Kernels": the scale/pack/GEMM
 *     paths, the block-scale swizzle at every projection width, tensor
 *     scale/QDATA/SFA, alpha applied before the BF16 cast, the allocation-free
 *     caller-owned "_into" producer, one full-activation scale, modulation fused
 *     into scale/pack with exact BF16 values, and the removal of intermediate
 *     traffic across the scale/pack/GEMM boundaries;
 *   "H3 Runtime Current State", "Implemented And Validated": fused modulation
 *     and residual gates;
 *   "H3 Blackwell Runtime Plan", "Next Performance Plan: Blackwell NVFP4
 *     GEMMs": qdata + cuBLAS tiled block-scale layout, signed zero,
 *     tie-to-even FP4 rounding; residual, norms and modulation stay BF16.
 *
 * Data formats
 *   bf16 tensors      row-major, contiguous, 16-byte aligned base.
 *   codes             [rows][K/2] bytes; byte j of a row holds element 2j in
 *                     bits 0-3 and element 2j+1 in bits 4-7 (E2M1: sign bit 3,
 *                     magnitudes {0,0.5,1,1.5,2,3,4,6}).
 *   sf (block scales) E4M3 bytes, one per (row, 16-element block), stored in
 *                     128x4 tiles of 512 bytes:
 *                       offset(r, c) = ((r/128)*(K/64) + c/4)*512
 *                                      + (r%32)*16 + ((r%128)/32)*4 + c%4
 *                     rows padded to a multiple of 128 with zero bytes.
 *   global scale      one fp32 in DEVICE memory: s = amax / (6*448), or 1 for
 *                     an all-zero tensor.  Dequantised value = e2m1 * e4m3 * s.
 *
 * Quantiser (bit-exact contract, every step one IEEE fp32 round-to-nearest op):
 *   bmax = max|m| over the block; S = e4m3_rne_sat((bmax / 6) / s);
 *   eff = S * s; r = (eff == 0) ? 0 : min(1 / eff, FLT_MAX);
 *   q_i = e2m1_rne_sat(m_i * r), sign kept (negative values that round to
 *   zero give -0).  Inputs must be finite.
 *
 * Common rules
 *   - Every device buffer is caller-owned; the library never allocates
 *     device memory and never synchronises the stream.
 *   - All calls are asynchronous on `stream`; the return value reports host
 *     validation and launch errors only.  Device-side wait timeouts are
 *     recorded in the workspace status word; read them with h3fp4_check().
 *   - Shapes: K % 64 == 0, N % 8 == 0, rows >= 1; 16-byte aligned pointers
 *     (codes, sf, bf16 tensors, workspace); violations return
 *     H3FP4_ERR_SHAPE / H3FP4_ERR_ALIGN and launch nothing.
 *   - Only sm_103 devices are accepted (H3FP4_ERR_UNSUPPORTED_DEVICE
 *     otherwise).  There is no CPU fallback and no other backend.
 *   - Kernels launch with programmatic dependent launch: a kernel may start
 *     its prologue while the previous kernel of the stream drains, and reads
 *     nothing written before it until that kernel has completed.  Stream
 *     order is unchanged.
 *   - The GEMM runs as clusters of two CTAs (512 threads, ~228 KB of shared
 *     memory and all 512 TMEM columns each), one CTA per SM, over every SM
 *     pair that can be co-resident.
 *   - Calls issue only kernel launches and (with H3FP4_EPI_AMAX) one memset
 *     on `stream`, so a fixed sequence of calls can be captured into a CUDA
 *     graph.  Make one eager call per device before the first capture: it
 *     performs the library's one-time per-device setup (kernel attributes,
 *     occupancy queries).
 */
#ifndef H3FP4_H
#define H3FP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define H3FP4_API __attribute__((visibility("default")))
#else
#define H3FP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    H3FP4_OK = 0,
    H3FP4_ERR_INVALID = 1,            /* null pointer, bad flag combination, bad segments */
    H3FP4_ERR_SHAPE = 2,              /* K % 64, N % 8, rows < 1, too many segments       */
    H3FP4_ERR_ALIGN = 3,              /* a pointer is not 16-byte aligned                 */
    H3FP4_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed                */
    H3FP4_ERR_TIMEOUT = 5,            /* a bounded device wait ran out (h3fp4_check)      */
    H3FP4_ERR_UNSUPPORTED_DEVICE = 6  /* the current device is not sm_103                 */
} h3fp4_status;

enum {
    H3FP4_PROLOGUE_MOD = 1,    /* apply m = bf16(fma(x, 1 + scale[seg][k], shift[seg][k]))        */
    H3FP4_EPI_BIAS = 2,        /* add bias[n] (bf16)                                               */
    H3FP4_EPI_GATE_RESID = 4,  /* out = R[m][n] + gate[seg][n] * v   (gate fp32 [nseg][N])         */
    H3FP4_GSCALE_GIVEN = 16,   /* activation global scale read from a_gscale (device fp32 > 0)     */
    H3FP4_A_PREQUANT = 32,     /* x is already NVFP4: codes + a_sf + a_gscale                     */
    H3FP4_EPI_SWIGLU = 64,     /* out[M][N/2] = bf16(silu(g) * u), see h3fp4_linear                */
    H3FP4_EPI_AMAX = 128,      /* also write max|out| to h3fp4_ws_out_amax(ws)                    */
    H3FP4_FUSED_QUANT = 256    /* quantise x inside the GEMM kernel, see h3fp4_linear              */
};

#define H3FP4_MAX_SEGMENTS 8

/* Bytes of the E2M1 codes of a [rows, K] operand: rows * K / 2. */
H3FP4_API size_t h3fp4_codes_bytes(int64_t rows, int64_t K);

/* Bytes of the block-scale tiles of a [rows, K] operand:
 * ceil(rows/128) * 128 * (K/64) * 4. */
H3FP4_API size_t h3fp4_sf_bytes(int64_t rows, int64_t K);

/* Workspace bytes h3fp4_linear needs for (M, N, K, flags); also enough for
 * h3fp4_quantize_act / h3fp4_quantize_weight of M (or N) rows.  Holds the
 * device status word, the amax partial maxima and, unless A_PREQUANT, the
 * activation's codes, block scales, global scale and (H3FP4_FUSED_QUANT)
 * the ready flags of its tiles.  Zero the workspace (at least the status word,
 * its first 256 bytes, and the flags) once before first use, and write it
 * with nothing but this library afterwards: the flags hold call numbers that
 * never repeat within a process.  Concurrent calls must not share one
 * workspace. */
H3FP4_API size_t h3fp4_workspace_bytes(int64_t M, int64_t N, int64_t K, int flags);

/* Quantise a weight W [N, K] bf16 to NVFP4 (offline step; same algorithm as
 * the activations, no prologue).  Passage: "H3 Blackwell Runtime" README,
 * "Checkpoints" (pre-quantised NVFP4 weights, not converted at run time);
 * the format as in h3fp4_quantize_act.  Writes codes [N][K/2], sf
 * (h3fp4_sf_bytes(N, K)) and *w_gscale (device).  ws: h3fp4_workspace_bytes
 * (N, 0, K, 0) bytes. */
H3FP4_API h3fp4_status h3fp4_quantize_weight(const void* w_bf16, int64_t N, int64_t K,
                                   void* codes, void* sf, float* w_gscale,
                                   void* ws, cudaStream_t stream);

/* Quantise an activation X [M, K] bf16.  Passages: "H3 Runtime Current
 * State", "Owned Performance Kernels" (scale discovery then pack into
 * QDATA + swizzled block scales; one full-activation scale; modulation fed
 * into scale/pack as exact BF16 values) and "H3 Blackwell Runtime Plan",
 * "Next Performance Plan: Blackwell NVFP4 GEMMs" (signed zero, tie-to-even FP4
 * rounding, cuBLAS tiled block-scale layout).
 *   shift, scale: fp32 [nseg][K] (device), required with H3FP4_PROLOGUE_MOD.
 *   seg_off: HOST array of nseg + 1 row offsets, seg_off[0] = 0,
 *            non-decreasing, seg_off[nseg] = M; NULL means one segment.
 *            1 <= nseg <= H3FP4_MAX_SEGMENTS.
 *   flags: H3FP4_PROLOGUE_MOD, H3FP4_GSCALE_GIVEN (then *gscale is an input;
 *          otherwise it is written with amax/(6*448) over all segments).
 *   codes [M][K/2], sf (h3fp4_sf_bytes(M, K)), gscale: device outputs. */
H3FP4_API h3fp4_status h3fp4_quantize_act(const void* x_bf16, int64_t M, int64_t K,
                                const float* shift, const float* scale,
                                const int64_t* seg_off, int nseg,
                                void* codes, void* sf, float* gscale,
                                int flags, void* ws, cudaStream_t stream);

/* The NVFP4 linear: out[M][N] (bf16) from X and a quantised weight.
 * Passages: "H3 Runtime Current State", "Owned Performance Kernels" (the
 * block-scaled NVFP4 GEMM of the four projections, alpha applied before the
 * BF16 cast, gate/add epilogue; removing intermediate traffic across the
 * scale/pack/GEMM boundaries) and "Implemented And Validated" (fused
 * modulation and residual gates over packed video+audio tokens).
 *   x: bf16 [M][K], or codes [M][K/2] with H3FP4_A_PREQUANT (then a_sf and
 *      a_gscale describe it).  With H3FP4_GSCALE_GIVEN a_gscale (device) is
 *      the activation global scale; otherwise it may be NULL and the scale is
 *      computed (one amax over all rows and segments).
 *   w_codes/w_sf/w_gscale: output of h3fp4_quantize_weight.
 *   shift/scale: as in h3fp4_quantize_act (with H3FP4_PROLOGUE_MOD).
 *   gate: fp32 [nseg][N] and resid: bf16 [M][N], with H3FP4_EPI_GATE_RESID.
 *   bias: bf16 [N], with H3FP4_EPI_BIAS.
 *   out may not alias x, resid or the weights.
 *
 * SwiGLU producer (H3FP4_EPI_SWIGLU; "H3 Runtime Current State", "Owned
 * Performance Kernels": the exact SwiGLU-to-FC2 NVFP4 producer fusion that
 * keeps the two reference BF16 boundaries).  N % 256 == 0, and the weight
 * rows (and bias) come in groups of 256: rows [256 t, 256 t + 128) are the
 * gate rows and rows [256 t + 128, 256 t + 256) the up rows of hidden units
 * [128 t, 128 t + 128).  With g, u the bf16 outputs the plain epilogue would
 * write for a gate and its up row (the FC1 output boundary),
 *     out[m][128 t + i] = bf16(silu(g) * u),  silu(g) = g / (1 + e^-g),
 * evaluated in fp32 from the hardware's approximate 2^x and 1/x in a form that
 * cannot overflow (within one bf16 step of the exact value for every bf16 g);
 * out is [M][N/2].  Not with
 * H3FP4_EPI_GATE_RESID.
 *
 * Output amax (H3FP4_EPI_AMAX; "H3 Blackwell Runtime Plan", "Next Performance
 * Plan: Blackwell NVFP4 GEMMs": scale discovery): the call also stores
 * max |out| over all M rows of its bf16 output, as fp32, at
 * h3fp4_ws_out_amax(ws).  A following h3fp4_gscale_from_amax and
 * H3FP4_GSCALE_GIVEN quantisation of `out` (no prologue) then produce the
 * same codes, block scales and global scale as the two-pass quantisation,
 * with one pass over `out` instead of two.
 *
 * Quantise-once producer (H3FP4_FUSED_QUANT; "H3 Runtime Current State",
 * "Owned Performance Kernels": a producer that quantises each (M, K) tile
 * once and shares it across the N consumers, with one full-activation
 * scale): the GEMM kernel's packer warps quantise x tile by tile (128 rows x
 * 256 columns) into the workspace while the same kernel's GEMM consumes the
 * tiles, each behind a ready flag it waits for (bounded; a timeout is
 * reported by h3fp4_check).  With the computed scale an amax pass runs
 * first; with H3FP4_GSCALE_GIVEN the GEMM kernel is the only launch.  Codes,
 * block scales, global scale and out are the bytes of the two-pass path.
 * Not with H3FP4_A_PREQUANT or H3FP4_EPI_SWIGLU; K <= 16384; not on a stream
 * being captured into a CUDA graph (H3FP4_ERR_INVALID: the flags hold a call
 * number fixed at launch, which a replayed launch would repeat). */
H3FP4_API h3fp4_status h3fp4_linear(const void* x, const void* a_sf, const float* a_gscale,
                          int64_t M, int64_t N, int64_t K,
                          const void* w_codes, const void* w_sf, const float* w_gscale,
                          const float* shift, const float* scale, const float* gate,
                          const int64_t* seg_off, int nseg,
                          const void* bias_bf16, const void* resid_bf16, void* out_bf16,
                          int flags, void* ws, cudaStream_t stream);

/* FC1 with the SwiGLU producer writing h straight to NVFP4: the FC2 operand
 * leaves the FC1 epilogue as codes and block scales, so h is never stored in
 * bf16 and FC2 needs no quantisation pass ("H3 Runtime Current State", "Owned
 * Performance Kernels": the exact SwiGLU-to-FC2 NVFP4 producer fusion that
 * emits tensor scale/QDATA/SFA).
 *   Arguments as in h3fp4_linear with H3FP4_EPI_SWIGLU (N % 256 == 0, the
 *   weight's [gate 128 | up 128] row groups); flags: H3FP4_PROLOGUE_MOD,
 *   H3FP4_EPI_BIAS, H3FP4_GSCALE_GIVEN, H3FP4_A_PREQUANT (the activation x).
 *   h_gscale: device fp32 > 0, the global scale of h, an INPUT (for instance
 *   h3fp4_gscale_from_amax of the EPI_AMAX output of an earlier call, or a
 *   calibrated scale).  h_codes [M][N/4] bytes and h_sf
 *   (h3fp4_sf_bytes(M, N/2)) receive exactly what
 *   h3fp4_quantize_act(h, ..., H3FP4_GSCALE_GIVEN with *h_gscale) would write
 *   for the bf16 h that h3fp4_linear's SwiGLU epilogue stores; a following
 *   h3fp4_linear with H3FP4_A_PREQUANT (a_sf = h_sf, a_gscale = h_gscale)
 *   consumes them.  h_codes may not alias x or the weights. */
H3FP4_API h3fp4_status h3fp4_linear_swiglu_nvfp4(const void* x, const void* a_sf, const float* a_gscale,
                                    int64_t M, int64_t N, int64_t K,
                                    const void* w_codes, const void* w_sf, const float* w_gscale,
                                    const float* shift, const float* scale,
                                    const int64_t* seg_off, int nseg, const void* bias_bf16,
                                    const float* h_gscale, void* h_codes, void* h_sf,
                                    int flags, void* ws, cudaStream_t stream);

/* Quantise an activation exactly like h3fp4_quantize_act, but without a
 * workspace and without allocating anything, for callers that are handed only
 * their input and output buffers: for example a plugin whose host application
 * owns all device memory and gives it no workspace, or a serving loop that
 * forbids device allocation once it runs (cudaMalloc/cudaFree can synchronise
 * the device and fragment a pool another allocator manages).  The pages have
 * no counterpart for this entry point; it is a convenience of this library.
 *   Scratch: the amax partial maxima live in a static device array of the
 *   library (4096 fp32 = 16 KiB), held by every GPU that loads the library
 *   until the process exits.  The first call on a device looks up the array's
 *   device address (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture.  The address is cached per device
 *   for the life of the process (a failed look-up is retried by the next
 *   call); cudaDeviceReset reloads the library's device code, so a process
 *   that resets a device must not call this entry point on it afterwards.
 *   All calls share the array: calls that can overlap on the GPU (several
 *   streams or host threads) race on it and must be serialised by the caller.
 *   Limit: K <= 4096 * 1024 columns (one partial per 1024-column slab at
 *   least); larger K returns H3FP4_ERR_SHAPE.
 *   Other arguments, results and errors as in h3fp4_quantize_act. */
H3FP4_API h3fp4_status h3fp4_quantize_act_noalloc(const void* x_bf16, int64_t M, int64_t K,
                                                  const float* shift, const float* scale,
                                                  const int64_t* seg_off, int nseg,
                                                  void* codes, void* sf, float* gscale,
                                                  int flags, cudaStream_t stream);

/* Amax of the (modulated) activation rows of this call -> *amax (device fp32).
 * Building block of the multi-device split of one activation along M (token
 * rows, "H3 Runtime Current State", "Distributed Execution": sequence-sharded
 * execution): every device computes the amax of its rows, the caller
 * max-reduces the per-device values (one fp32 all-reduce(MAX)), turns the
 * result into the global scale with h3fp4_gscale_from_amax and quantises its
 * rows with H3FP4_GSCALE_GIVEN.  The codes and block scales are then
 * bit-identical to a single-device quantisation of the whole tensor.
 * Arguments as in h3fp4_quantize_act (flags: H3FP4_PROLOGUE_MOD only). */
H3FP4_API h3fp4_status h3fp4_act_amax(const void* x_bf16, int64_t M, int64_t K,
                                      const float* shift, const float* scale,
                                      const int64_t* seg_off, int nseg,
                                      float* amax, int flags, void* ws, cudaStream_t stream);

/* Device address inside the workspace where an H3FP4_EPI_AMAX call of
 * h3fp4_linear leaves max|out| (fp32); valid until the workspace's next
 * EPI_AMAX call.  NULL for a NULL workspace.  No device access. */
H3FP4_API float* h3fp4_ws_out_amax(void* ws);

/* *gscale = (*amax == 0) ? 1 : *amax / (6*448), on the device (one thread). */
H3FP4_API h3fp4_status h3fp4_gscale_from_amax(const float* amax, float* gscale, cudaStream_t stream);

/* Failure-detection self-test: runs the GEMM kernel on a dummy 128x256x256
 * problem with its TMA producer disabled, so every consumer wait must run out
 * after limit_ns; the kernel then records the timeout in the status word of
 * `ws` (h3fp4_workspace_bytes(128, 256, 256, 0) bytes), frees
 * its TMEM and returns.  h3fp4_check(ws) must afterwards report
 * H3FP4_ERR_TIMEOUT.  No data is read or written besides the status word. */
H3FP4_API h3fp4_status h3fp4_selftest_timeout(void* ws, uint64_t limit_ns, cudaStream_t stream);

/* The same for the quantise-once producer's ready flags: the fused GEMM
 * (H3FP4_FUSED_QUANT, given scale *a_gscale) on a 128x256x256 problem whose
 * packer quantises x (bf16 [128][256], device) into the workspace but
 * publishes no tile, so the GEMM's waits for the tiles run out after
 * limit_ns and the kernel returns.  ws: h3fp4_workspace_bytes(128, 256, 256,
 * 0) bytes; h3fp4_check(ws) must afterwards report H3FP4_ERR_TIMEOUT. */
H3FP4_API h3fp4_status h3fp4_selftest_pack_timeout(const void* x_bf16, const float* a_gscale, void* ws,
                                                   uint64_t limit_ns, cudaStream_t stream);

/* Measured tensor-core ceiling for the GEMM's instruction on the current
 * device: back-to-back tcgen05.mma.kind::mxf4nvf4.block_scale (M=128, N=256,
 * K=64) on every SM with operands resident in shared memory and scales in
 * TMEM (no global traffic), `iters` MMAs per SM (e.g. 20000).  Synchronous
 * (default stream); writes TFLOP/s to *tflops.  ws: any workspace (status
 * word only).  The roofline reports of the benchmark quote this beside the
 * nominal dense FP4 figure. */
H3FP4_API h3fp4_status h3fp4_measure_fp4_peak(int iters, float* tflops, void* ws);

/* The same ceiling for the paired form the GEMM issues:
 * tcgen05.mma.cta_group::2 (M=256 over a 2-CTA cluster, N=256, K=64), `iters`
 * MMAs by the leader of every cluster that fits on the device (synchronous,
 * default stream).  Writes TFLOP/s to *tflops; ws: any workspace (status word
 * only).  No counterpart in the pages: it measures this GPU. */
H3FP4_API h3fp4_status h3fp4_measure_fp4_pair_peak(int iters, float* tflops, void* ws);

/* The tcgen05 forms of the NVFP4 block-scaled MMA (kind::mxf4nvf4,
 * scale_vec::4X: E2M1 operands, 16-element blocks with E4M3 scales -- the only
 * kind that carries NVFP4) that h3fp4_measure_fp4_form can time. */
typedef enum {
    H3FP4_MMA_SINGLE = 0,                 /* cta_group::1, M=128, N=256, K=64, A in shared memory */
    H3FP4_MMA_PAIR = 1,                   /* cta_group::2, M=256, N=256, K=64 (the GEMM's form)     */
    H3FP4_MMA_SINGLE_TMEM_A = 2,          /* cta_group::1 with A read from TMEM                     */
    H3FP4_MMA_PAIR_TMEM_A = 3,            /* cta_group::2 with A read from TMEM                     */
    H3FP4_MMA_SINGLE_N128 = 4,            /* cta_group::1, two N=128 MMAs per K step sharing A      */
    H3FP4_MMA_SINGLE_N128_COLLECTOR = 5,  /* the same through .collector::a::fill / ::lastuse       */
    H3FP4_MMA_PAIR_N128 = 6               /* cta_group::2, two N=128 MMAs per K step sharing A      */
} h3fp4_mma_form;

/* Measured ceiling (TFLOP/s, synchronous) of one MMA form, issued back to back
 * by one thread per CTA (or CTA pair) on every SM with operands and scales
 * resident on chip; flops counted as 2 * 128 * 256 * 64 per CTA per K step.
 * Entry point for roofline evidence only; no counterpart on the pages. */
H3FP4_API h3fp4_status h3fp4_measure_fp4_form(int form, int iters, float* tflops, void* ws);

/* Synchronises `stream`, reads and clears the workspace status word.
 * Returns H3FP4_OK, or H3FP4_ERR_TIMEOUT when a kernel gave up early (a
 * bounded device wait ran out, or shared memory came up misaligned); the
 * outputs of that call are then undefined. */
H3FP4_API h3fp4_status h3fp4_check(void* ws, cudaStream_t stream);

/* Maximum wait of every device-side spin in nanoseconds (default 2e9).
 * Process-wide; meant for tests of the timeout path. */
H3FP4_API void h3fp4_set_wait_limit_ns(uint64_t ns);

/* Human-readable status. */
H3FP4_API const char* h3fp4_status_string(h3fp4_status s);

#ifdef __cplusplus
}
#endif
#endif /* H3FP4_H */
