/*
 * h3fp4 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct restatement of the NVFP4 linear path that
 * the H3 Blackwell Runtime pages describe: optional AdaLN modulation, one
 * full-activation global scale, per-16-element E4M3 block scales in the
 * tiled/swizzled layout the block-scaled MMA consumes, round-to-nearest-even
 * E2M1 codes packed two per byte, a float64 GEMM on the dequantised operands
 * and the bias + residual-gate epilogue.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The product path (the CUDA library) shares no code
 * with it.
 *
 * Sources (page title / section):
 *   [CS]   "H3 Runtime Current State", section "Owned Performance Kernels"
 *          (block-scale swizzle at every projection width; tensor
 *          scale/QDATA/SFA; alpha applied before the BF16 cast; one
 *          full-activation scale for the packed ring; modulation values fed
 *          as exact BF16 into scale/pack).
 *   [PLAN] "H3 Blackwell Runtime Plan", section "Next Performance Plan:
 *          Blackwell NVFP4 GEMMs" (qdata, cuBLAS tiled block-scale layout,
 *          signed zero, tie-to-even FP4 rounding; modulation kept in BF16).
 *   [FMT]  The NVFP4 format: E2M1 elements with magnitudes
 *          {0, 0.5, 1, 1.5, 2, 3, 4, 6}, E4M3 ("fn": bias 7, no infinity,
 *          0x7F/0xFF NaN, maximum 448) block scales over 16 elements, and an
 *          fp32 global scale amax / (6 * 448).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   R1 encode order: S = e4m3((bmax / 6) / s_g); eff = S * s_g;
 *      r = 1 / eff; q = e2m1(m * r), every step one IEEE fp32 RN operation.
 *   R2 the modulated value is rounded to bf16 before quantisation; the
 *      modulation itself is one fp32 fma: m = bf16(fma(x, 1 + scale, shift)).
 *   R3 s_g = amax / 2688 (fp32 RN); an all-zero tensor gets s_g = 1.
 *   R4 E2M1 and E4M3 round to nearest, ties to the even code, and saturate
 *      to the largest finite value; the E2M1 sign bit is copied from the
 *      input, so negative values that round to zero give -0 (code 8).
 *   R5 eff == 0 gives r = 0 (all codes +-0); 1/eff is clamped to FLT_MAX so
 *      that a block of tiny values cannot form 0 * inf.
 *   R6 nibble order: element 2j in bits 0-3, element 2j+1 in bits 4-7; the
 *      block-scale byte for (row r, block c) sits at
 *      ((r/128)*Kb4 + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *      Kb4 = ceil(K/64); padding bytes are zero.
 *   R7 segments: rows [seg_off[i], seg_off[i+1]) use shift/scale/gate row i.
 *   R8 SwiGLU producer ([CS], the exact SwiGLU-to-FC2 producer fusion that
 *      keeps the two reference BF16 boundaries): the gate value g and the up
 *      value u are the bf16 FC1 outputs; h = bf16(silu(g) * u) with
 *      silu(g) = g / (1 + e^-g), one rounding to bf16 of the real value.
 *
 * Build: gcc -std=c11 -O2 -fno-fast-math -ffp-contract=off -fopenmp
 *        -shared -fPIC  (strict IEEE fp32, no fused multiply-add contraction).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                        */
/* ------------------------------------------------------------------ */

static inline float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static inline uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the top half of an fp32; round to nearest, ties to even.
 * Inputs are finite by precondition (the path is defined on finite data). */
ORC_API uint16_t orc_bf16_from_float(float f)
{
    uint32_t u = bits_from_f32(f);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

ORC_API float orc_bf16_to_float(uint16_t h) { return f32_from_bits(((uint32_t)h) << 16); }

/* ------------------------------------------------------------------ */
/* E2M1 [FMT]: 1 sign, 2 exponent (bias 1), 1 mantissa, no inf/NaN.    */
/* ------------------------------------------------------------------ */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

ORC_API double orc_e2m1_decode(uint8_t c)
{
    double v = E2M1_MAG[c & 7u];
    return (c & 8u) ? -v : v;
}

/* Nearest grid magnitude by explicit distance; on a tie the even code wins;
 * values beyond 6 land on 6 because 6 is the nearest grid point (saturate).
 * The sign bit is copied from the input (signed zero, [PLAN]). */
ORC_API uint8_t orc_e2m1_encode(float f)
{
    double a = fabs((double)f);
    int best = 0;
    double bestd = a; /* distance to magnitude 0 */
    /* Above 6 the nearest grid point is 6; handled first because for huge a
     * the double distances |a - 6| and |a - 0| round to the same value. */
    if (a >= 6.0) {
        best = 7;
        bestd = 0.0;
    }
    for (int c = 1; c < 8 && best != 7; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < bestd || (d == bestd && (c % 2 == 0) && (best % 2 != 0))) {
            best = c;
            bestd = d;
        }
    }
    uint8_t sign = signbit(f) ? 8u : 0u;
    return (uint8_t)(sign | (uint8_t)best);
}

/* ------------------------------------------------------------------ */
/* E4M3 "fn" [FMT]: bias 7, subnormals, 0x7F/0xFF NaN, max 448.        */
/* ------------------------------------------------------------------ */

ORC_API double orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return s ? -v : v;
}

/* Non-negative finite input only (block maxima are non-negative).
 * Round to nearest on the E4M3 grid, ties to even mantissa, saturate to 448. */
ORC_API uint8_t orc_e4m3_encode(float f)
{
    double a = (double)f;
    if (!(a >= 0.0)) return 0x7Fu; /* precondition violated: NaN code */
    if (a >= 448.0) return 0x7Eu;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: integer multiple of 2^-9, half-even; 8 -> min normal */
        double q = rint(a * 512.0); /* exact scaling; rint is half-even */
        return (uint8_t)q;          /* 0..8; code 8 is 2^-6 */
    }
    int ex;
    (void)frexp(a, &ex);            /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;                 /* a in [2^E, 2^(E+1)) */
    double n = rint(ldexp(a, 3 - E)); /* mantissa in units of 2^(E-3): [8, 16] */
    if (n == 16.0) { E += 1; n = 8.0; }
    int code = ((E + 7) << 3) | ((int)n - 8);
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)code;
}

ORC_API void orc_e2m1_encode_array(const float* x, int64_t n, uint8_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(x[i]);
}

ORC_API void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------ */
/* Block-scale layout (R6, [PLAN] "cuBLAS tiled block-scale layout",    */
/* [CS] "generalizing the block-scale swizzle").                        */
/* ------------------------------------------------------------------ */

ORC_API int64_t orc_sf_cols4(int64_t K) { return (K / 16 + 3) / 4; }

ORC_API int64_t orc_sf_bytes(int64_t rows, int64_t K)
{
    return ((rows + 127) / 128) * 128 * orc_sf_cols4(K) * 4;
}

ORC_API int64_t orc_sf_offset(int64_t r, int64_t c, int64_t K)
{
    int64_t kb4 = orc_sf_cols4(K);
    return ((r / 128) * kb4 + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* ------------------------------------------------------------------ */
/* Modulation prologue (R2, R7; [CS] modulation fused into scale/pack,  */
/* exact BF16 values; [PLAN] modulation stays BF16).                    */
/* ------------------------------------------------------------------ */

static int seg_of_row(int64_t r, const int64_t* seg_off, int nseg)
{
    for (int i = 0; i < nseg; ++i)
        if (r >= seg_off[i] && r < seg_off[i + 1]) return i;
    return nseg - 1;
}

static inline uint16_t modulate_one(uint16_t x, float sh, float sc)
{
    float one_plus = 1.0f + sc;                 /* fp32 RN */
    float v = fmaf(orc_bf16_to_float(x), one_plus, sh); /* one rounding */
    return orc_bf16_from_float(v);
}

/* m[r][k] = bf16(fma(x, 1 + scale[seg][k], shift[seg][k])); without
 * vectors (shift == NULL) m = x. */
ORC_API void orc_modulate(const uint16_t* x, int64_t M, int64_t K,
                          const float* shift, const float* scale,
                          const int64_t* seg_off, int nseg, uint16_t* m)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        if (!shift) {
            memcpy(m + r * K, x + r * K, (size_t)K * 2);
            continue;
        }
        int s = seg_of_row(r, seg_off, nseg);
        for (int64_t k = 0; k < K; ++k)
            m[r * K + k] = modulate_one(x[r * K + k], shift[s * K + k], scale[s * K + k]);
    }
}

/* ------------------------------------------------------------------ */
/* Global scale (R3; [CS] "one full-activation scale")                 */
/* ------------------------------------------------------------------ */

ORC_API float orc_amax(const uint16_t* m, int64_t n)
{
    float best = 0.0f;
#pragma omp parallel for reduction(max : best) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(orc_bf16_to_float(m[i]));
        if (a > best) best = a;
    }
    return best;
}

ORC_API float orc_global_scale(float amax)
{
    if (amax == 0.0f) return 1.0f;
    return amax / 2688.0f; /* 6 * 448 */
}

/* ------------------------------------------------------------------ */
/* Block quantiser (R1, R4, R5).                                        */
/* ------------------------------------------------------------------ */

/* One 16-element block: returns the E4M3 scale code, writes 16 E2M1 codes. */
ORC_API uint8_t orc_quantize_block(const float* m16, float s_g, uint8_t* q16)
{
    float bmax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(m16[i]);
        if (a > bmax) bmax = a;
    }
    float t = bmax / 6.0f;
    t = t / s_g;
    uint8_t S = orc_e4m3_encode(t);
    float eff = (float)orc_e4m3_decode(S) * s_g;
    float r = 0.0f;
    if (eff != 0.0f) {
        r = 1.0f / eff;
        if (r > FLT_MAX) r = FLT_MAX;
    }
    for (int i = 0; i < 16; ++i) q16[i] = orc_e2m1_encode(m16[i] * r);
    return S;
}

/* Full quantisation of a [rows, K] bf16 operand (K % 16 == 0).
 *   shift/scale: [nseg][K] fp32 or NULL (no modulation)
 *   gscale: in/out; if gscale_given, *gscale is used, else it is computed.
 *   codes: [rows][K/2] bytes; sf: orc_sf_bytes(rows, K) bytes (zeroed here). */
ORC_API void orc_quantize(const uint16_t* x, int64_t rows, int64_t K,
                          const float* shift, const float* scale,
                          const int64_t* seg_off, int nseg,
                          int gscale_given, float* gscale,
                          uint8_t* codes, uint8_t* sf)
{
    uint16_t* m = (uint16_t*)malloc((size_t)(rows * K) * 2);
    orc_modulate(x, rows, K, shift, scale, seg_off, nseg, m);
    float s_g = gscale_given ? *gscale : orc_global_scale(orc_amax(m, rows * K));
    *gscale = s_g;
    memset(sf, 0, (size_t)orc_sf_bytes(rows, K));
    int64_t nblk = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float mf[16];
        uint8_t q[16];
        for (int64_t c = 0; c < nblk; ++c) {
            for (int i = 0; i < 16; ++i) mf[i] = orc_bf16_to_float(m[r * K + c * 16 + i]);
            uint8_t S = orc_quantize_block(mf, s_g, q);
            sf[orc_sf_offset(r, c, K)] = S;
            for (int j = 0; j < 8; ++j)
                codes[r * (K / 2) + c * 8 + j] = (uint8_t)((q[2 * j] & 15u) | ((q[2 * j + 1] & 15u) << 4));
        }
    }
    free(m);
}

/* Exact dequantisation to float64 (at most 2 + 4 + 24 significant bits). */
ORC_API void orc_dequantize(const uint8_t* codes, const uint8_t* sf, float gscale,
                            int64_t rows, int64_t K, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = codes[r * (K / 2) + k / 2];
            uint8_t q = (k % 2 == 0) ? (byte & 15u) : (byte >> 4);
            double S = orc_e4m3_decode(sf[orc_sf_offset(r, k / 16, K)]);
            out[r * K + k] = orc_e2m1_decode(q) * S * (double)gscale;
        }
}

/* ------------------------------------------------------------------ */
/* SwiGLU at the FC1 -> FC2 boundary (R8).                              */
/* ------------------------------------------------------------------ */

/* Round a finite double d to the nearest bf16 (8 significant bits;
 * subnormals on the 2^-133 grid; overflow past the largest finite bf16 gives
 * infinity, as in fp32 -> bf16).  `dir` is the sign of (true value - d) when d
 * is only the leading part of the value being rounded: an exact midpoint then
 * goes to the side the true value lies on; with dir = 0 ties go to even. */
static uint16_t bf16_round(double d, int dir)
{
    uint16_t sign = signbit(d) ? 0x8000u : 0u;
    double a = fabs(d);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                /* quantum of an 8-bit significand */
    if (q < -133) q = -133;       /* bf16 subnormal spacing */
    double x = ldexp(a, -q);      /* exact: the bf16 grid becomes the integers */
    double n = nearbyint(x);      /* default rounding mode: nearest, ties to even */
    if (dir != 0 && x - floor(x) == 0.5) {
        int up = (dir > 0) == (sign == 0);  /* the true magnitude lies above a */
        n = up ? ceil(x) : floor(x);
    }
    float r = (float)ldexp(n, q); /* exact in fp32 unless it overflows */
    return (uint16_t)(sign | (bits_from_f32(r) >> 16));
}

ORC_API uint16_t orc_swiglu_bf16(uint16_t g, uint16_t u)
{
    double gd = (double)orc_bf16_to_float(g), ud = (double)orc_bf16_to_float(u);
    if (fabs(gd) < 0x1p-30) {
        /* silu(g) = g/2 + g^2/4 + O(g^4).  (g/2) * u is exact in double (two
         * 8-bit significands); the remainder (g^2/4) * u is far below every
         * bf16 spacing but has the sign of u, which decides exact midpoints. */
        int dir = (gd == 0.0 || ud == 0.0) ? 0 : (ud > 0.0 ? 1 : -1);
        return bf16_round(0.5 * gd * ud, dir);
    }
    double silu = gd / (1.0 + exp(-gd));
    return bf16_round(silu * ud, 0);
}

/* silu(g) * u for real-valued g, u, in float64 with no rounding to bf16: the
 * value the SwiGLU producer rounds (R8), here taken at the unrounded float64
 * FC1 outputs, so that an end-to-end bound can be stated around it.  Small |g|
 * uses silu(g) = g/2 + g^2/4 + O(g^4), where g / (1 + e^-g) would lose the
 * g^2 term to rounding. */
ORC_API void orc_silu_mul_f64(const double* g, const double* u, int64_t n, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double gd = g[i];
        double silu = fabs(gd) < 0x1p-20 ? 0.5 * gd + 0.25 * gd * gd : gd / (1.0 + exp(-gd));
        out[i] = silu * u[i];
    }
}

/* Elementwise over an FC1 output in the SwiGLU row layout: y [rows][2*H] holds,
 * for every group t of 128 hidden units, the 128 gate columns [256 t, 256 t + 128)
 * followed by the matching 128 up columns; h [rows][H]. */
ORC_API void orc_swiglu_rows(const uint16_t* y, int64_t rows, int64_t H, uint16_t* h)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < H; ++j) {
            int64_t t = j / 128, i = j % 128;
            h[r * H + j] = orc_swiglu_bf16(y[r * 2 * H + 256 * t + i], y[r * 2 * H + 256 * t + 128 + i]);
        }
}

/* ------------------------------------------------------------------ */
/* GEMM + epilogue in float64 ([CS] alpha before the BF16 cast;        */
/* [CS] "Implemented And Validated": fused residual gates).            */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint8_t *a_codes, *a_sf;
    float a_gs;
    const uint8_t *w_codes, *w_sf;
    float w_gs;
    int64_t M, N, K;
    const uint16_t* bias;   /* bf16 [N] or NULL */
    const float* gate;      /* fp32 [nseg][N] or NULL */
    const uint16_t* resid;  /* bf16 [M][N] or NULL (required with gate) */
    const int64_t* seg_off; /* nseg + 1 entries (host) */
    int nseg;
} orc_linear_args;

static inline double deq_elem(const uint8_t* codes, const uint8_t* sf, int64_t r, int64_t k, int64_t K)
{
    uint8_t byte = codes[r * (K / 2) + k / 2];
    uint8_t q = (k % 2 == 0) ? (byte & 15u) : (byte >> 4);
    return orc_e2m1_decode(q) * orc_e4m3_decode(sf[orc_sf_offset(r, k / 16, K)]);
}

/* One output element: out = R + g*(alpha*acc + b) (or alpha*acc + b), plus
 * the error bound 2^-8*|out| + 1e-5*|g|*sum_k|a_k*w_k| (g = 1 without gate). */
static void linear_point(const orc_linear_args* A, int64_t m, int64_t n, double* out, double* bound)
{
    int64_t K = A->K;
    double acc = 0.0, absacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = deq_elem(A->a_codes, A->a_sf, m, k, K) * deq_elem(A->w_codes, A->w_sf, n, k, K);
        acc += p;
        absacc += fabs(p);
    }
    double alpha = (double)A->a_gs * (double)A->w_gs;
    double y = alpha * acc;
    double b = A->bias ? (double)orc_bf16_to_float(A->bias[n]) : 0.0;
    double v = y + b;
    double g = 1.0, o = v;
    if (A->gate) {
        int s = seg_of_row(m, A->seg_off, A->nseg);
        g = (double)A->gate[(int64_t)s * A->N + n];
        double R = A->resid ? (double)orc_bf16_to_float(A->resid[m * A->N + n]) : 0.0;
        o = R + g * v;
    }
    *out = o;
    *bound = ldexp(fabs(o), -8) + 1e-5 * fabs(g) * fabs(alpha) * absacc;
}

ORC_API void orc_linear_points(const orc_linear_args* A, const int64_t* mn, int64_t npts,
                               double* out, double* bound)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < npts; ++i) linear_point(A, mn[2 * i], mn[2 * i + 1], out + i, bound + i);
}

/* Every output element, by the definition (row-parallel, plain loops). */
ORC_API void orc_linear_full(const orc_linear_args* A, double* out, double* bound)
{
    int64_t M = A->M, N = A->N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) linear_point(A, m, n, out + m * N + n, bound + m * N + n);
}

/* Plain float64 GEMM on already-dequantised operands: C = A * W^T
 * (used by the pins against a library dgemm). */
ORC_API void orc_gemm_f64(const double* a, const double* w, int64_t M, int64_t N, int64_t K, double* c)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += a[m * K + k] * w[n * K + k];
            c[m * N + n] = acc;
        }
}

ORC_API int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
