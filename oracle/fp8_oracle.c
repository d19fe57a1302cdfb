/*
 * fp8_oracle.c -- plain, slow CPU oracle for the FP8 scaling/quantisation/GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no source with the CUDA path.
 *
 * Every function is the definition of what it computes, written out with no
 * blocking, fusion or reordering beyond that definition:
 *
 *  - FP8 codec (decode/encode).  The pages name the two formats only as
 *    "FP8_E4" (weights, activations) and "FP8_E5" (gradients)
 *    ("Training and inference of large language models using 8-bit floating
 *    point", section "Proposed method").  They are read as the OFP8 encodings
 *    E4M3 (bias 7, no infinities, NaN = S.1111.111, max 448) and E5M2 (bias 15,
 *    IEEE-like, max 57344).  Encoding is round-to-nearest-even followed by
 *    saturation to the largest finite magnitude, done by exact comparison with
 *    the midpoints between neighbouring representable values.
 *
 *  - compute_bias: the per-tensor exponent bias is floor(log2(fmax/amax)) minus
 *    a margin (same page, "Proposed method": the bias is the base-2 logarithm
 *    of the format maximum over the tensor's amax, less a margin).
 *
 *  - quantise: scale before the cast (same page, "Proposed method"): q =
 *    Encode(x * 2^e), the product taken in fp32, the precision of the kernels.
 *    Per-block scaling gives each block its own e from its own amax
 *    ("Per-Tensor and Per-Block Scaling Strategies for Effective FP8 Training",
 *    "Key Questions Answered": per-block scaling and MXFP8).  The column-wise
 *    copy is the row-wise quantisation of the transposed matrix.
 *
 *  - delayed scaling: the scale for the next step comes from the maximum of the
 *    amax values recorded over the last L steps (first page, "Key Questions
 *    Answered": the delayed scale looks back over a window of past steps).
 *
 *  - GEMM: the exact fp64 product of the dequantised operands: the FP8 product
 *    is unscaled after the multiplication (second page, "Proposed method").
 *
 * Compile with -ffp-contract=off and without -ffast-math.
 */
#include <stdint.h>
#include <math.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FMT_E4M3 0
#define FMT_E5M2 1

#define GRAN_TENSOR 0
#define GRAN_1x128 1
#define GRAN_128x128 2
#define GRAN_MX32 3
#define GRAN_MX32_OCP 4 /* 1x32 blocks, E8M0, the OCP MX bias rule */

/* ------------------------------------------------------------------ formats */

static int fmt_mbits(int fmt) { return fmt == FMT_E4M3 ? 3 : 2; }
static int fmt_ebits(int fmt) { return fmt == FMT_E4M3 ? 4 : 5; }
static int fmt_bias(int fmt) { return fmt == FMT_E4M3 ? 7 : 15; }
/* largest finite positive code: E4M3 0.1111.110 = 448, E5M2 0.11110.11 = 57344 */
static int fmt_maxcode(int fmt) { return fmt == FMT_E4M3 ? 0x7E : 0x7B; }

int fp8o_maxcode(int fmt) { return fmt_maxcode(fmt); }

/* Textbook decode: (-1)^s 2^(E-bias) (1 + m/2^M) for normals,
 * (-1)^s 2^(1-bias) (m/2^M) for subnormals. */
double fp8o_decode(int code, int fmt)
{
    int s = (code >> 7) & 1;
    int mb = fmt_mbits(fmt), eb = fmt_ebits(fmt), bias = fmt_bias(fmt);
    int E = (code >> mb) & ((1 << eb) - 1);
    int m = code & ((1 << mb) - 1);
    double v;
    if (fmt == FMT_E4M3) {
        if (E == 15 && m == 7) return NAN;
    } else {
        if (E == 31) {
            if (m == 0) return s ? -INFINITY : INFINITY;
            return NAN;
        }
    }
    if (E == 0)
        v = ldexp((double)m, 1 - bias - mb);
    else
        v = ldexp((double)((1 << mb) + m), E - bias - mb);
    return s ? -v : v;
}

/* magnitudes of the non-negative finite codes 0..maxcode, increasing */
static double g_mag[2][128];

__attribute__((constructor)) static void fp8o_init_tables(void)
{
    for (int f = 0; f < 2; ++f)
        for (int c = 0; c <= fmt_maxcode(f); ++c) g_mag[f][c] = fp8o_decode(c, f);
}

/* Encode(v): round to nearest representable value, ties to the code whose
 * mantissa LSB is 0 (the code LSB), then saturate to +-fmax.  Clamping first is
 * the same thing because fmax itself is representable.  NaN maps to the NaN
 * code 0x7F (E4M3 S.1111.111, E5M2 S.11111.11). */
int fp8o_encode(float v, int fmt)
{
    if (isnan(v)) return 0x7F;
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    int maxc = fmt_maxcode(fmt);
    const double *t = g_mag[fmt];
    if (a >= t[maxc]) return sign | maxc;
    int lo = 0, hi = maxc; /* t[lo] <= a < t[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (t[mid] <= a) lo = mid; else hi = mid;
    }
    if (t[lo] == a) return sign | lo;
    double midpoint = 0.5 * (t[lo] + t[hi]); /* exact: <= 5 significant bits */
    int c;
    if (a < midpoint) c = lo;
    else if (a > midpoint) c = hi;
    else c = (lo & 1) ? hi : lo;
    return sign | c;
}

void fp8o_encode_array(const float *v, int64_t n, int fmt, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)fp8o_encode(v[i], fmt);
}

void fp8o_decode_array(const uint8_t *c, int64_t n, int fmt, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fp8o_decode(c[i], fmt);
}

static float bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------ compute_bias */

static double fmt_max(int fmt) { return fmt == FMT_E4M3 ? 448.0 : 57344.0; }

/* e = floor(log2(fmax / amax)) - margin, clamped to [-126, 127] so that both
 * 2^e and 2^-e are exact fp32 numbers and 127 - e is a valid E8M0 code.
 * Readings where the pages are silent: amax == 0 gives e = 0 (scale 1); a
 * non-finite amax gives e = 0 and raises *nonfinite.
 * floor(log2(r)) is read off frexp: r = f 2^x with f in [0.5, 1) gives x - 1.
 * r = fmax/amax in fp64 cannot round across a power of two for an fp32 amax
 * (the nearest fp32 amax to a boundary is a relative 2^-24 away). */
int fp8o_compute_bias(float amax, int fmt, int margin, int *nonfinite)
{
    if (isnan(amax) || isinf(amax)) {
        if (nonfinite) *nonfinite = 1;
        return 0;
    }
    double a = fabs((double)amax);
    if (a == 0.0) return 0;
    double r = fmt_max(fmt) / a;
    int x;
    frexp(r, &x);
    long e = (long)(x - 1) - (long)margin;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return (int)e;
}

float fp8o_pow2f(int e) { return ldexpf(1.0f, e); }

/* The OCP MX alternative to compute_bias for MX blocks, not the default: the
 * block's largest magnitude is moved into the top binade of the format,
 * e = emax - floor(log2(amax)) - margin with emax = 8 (E4M3) or 15 (E5M2), so a
 * block whose amax has a significand above 1.75 saturates.  Same clamping and
 * special cases as compute_bias.  floor(log2(amax)) is read off frexp. */
int fp8o_compute_bias_ocp(float amax, int fmt, int margin, int *nonfinite)
{
    if (isnan(amax) || isinf(amax)) {
        if (nonfinite) *nonfinite = 1;
        return 0;
    }
    double a = fabs((double)amax);
    if (a == 0.0) return 0;
    int x;
    frexp(a, &x);
    long e = (long)(fmt == FMT_E4M3 ? 8 : 15) - (long)(x - 1) - (long)margin;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return (int)e;
}

/* The non-power-of-two alternative for per-tensor scales, not the default:
 * s = fmax / amax and s_inv = 1 / s, each one fp32 division rounded to nearest
 * (so the cast rounds twice: the product x s, then Encode).  amax == 0 gives
 * s = 1; a non-finite amax gives s = 1 and returns 1. */
int fp8o_compute_scale_ratio(float amax, int fmt, float *scale, float *scale_inv)
{
    int nf = isnan(amax) || isinf(amax);
    float a = fabsf(amax);
    float s = (nf || a == 0.0f) ? 1.0f : (float)fmt_max(fmt) / a;
    *scale = s;
    *scale_inv = 1.0f / s;
    return nf;
}

/* ------------------------------------------------------------------ amax */

/* max |x| over a bf16 matrix; a NaN anywhere makes the result NaN */
static float amax_of(const uint16_t *x, int64_t rows, int64_t cols, int64_t rs, int64_t cs)
{
    float m = 0.0f;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            float a = fabsf(bf16_value(x[i * rs + j * cs]));
            if (isnan(m)) continue;
            if (isnan(a) || a > m) m = a;
        }
    return m;
}

float fp8o_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld)
{
    return amax_of(x, rows, cols, ld, 1);
}

/* ------------------------------------------------------------- quantise */

/* Per-tensor cast with a given scale s (= 2^e), row-wise into q_row
 * [rows x cols] and column-wise (transposed) into q_col [cols x rows]. */
void fp8o_quantize_tensor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld, int fmt, float scale,
                          uint8_t *q_row, uint8_t *q_col)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            float p = bf16_value(x[i * ld + j]) * scale;
            int code = fp8o_encode(p, fmt);
            if (q_row) q_row[i * cols + j] = (uint8_t)code;
            if (q_col) q_col[j * rows + i] = (uint8_t)code;
        }
}

/* Per-tensor cast of an fp32 array x[n] with scale s: q[i] = Encode(x[i] * s),
 * the product one fp32 multiplication (the same "scale, then cast" step, for
 * tensors held in fp32).  Its amax is max |x[i]|, NaN if any element is NaN. */
void fp8o_quantize_f32(const float *x, int64_t n, int fmt, float s, uint8_t *q)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float p = x[i] * s;
        q[i] = (uint8_t)fp8o_encode(p, fmt);
    }
}

float fp8o_amax_f32(const float *x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (isnan(a)) return a;
        if (a > m) m = a;
    }
    return m;
}

/* Block-scaled cast of the rows x cols matrix v(i,j) = x[i*rs + j*cs] with
 * br x bc blocks (a partial block at an edge covers the elements that exist).
 * Each block b: amax_b, e_b = compute_bias(amax_b, margin), q = Encode(v 2^e_b).
 * The stored scale is the dequantisation factor 2^-e_b, as fp32 (sf_f32) or as
 * the E8M0 code 127 - e_b (sf_e8m0), at [block_row * nbc + block_col]. */
static void quant_blocks(const uint16_t *x, int64_t rows, int64_t cols, int64_t rs, int64_t cs, int fmt,
                         int margin, int64_t br, int64_t bc, int ocp, uint8_t *q, float *sf_f32, uint8_t *sf_e8m0,
                         int *nonfinite)
{
    int64_t nbr = (rows + br - 1) / br, nbc = (cols + bc - 1) / bc;
    int flag = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : flag)
    for (int64_t b = 0; b < nbr * nbc; ++b) {
        int64_t bi = b / nbc, bj = b % nbc;
        int64_t i0 = bi * br, j0 = bj * bc;
        int64_t ni = rows - i0 < br ? rows - i0 : br;
        int64_t nj = cols - j0 < bc ? cols - j0 : bc;
        float amax = amax_of(x + i0 * rs + j0 * cs, ni, nj, rs, cs);
        int nf = 0;
        int e = ocp ? fp8o_compute_bias_ocp(amax, fmt, margin, &nf) : fp8o_compute_bias(amax, fmt, margin, &nf);
        flag |= nf;
        float s = ldexpf(1.0f, e);
        for (int64_t i = i0; i < i0 + ni; ++i)
            for (int64_t j = j0; j < j0 + nj; ++j) {
                float p = bf16_value(x[i * rs + j * cs]) * s;
                q[i * cols + j] = (uint8_t)fp8o_encode(p, fmt);
            }
        if (sf_f32) sf_f32[b] = ldexpf(1.0f, -e);
        if (sf_e8m0) sf_e8m0[b] = (uint8_t)(127 - e);
    }
    if (nonfinite && flag) *nonfinite = 1;
}

static void gran_block(int gran, int64_t *br, int64_t *bc)
{
    switch (gran) {
    case GRAN_1x128: *br = 1; *bc = 128; break;
    case GRAN_128x128: *br = 128; *bc = 128; break;
    default: *br = 1; *bc = 32; break; /* MX 1x32, either bias rule */
    }
}

/* Block granularities.  Row-wise output: blocks over x as stored.
 * Column-wise output: the same quantisation applied to x transposed, so
 * 1x128 -> 128x1 blocks down the columns, 1x32 -> 32x1, 128x128 unchanged.
 * Scales are fp32 2^-e (1x128, 128x128) or E8M0 codes (1x32; granularity 4 is
 * 1x32 with the OCP MX bias rule). */
int fp8o_quantize_block(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld, int fmt, int gran, int margin,
                        uint8_t *q_row, void *sf_row, uint8_t *q_col, void *sf_col)
{
    int64_t br, bc;
    gran_block(gran, &br, &bc);
    int mx = gran == GRAN_MX32 || gran == GRAN_MX32_OCP;
    int ocp = gran == GRAN_MX32_OCP;
    int nf = 0;
    if (q_row)
        quant_blocks(x, rows, cols, ld, 1, fmt, margin, br, bc, ocp, q_row, mx ? NULL : (float *)sf_row,
                     mx ? (uint8_t *)sf_row : NULL, &nf);
    if (q_col)
        quant_blocks(x, cols, rows, 1, ld, fmt, margin, br, bc, ocp, q_col, mx ? NULL : (float *)sf_col,
                     mx ? (uint8_t *)sf_col : NULL, &nf);
    return nf;
}

/* ----------------------------------------------------- delayed scaling */

/* One delayed-scaling update: record this step's amax in the ring at
 * pos mod L, advance pos, and derive the next step's bias from the maximum of
 * the recorded window (the last min(pos, L) amax values); reset amax to 0. */
int fp8o_history_update(float *hist, int32_t L, int64_t *pos, float *amax, int fmt, int margin, int32_t *bias,
                        float *scale, float *scale_inv)
{
    hist[*pos % L] = *amax;
    *pos += 1;
    int64_t n = *pos < L ? *pos : L;
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(m)) break;
        if (isnan(hist[i]) || hist[i] > m) m = hist[i];
    }
    int nf = 0;
    int e = fp8o_compute_bias(m, fmt, margin, &nf);
    *bias = e;
    *scale = ldexpf(1.0f, e);
    *scale_inv = ldexpf(1.0f, -e);
    *amax = 0.0f;
    return nf;
}

/* ----------------------------------------------------------------- GEMM */

/* Dequantisation factor of element (row, k) of an operand stored [rows x K]. */
static double operand_scale(int gran, const void *sf, int64_t row, int64_t k, int64_t K)
{
    switch (gran) {
    case GRAN_TENSOR: return (double)((const float *)sf)[0];
    case GRAN_1x128: return (double)((const float *)sf)[row * ((K + 127) / 128) + k / 128];
    case GRAN_128x128: return (double)((const float *)sf)[(row / 128) * ((K + 127) / 128) + k / 128];
    default: {
        uint8_t c = ((const uint8_t *)sf)[row * ((K + 31) / 32) + k / 32];
        if (c == 255) return NAN;
        return ldexp(1.0, (int)c - 127);
    }
    }
}

/* y[m,n] = sum_k deq(A[m,k]) deq(B[n,k]) in fp64 for the listed (m, n) pairs,
 * and the magnitude sum_k |deq(A[m,k]) deq(B[n,k])| used by the tolerance.
 * A is [M x K] and B is [N x K], both K-major. */
void fp8o_gemm_sample(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, int fa, int ga,
                      const void *sfa, const uint8_t *B, int64_t ldb, int fb, int gb, const void *sfb,
                      int64_t count, const int64_t *ms, const int64_t *ns, double *out, double *out_abs)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t s = 0; s < count; ++s) {
        int64_t m = ms[s], n = ns[s];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k, K);
            double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, n, k, K);
            acc += a * b;
            mag += fabs(a * b);
        }
        out[s] = acc;
        if (out_abs) out_abs[s] = mag;
    }
}

/* The whole M x N product (small shapes). */
void fp8o_gemm_full(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, int fa, int ga,
                    const void *sfa, const uint8_t *B, int64_t ldb, int fb, int gb, const void *sfb, double *out,
                    double *out_abs)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k, K);
                double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, n, k, K);
                acc += a * b;
                mag += fabs(a * b);
            }
            out[m * N + n] = acc;
            if (out_abs) out_abs[m * N + n] = mag;
        }
}

/* ----------------------------------------------------- cast statistics */

/* FP8-CSCALE keeps one fixed bias per tensor instead of deriving it from the
 * amax, and fixed biases work only in a narrow range ("Training and inference
 * of large language models using 8-bit floating point", "Proposed method" and
 * "Key findings": the fixed-scaling sweep).  What a fixed scale does to a
 * tensor is counted here by definition, for each scale s_j:
 *   saturated[j] += #{ x : x not NaN, |fl32(x s_j)| > fmax }   (the cast clips it)
 *   underflow[j] += #{ x : x not NaN, x != 0, Encode(fl32(x s_j)) = +-0 }  (flushed)
 * Counts are accumulated into the caller's arrays. */
void fp8o_cast_stats(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld, int fmt, const float *scales,
                     int n, uint64_t *saturated, uint64_t *underflow)
{
    const double fmax = fmt_max(fmt);
    for (int j = 0; j < n; ++j) {
        uint64_t sat = 0, und = 0;
#pragma omp parallel for reduction(+ : sat, und) schedule(static)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                const float xv = bf16_value(x[r * ld + c]);
                if (isnan(xv)) continue;
                const float v = xv * scales[j];
                if (!isnan(v) && fabs((double)v) > fmax) ++sat;
                if (xv != 0.0f && (fp8o_encode(v, fmt) & 0x7F) == 0) ++und;
            }
        saturated[j] += sat;
        underflow[j] += und;
    }
}

/* ------------------------------------------------------------ threads */

int fp8o_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void fp8o_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
