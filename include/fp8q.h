/*
 * fp8q.h -- C ABI of the FP8 amax / scale-selection / scaled-cast / scaled-GEMM
 * library for one GB300 GPU (sm_103a).
 *
 * The method (papers and posts cited by title and section):
 *   - per-tensor scaling with the FP8-AMAX rule: a bias per tensor from the
 *     tensor's maximum absolute value, e = floor(log2(fmax/amax)) - margin
 *     ("Training and inference of large language models using 8-bit floating
 *     point", section "Proposed method");
 *   - the operands are multiplied by their scales before the FP8 cast and the
 *     matrix product is divided by them afterwards (same section);
 *   - FP8_E4 (E4M3) for weights and activations, FP8_E5 (E5M2) for gradients
 *     (same section);
 *   - delayed scaling from the maximum amax over a window of past iterations,
 *     and per-block / MXFP8 scaling with one scale per block ("Per-Tensor and
 *     Per-Block Scaling Strategies for Effective FP8 Training", "Key Questions
 *     Answered").
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument that names a tensor is a DEVICE pointer into memory
 *     the caller allocated and owns.  The library allocates no device memory and
 *     keeps no state between calls (the one exception is the static scratch of
 *     fp8_quantize_current_noalloc).  Every entry point except
 *     fp8_quantize_current_noalloc is safe to call from several host threads on
 *     different streams; calls of that one must be ordered on the GPU.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     only enqueues work on that stream and returns; none synchronises the host.
 *   - Arguments are validated on the host before anything is enqueued:
 *     a NULL required pointer, a negative size or an inconsistent leading
 *     dimension returns FP8_ERR_INVALID_ARG; a shape or alignment the kernels do
 *     not handle returns FP8_ERR_UNSUPPORTED (never a silent slow path).  A
 *     failed launch returns FP8_ERR_CUDA.  A size of zero is a valid no-op.
 *   - Conditions only the device can see (a non-finite amax, a non-power-of-two
 *     block scale, an internal wait that gave up) are ORed as bits into an
 *     optional device status word (`status`, int32, may be NULL); kernels never
 *     trap.
 *   - bf16 inputs are row-major [rows x cols] with leading dimension `ld`
 *     (elements, ld >= cols).  FP8 outputs are one byte per element, OFP8 E4M3
 *     or E5M2 bit patterns, row-major and dense.
 *   - The scales this library derives are powers of two.  A per-tensor
 *     quantisation scale is the multiplier s = 2^e applied before the cast; the
 *     GEMM takes the dequantisation factor s^-1 = 2^-e.  Block scales are stored
 *     as dequantisation factors (fp32 2^-e, or the E8M0 code 127 - e).
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>

/* Symbols of the C ABI are the only ones the shared library exports. */
#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,
    FP8_ERR_UNSUPPORTED = 2,
    FP8_ERR_CUDA = 3,
    FP8_ERR_TIMEOUT = 4
} fp8_status;

typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format;

typedef enum {
    FP8_SCALE_TENSOR = 0,        /* one scale for the whole tensor */
    FP8_SCALE_BLOCK_1x128 = 1,   /* activation blocks: 1 row x 128 columns */
    FP8_SCALE_BLOCK_128x128 = 2, /* weight blocks: 128 x 128 */
    FP8_SCALE_MX_1x32 = 3,       /* MXFP8: 1 x 32 blocks, E8M0 scales */
    FP8_SCALE_MX_1x32_OCP = 4    /* the same blocks and storage with the OCP MX bias rule (option) */
} fp8_granularity;

typedef enum { FP8_GEMM_FPROP = 0, FP8_GEMM_DGRAD = 1, FP8_GEMM_WGRAD = 2 } fp8_gemm_op;

typedef enum { FP8_OUT_F32 = 0, FP8_OUT_BF16 = 1 } fp8_out_dtype;

/* Bits of the device status word. */
#define FP8_STATUS_NONFINITE_AMAX 1  /* an amax was NaN or Inf; its bias was set to 0 */
#define FP8_STATUS_TIMEOUT 2         /* a bounded wait inside a kernel gave up; output invalid */
#define FP8_STATUS_BAD_BLOCK_SCALE 4 /* a block scale given to the GEMM was not a power of two */

/*
 * fp8_amax -- maximum absolute value of a bf16 tensor.
 * Source: the per-tensor statistic the FP8-AMAX scales are computed from
 * ("Training and inference of large language models using 8-bit floating
 * point", "Proposed method").
 *
 *   x      device, bf16 [rows x cols], leading dimension ld (elements), 16-byte
 *          aligned; cols and ld must be multiples of 8 (else UNSUPPORTED).
 *   amax   device, one fp32.  ACCUMULATED: the call stores max(*amax, max|x|),
 *          so the caller zeroes it first (fp8_amax_history_update resets it).
 *          A NaN anywhere in x makes the result NaN.
 */
FP8Q_API fp8_status fp8_amax(const void *x, int64_t rows, int64_t cols, int64_t ld, float *amax, void *stream);

/*
 * fp8_compute_scale -- the FP8-AMAX compute_bias rule for current scaling.
 * Source: the compute_bias rule of FP8-AMAX, a base-2 logarithm of the format
 * maximum over the tensor's amax less a margin ("Training and inference of
 * large language models using 8-bit floating point", "Proposed method").
 *
 *   e = floor(log2(fmax / amax)) - margin, fmax = 448 (E4M3) or 57344 (E5M2),
 *   computed exactly from the exponent and mantissa bits of amax, clamped to
 *   [-126, 127].  amax == 0 gives e = 0; a non-finite amax gives e = 0 and sets
 *   FP8_STATUS_NONFINITE_AMAX.
 *
 *   amax       device, one fp32 (read).
 *   bias       device, one int32 (written: e).          May be NULL.
 *   scale      device, one fp32 (written: 2^e).          May be NULL.
 *   scale_inv  device, one fp32 (written: 2^-e).         May be NULL.
 *   status     device, one int32 (bits ORed in).         May be NULL.
 */
FP8Q_API fp8_status fp8_compute_scale(const float *amax, fp8_format fmt, int32_t margin, int32_t *bias, float *scale,
                             float *scale_inv, int32_t *status, void *stream);

/*
 * fp8_compute_scale_ratio -- the non-power-of-two alternative to compute_bias.
 * Source: the scale taken as the ratio of the format maximum to the tensor's
 * amax itself, the quantity whose logarithm the compute_bias rule floors
 * ("Training and inference of large language models using 8-bit floating
 * point", "Proposed method").  Not the default.
 *
 *   scale = fmax / amax, scale_inv = 1 / scale, each one fp32 division rounded
 *   to nearest; amax == 0 gives 1, 1; a non-finite amax gives 1, 1 and sets
 *   FP8_STATUS_NONFINITE_AMAX.  A cast with such a scale rounds twice (the
 *   fp32 product, then the FP8 encoding); fp8_quantize and fp8_scaled_gemm take
 *   it like any per-tensor scale.
 *
 *   amax       device, one fp32 (read).
 *   scale, scale_inv: device, one fp32 each (written; either may be NULL, not both).
 *   status     device int32 or NULL.
 */
FP8Q_API fp8_status fp8_compute_scale_ratio(const float *amax, fp8_format fmt, float *scale, float *scale_inv,
                                            int32_t *status, void *stream);

/*
 * fp8_amax_history_update -- one delayed-scaling step.
 * Source: delayed scaling, where the scale comes from the largest amax seen
 * in a window of past steps ("Per-Tensor and Per-Block Scaling Strategies for
 * Effective FP8 Training", "Key Questions Answered").
 *
 *   history[pos mod len] = *amax;  pos += 1;
 *   e = compute_bias(max(history[0 .. min(pos, len) - 1]), fmt, margin);
 *   bias = e; scale = 2^e; scale_inv = 2^-e;  *amax = 0.
 *
 *   history    device, fp32[len], zero-initialised by the caller before step 0.
 *   len        window length, 1 <= len <= 65536.
 *   pos        device, one int64 (read and incremented).
 *   amax       device, one fp32 (read, then reset to 0 for the next step).
 *   bias, scale, scale_inv, status: as for fp8_compute_scale (bias/scale/
 *              scale_inv required here).
 * The state (history, pos, bias, scale, scale_inv) is plain device memory:
 * copying it out and back in resumes the sequence exactly.
 */
FP8Q_API fp8_status fp8_amax_history_update(float *history, int32_t len, int64_t *pos, float *amax, fp8_format fmt,
                                   int32_t margin, int32_t *bias, float *scale, float *scale_inv,
                                   int32_t *status, void *stream);

/*
 * fp8_amax_history_update_batch -- fp8_amax_history_update for n independent
 * delayed-scaling states in one launch.
 * Source: as fp8_amax_history_update (delayed scaling, "Per-Tensor and
 * Per-Block Scaling Strategies for Effective FP8 Training", "Key Questions
 * Answered").  A model keeps one state per FP8 tensor; updating them together
 * takes one kernel launch per 48 states instead of one per state.
 *
 *   states   HOST array of n records, read during the call only.  Each record
 *            holds the arguments of one fp8_amax_history_update call: device
 *            pointers history, pos, amax, bias, scale and scale_inv (all
 *            required) and status (or NULL); len in [1, 65536]; fmt; margin.
 *            `reserved` must be 0.  Records must not share history, pos,
 *            amax, bias, scale or scale_inv (they may share a status word).
 *   n        number of records, n >= 0; 0 is a no-op (states may then be NULL).
 * Every state ends exactly as fp8_amax_history_update would leave it.
 */
typedef struct {
    float *history;
    int64_t *pos;
    float *amax;
    int32_t *bias;
    float *scale;
    float *scale_inv;
    int32_t *status;
    int32_t len;
    int32_t fmt;    /* fp8_format */
    int32_t margin;
    int32_t reserved;
} fp8_history_state;
FP8Q_API fp8_status fp8_amax_history_update_batch(const fp8_history_state *states, int32_t n, void *stream);

/*
 * fp8_set_bias -- a fixed exponent bias (FP8-CSCALE).
 * Source: fixed scaling, a bias chosen once per tensor instead of derived
 * from its amax, compared against FP8-AMAX in a sweep of fixed values
 * ("Training and inference of large language models using 8-bit floating
 * point", "Proposed method" and "Key findings").
 *
 *   bias = e; scale = 2^e; scale_inv = 2^-e.    e in [-126, 127], else INVALID_ARG.
 *   bias, scale, scale_inv: device, each may be NULL (not all three).
 * The outputs feed fp8_quantize and fp8_scaled_gemm like those of
 * fp8_compute_scale.
 */
FP8Q_API fp8_status fp8_set_bias(int32_t e, int32_t *bias, float *scale, float *scale_inv, void *stream);

/*
 * fp8_cast_stats -- what a cast at given scales does to a tensor.
 * Source: the range problem fixed scaling runs into, overflow and underflow
 * of the FP8 range ("Training and inference of large language models using
 * 8-bit floating point", "Motivation & Objective" and "Key findings", the
 * fixed-scaling sweep).
 *
 *   for j < n:  saturated[j] += #{ x not NaN : |fl32(x * scales[j])| > fmax }
 *               underflow[j] += #{ x not NaN, x != 0 : cast of fl32(x * scales[j]) is +-0 }
 *
 *   x          as for fp8_amax (bf16 [rows x cols], ld, 16-byte aligned, cols
 *              and ld multiples of 8).
 *   fmt        the format the cast targets (fmax 448 or 57344).
 *   scales     device fp32[n], 1 <= n <= 8 (any values; powers of two from
 *              fp8_set_bias or fp8_compute_scale in the usual case).
 *   saturated, underflow: device uint64[n], ACCUMULATED (the caller zeroes them).
 * The counts are exactly what fp8_quantize would clip and flush with that
 * scale.  Empty x is a no-op.
 */
FP8Q_API fp8_status fp8_cast_stats(const void *x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt,
                                   const float *scales, int32_t n, uint64_t *saturated, uint64_t *underflow,
                                   void *stream);

/*
 * fp8_quantize -- the scaled cast to FP8, row-wise and/or column-wise.
 * Source: the scaling step that precedes the FP8 cast ("Training and
 * inference of large language models using 8-bit floating point", "Proposed
 * method");
 * per-block and MXFP8 block scales ("Per-Tensor and Per-Block Scaling
 * Strategies for Effective FP8 Training", "Key Questions Answered").
 *
 *   q = RNE_saturate_fmt(x * 2^e) with the product taken in fp32.
 *
 *   x        device, bf16 [rows x cols], leading dimension ld; 16-byte aligned,
 *            cols and ld multiples of 8; rows and cols below 2^31 (else
 *            UNSUPPORTED: tiles are addressed with 32-bit coordinates).
 *   gran     FP8_SCALE_TENSOR: e from `scale` (device fp32 2^e, required);
 *              sf_row and sf_col must be NULL.
 *            FP8_SCALE_BLOCK_1x128 / _128x128 / FP8_SCALE_MX_1x32: each block
 *              gets e_b = compute_bias(amax_b, fmt, margin); `scale` must be NULL.
 *            FP8_SCALE_MX_1x32_OCP: MX blocks with the alternative rule of the
 *              OCP MX format, e_b = emax - floor(log2(amax_b)) - margin (emax 8
 *              for E4M3, 15 for E5M2): the block's largest magnitude lands in
 *              the format's top binade and saturates when its significand
 *              exceeds 1.75.  Not the default; scales stored as for MX.
 *              A partial block at an edge uses the elements that exist.
 *   margin   used by the block granularities only.
 *   q_row    device u8 [rows x cols] (dense, 8-byte aligned), or NULL.
 *   q_col    device u8 [cols x rows] (dense, the transposed copy, 16-byte
 *            aligned), or NULL.  Misalignment of either is UNSUPPORTED.
 *            At least one of q_row / q_col.  With q_col, rows must be a
 *            multiple of 16.  The column-wise copy is the row-wise
 *            quantisation of x transposed: per-tensor and 128x128 use the same
 *            scales as row-wise; 1x128 becomes 128x1 blocks down each column and
 *            MX 1x32 becomes 32x1.
 *   sf_row   block scales of q_row (required iff q_row and gran != TENSOR):
 *              1x128:   fp32 [rows x ceil(cols/128)]
 *              128x128: fp32 [ceil(rows/128) x ceil(cols/128)]
 *              MX 1x32 (either rule): u8 E8M0 [rows x ceil(cols/32)]
 *   sf_col   block scales of q_col (required iff q_col and gran != TENSOR):
 *              1x128:   fp32 [cols x ceil(rows/128)]
 *              128x128: fp32 [ceil(cols/128) x ceil(rows/128)]
 *              MX 1x32: u8 E8M0 [cols x ceil(rows/32)]
 *            Stored values are dequantisation factors 2^-e_b (fp32) or 127-e_b.
 *   amax     device fp32 or NULL: if given, max|x| is accumulated into it
 *            (fused amax for delayed scaling; same semantics as fp8_amax).
 */
FP8Q_API fp8_status fp8_quantize(const void *x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt,
                        fp8_granularity gran, int32_t margin, const float *scale, uint8_t *q_row, uint8_t *q_col,
                        void *sf_row, void *sf_col, float *amax, void *stream);

/*
 * fp8_quantize_batch -- several fp8_quantize casts in one launch.
 * Source: the casts of one FP8 linear layer's operands (activations and weights,
 * and the gradient in the backward pass), each with its own scale ("Training
 * and inference of large language models using 8-bit floating point",
 * "Proposed method"; per-block scales: "Per-Tensor and Per-Block Scaling
 * Strategies for Effective FP8 Training", "Key Questions Answered").
 *
 *   descs    HOST array of n descriptors; each names one cast with exactly the
 *            arguments of fp8_quantize (device pointers, sizes, format,
 *            granularity, margin) and `reserved` = 0.  Formats and granularities
 *            may differ between descriptors.
 *   n        0 .. FP8_QUANTIZE_BATCH_MAX; n = 0 is a no-op.
 * Every output (codes, scales, amax) equals that of the n fp8_quantize calls
 * made one after another; an amax shared by several descriptors accumulates
 * the maximum over all of them.  The casts run concurrently, so no output may
 * overlap another descriptor's input or output.  Each descriptor is validated
 * as fp8_quantize validates its arguments, and nothing is launched unless all
 * are valid (the error detail names the descriptor).  The grid is split among
 * the tensors in proportion to their 128x128 tiles.
 */
#define FP8_QUANTIZE_BATCH_MAX 4
typedef struct fp8_quantize_desc {
    const void *x;   /* bf16 [rows x cols], leading dimension ld (elements) */
    int64_t rows, cols, ld;
    int32_t fmt;      /* fp8_format */
    int32_t gran;     /* fp8_granularity */
    int32_t margin;
    int32_t reserved; /* must be 0 */
    const float *scale;
    uint8_t *q_row, *q_col;
    void *sf_row, *sf_col;
    float *amax;
} fp8_quantize_desc;
FP8Q_API fp8_status fp8_quantize_batch(const fp8_quantize_desc *descs, int32_t n, void *stream);

/*
 * fp8_quantize_f32 -- the per-tensor scaled cast of an fp32 tensor.
 * Source: the scaling step that precedes the FP8 cast ("Training and
 * inference of large language models using 8-bit floating point", "Proposed
 * method"), for tensors held in fp32 (master weights, fp32 GEMM outputs).
 *
 *   q[i] = RNE_saturate_fmt(fl32(x[i] * s)),  s = *scale, or 1 when scale is NULL.
 *
 *   x       device, fp32[n], dense, 16-byte aligned.
 *   n       element count; 0 is a no-op.
 *   scale   device fp32 (any value; 2^e from fp8_compute_scale in the usual
 *           case, when the product is exact) or NULL.
 *   q       device u8[n], 8-byte aligned.
 *   amax    device fp32 or NULL: if given, max|x| is accumulated into it
 *           (a NaN element makes it NaN), as for fp8_amax.
 * A NaN element casts to a NaN code; +-Inf and products beyond fmax saturate
 * to +-fmax.
 */
FP8Q_API fp8_status fp8_quantize_f32(const float *x, int64_t n, fp8_format fmt, const float *scale, uint8_t *q,
                                     float *amax, void *stream);

/*
 * fp8_quantize_current -- per-tensor current scaling and the cast, in one launch.
 * Source: FP8-AMAX scaling from the amax of the tensor being cast, the
 * compute_bias rule, then the scaled cast ("Training and inference of large
 * language models using 8-bit floating point", "Proposed method").
 *
 *   amax = max|x|;  e = compute_bias(amax, fmt, margin);  q = RNE_saturate_fmt(x * 2^e).
 *
 * The result is that of fp8_amax on a zeroed amax, then fp8_compute_scale,
 * then fp8_quantize(FP8_SCALE_TENSOR) with the new scale, bit for bit; x is
 * read twice, in one cooperative launch with a grid-wide barrier between the
 * amax and the cast.
 *
 *   x, rows, cols, ld, fmt, q_row, q_col: as for fp8_quantize.
 *   amax       device fp32 or NULL (written, not accumulated: max|x|).
 *   bias, scale, scale_inv: device, or NULL, as for fp8_compute_scale.
 *   workspace  device, FP8_QUANTIZE_CURRENT_WORKSPACE_BYTES bytes, 16-byte
 *              aligned, owned by the caller (the grid barrier uses its first
 *              16 bytes; the rest is reserved).  Zero it once before its first
 *              use; every call leaves it ready for the next one.  Calls that
 *              share a workspace must not run at the same time (same stream,
 *              or ordered by events).  After a call that reported
 *              FP8_STATUS_TIMEOUT, zero it again.
 *   status     device int32 or NULL (FP8_STATUS_NONFINITE_AMAX,
 *              FP8_STATUS_TIMEOUT: a CTA gave up waiting at the barrier and
 *              the codes are not valid).
 * An empty x writes amax 0, bias 0, scale 1, scale_inv 1.
 */
#define FP8_QUANTIZE_CURRENT_WORKSPACE_BYTES 4096
FP8Q_API fp8_status fp8_quantize_current(const void *x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt,
                                         int32_t margin, uint8_t *q_row, uint8_t *q_col, float *amax, int32_t *bias,
                                         float *scale, float *scale_inv, void *workspace, int32_t *status,
                                         void *stream);

/*
 * fp8_quantize_current_noalloc -- fp8_quantize_current without a workspace.
 * No counterpart in the method's sources: this entry point exists for callers
 * that cannot allocate device memory where they call it (a plugin or callback
 * given only its input and output buffers by a host framework, code whose
 * device memory is planned once against a fixed budget, loops that cannot
 * take the synchronisation cudaMalloc / cudaFree may cause).  It allocates
 * nothing.
 *
 * Arguments and results are those of fp8_quantize_current, without
 * `workspace`.  The scratch is a static 256-byte array in the library's device
 * code (the grid barrier's 16-byte header: arrival count, generation, scale and
 * the running max), present on every GPU that loads the library until the
 * process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that
 *     first call before any stream capture.
 *   - Every call shares the array and finds the previous call's contents in
 *     it; each call clears the barrier header on its stream first.  Calls
 *     whose kernels overlap on the GPU (different streams or host threads)
 *     race on the array: order them.
 */
FP8Q_API fp8_status fp8_quantize_current_noalloc(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                                 fp8_format fmt, int32_t margin, uint8_t *q_row, uint8_t *q_col,
                                                 float *amax, int32_t *bias, float *scale, float *scale_inv,
                                                 int32_t *status, void *stream);

/*
 * fp8_scaled_gemm -- D = unscale(A . B^T) on FP8 operands.
 * Source: the unscaling step that follows the FP8 matrix product ("Training
 * and inference of large language models using 8-bit floating point",
 * "Proposed method"); block
 * and MXFP8 scales ("Per-Tensor and Per-Block Scaling Strategies for Effective
 * FP8 Training", "Key Questions Answered").
 *
 *   D[m, n] = sum_k (A[m,k] sa(m,k)) (B[n,k] sb(n,k)),  fp32 accumulation.
 *
 *   op       FPROP (A = X_row, B = W_row), DGRAD (A = dY_row, B = W_col) or
 *            WGRAD (A = dY_col, B = X_col).  Every op is the same TN product
 *            over K-major operands; op only labels the call.
 *   A        device u8 [M x K], leading dimension lda (bytes), format fa.
 *   B        device u8 [N x K], leading dimension ldb (bytes), format fb.
 *            A and B 16-byte aligned; K, lda and ldb multiples of 16.
 *   ga, gb   scale granularity of A and of B:
 *              both FP8_SCALE_TENSOR: sfa / sfb point to ONE fp32 each, the
 *                dequantisation factor 2^-e of that tensor;
 *              otherwise neither may be TENSOR, and each of sfa / sfb is
 *                1x128:   fp32 [rows x ceil(K/128)]
 *                128x128: fp32 [ceil(rows/128) x ceil(K/128)]
 *                MX 1x32: u8 E8M0 [rows x K/32] (fp8_quantize writes codes
 *                  0..253; code 255, NaN in the OCP MX encoding, gives an
 *                  unspecified result)
 *              (rows = M for A, N for B).  fp32 block scales must be powers of
 *              two in [2^-127, 2^127] (what fp8_quantize writes); any other
 *              value sets FP8_STATUS_BAD_BLOCK_SCALE, and D is then
 *              unspecified.
 *   D        device, [M x N] fp32 or bf16 (out_dtype), leading dimension ldd
 *            (elements); 16-byte aligned, N and ldd multiples of 16.
 *   status   device int32 or NULL (FP8_STATUS_TIMEOUT, FP8_STATUS_BAD_BLOCK_SCALE).
 * K == 0 writes zeros.  Every block-scaled mode (1x128, 128x128 and MX 1x32
 * alike) needs K % 128 == 0 (one 128-wide K tile per scale load) and 4-byte
 * aligned sfa / sfb; other K return FP8_ERR_UNSUPPORTED.
 */
FP8Q_API fp8_status fp8_scaled_gemm(fp8_gemm_op op, int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                           fp8_format fa, fp8_granularity ga, const void *sfa, const uint8_t *B, int64_t ldb,
                           fp8_format fb, fp8_granularity gb, const void *sfb, void *D, fp8_out_dtype out_dtype,
                           int64_t ldd, int32_t *status, void *stream);

/*
 * fp8_scaled_gemm_quantize -- per-tensor FP8 GEMM whose epilogue casts D to FP8.
 * Source: in a stack of FP8 linear layers the output of one layer is the
 * input the next one scales and casts, and its scale comes from its amax
 * ("Training and inference of large language models using 8-bit floating
 * point", "Proposed method"); here that cast, and the amax, are done where
 * D leaves the accumulator.
 *
 *   v[m, n]  = ((sum_k A[m,k] B[n,k]) * sa) * sb     (fp32 accumulation, fp32 products)
 *   Dq[m, n] = RNE_saturate_fd(v[m, n] * scale_d)     (one rounding, as fp8_quantize)
 *   amax_d   = max(amax_d, max |v|)                    (accumulated, like fp8_amax)
 *
 *   A, lda, fa, B, ldb, fb: as for fp8_scaled_gemm; sfa / sfb point to one fp32
 *            each (per-tensor dequantisation factors 2^-e).
 *   Dq       device u8 [M x N], leading dimension ldd (bytes); 16-byte aligned,
 *            N and ldd multiples of 16.
 *   fd       format of Dq.
 *   scale_d  device, one fp32: the scale of Dq (2^e; with delayed scaling the
 *            one fp8_amax_history_update chose from earlier steps).
 *   amax_d   device fp32 or NULL: max |v| is folded in (to be recorded by
 *            fp8_amax_history_update).  A NaN in v makes it NaN.
 *   status   device int32 or NULL (FP8_STATUS_TIMEOUT).
 * K == 0 writes zero codes and leaves amax_d unchanged.
 */
FP8Q_API fp8_status fp8_scaled_gemm_quantize(fp8_gemm_op op, int64_t M, int64_t N, int64_t K, const uint8_t *A,
                                             int64_t lda, fp8_format fa, const float *sfa, const uint8_t *B,
                                             int64_t ldb, fp8_format fb, const float *sfb, uint8_t *Dq, int64_t ldd,
                                             fp8_format fd, const float *scale_d, float *amax_d, int32_t *status,
                                             void *stream);

/* fp8_status_string -- static, human-readable name of a status code. */
FP8Q_API const char *fp8_status_string(fp8_status s);

/* fp8_last_error_detail -- static text describing the last non-OK status
 * returned on the calling host thread (thread-local; empty if none). */
FP8Q_API const char *fp8_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
