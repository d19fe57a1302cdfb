// api.cu -- the extern "C" entry points of libfp8q: argument validation on the
// host, then one or more asynchronous launches on the caller's stream.
// Declarations, argument meaning, layouts and error behaviour: include/fp8q.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace fp8q {

static thread_local char g_detail[512];

void set_error_detail(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
}

fp8_status launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax, cudaStream_t st);
fp8_status launch_compute_scale(const float* amax, int fmt, int margin, int32_t* bias, float* scale, float* scale_inv,
                                int32_t* status, cudaStream_t st);
fp8_status launch_compute_scale_ratio(const float* amax, int fmt, float* scale, float* scale_inv, int32_t* status,
                                      cudaStream_t st);
fp8_status launch_history(float* hist, int len, int64_t* pos, float* amax, int fmt, int margin, int32_t* bias,
                          float* scale, float* scale_inv, int32_t* status, cudaStream_t st);
fp8_status launch_quantize_current(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int margin,
                                   uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias, float* scale,
                                   float* scale_inv, void* workspace, int32_t* status, cudaStream_t st);
fp8_status launch_quantize_current_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt,
                                           int margin, uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias,
                                           float* scale, float* scale_inv, int32_t* status, cudaStream_t st);
fp8_status launch_set_bias(int e, int32_t* bias, float* scale, float* scale_inv, cudaStream_t st);
fp8_status launch_history_batch(const fp8_history_state* states, int n, cudaStream_t st);
fp8_status launch_quantize_f32(const float* x, int64_t n, int fmt, const float* scale, uint8_t* q, float* amax,
                               cudaStream_t st);
fp8_status launch_cast_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, const float* scales,
                             int n, uint64_t* saturated, uint64_t* underflow, cudaStream_t st);
fp8_status launch_quantize_batch(const fp8_quantize_desc* descs, int n, cudaStream_t st);
fp8_status launch_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int gran, int margin,
                           const float* scale, uint8_t* q_row, uint8_t* q_col, void* sf_row, void* sf_col,
                           float* amax, cudaStream_t st);
fp8_status launch_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int fa, int ga, const void* sfa,
                       const uint8_t* B, int64_t ldb, int fb, int gb, const void* sfb, void* D, int out,
                       int64_t ldd, const float* sd, float* amax_d, int32_t* status, cudaStream_t st);

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_fmt(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
bool valid_gran(int g) { return g >= FP8_SCALE_TENSOR && g <= FP8_SCALE_MX_1x32_OCP; }
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

fp8_status check_bf16_matrix(const void* x, int64_t rows, int64_t cols, int64_t ld) {
    FP8_REQUIRE(rows >= 0 && cols >= 0, FP8_ERR_INVALID_ARG, "negative size (rows=%lld cols=%lld)", (long long)rows,
                (long long)cols);
    FP8_REQUIRE(ld >= cols && ld >= 1, FP8_ERR_INVALID_ARG, "ld (%lld) < cols (%lld)", (long long)ld, (long long)cols);
    if (rows == 0 || cols == 0) return FP8_OK;
    FP8_REQUIRE(x != nullptr, FP8_ERR_INVALID_ARG, "x is NULL");
    FP8_REQUIRE(cols % 8 == 0 && ld % 8 == 0, FP8_ERR_UNSUPPORTED, "cols and ld must be multiples of 8 (16-byte rows)");
    FP8_REQUIRE(aligned(x, 16), FP8_ERR_UNSUPPORTED, "x must be 16-byte aligned");
    return FP8_OK;
}

// The casts address x and the column-wise output through TMA tensor maps, whose coordinates are 32-bit.
fp8_status check_tma_dims(int64_t rows, int64_t cols) {
    FP8_REQUIRE(rows < (1ll << 31) && cols < (1ll << 31), FP8_ERR_UNSUPPORTED,
                "rows and cols must be below 2^31 (rows=%lld cols=%lld)", (long long)rows, (long long)cols);
    return FP8_OK;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" {

const char* fp8_status_string(fp8_status s) {
    switch (s) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
        case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
        case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    }
    return "FP8_ERR_UNKNOWN";
}

const char* fp8_last_error_detail(void) { return g_detail; }

fp8_status fp8_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax, void* stream) {
    g_detail[0] = 0;
    fp8_status s = check_bf16_matrix(x, rows, cols, ld);
    if (s != FP8_OK) return s;
    FP8_REQUIRE(amax != nullptr, FP8_ERR_INVALID_ARG, "amax is NULL");
    FP8_REQUIRE(aligned(amax, 4), FP8_ERR_INVALID_ARG, "amax must be 4-byte aligned");
    if (rows == 0 || cols == 0) return FP8_OK;
    return launch_amax(x, rows, cols, ld, amax, as_stream(stream));
}

fp8_status fp8_compute_scale(const float* amax, fp8_format fmt, int32_t margin, int32_t* bias, float* scale,
                             float* scale_inv, int32_t* status, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(amax != nullptr, FP8_ERR_INVALID_ARG, "amax is NULL");
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(bias || scale || scale_inv, FP8_ERR_INVALID_ARG, "no output (bias, scale, scale_inv all NULL)");
    return launch_compute_scale(amax, fmt, margin, bias, scale, scale_inv, status, as_stream(stream));
}

fp8_status fp8_compute_scale_ratio(const float* amax, fp8_format fmt, float* scale, float* scale_inv, int32_t* status,
                                   void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(amax != nullptr, FP8_ERR_INVALID_ARG, "amax is NULL");
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(scale || scale_inv, FP8_ERR_INVALID_ARG, "no output (scale and scale_inv both NULL)");
    return launch_compute_scale_ratio(amax, fmt, scale, scale_inv, status, as_stream(stream));
}

fp8_status fp8_amax_history_update(float* history, int32_t len, int64_t* pos, float* amax, fp8_format fmt,
                                   int32_t margin, int32_t* bias, float* scale, float* scale_inv, int32_t* status,
                                   void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(history && pos && amax && bias && scale && scale_inv, FP8_ERR_INVALID_ARG,
                "history, pos, amax, bias, scale and scale_inv are required");
    FP8_REQUIRE(len >= 1 && len <= 65536, FP8_ERR_INVALID_ARG, "len must be in [1, 65536] (got %d)", (int)len);
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(aligned(pos, 8), FP8_ERR_INVALID_ARG, "pos must be 8-byte aligned");
    return launch_history(history, len, pos, amax, fmt, margin, bias, scale, scale_inv, status, as_stream(stream));
}

static_assert(sizeof(fp8_history_state) == 72, "fp8_history_state is part of the ABI: 7 pointers and 4 int32");

fp8_status fp8_amax_history_update_batch(const fp8_history_state* states, int32_t n, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(n >= 0, FP8_ERR_INVALID_ARG, "negative count %d", (int)n);
    if (n == 0) return FP8_OK;
    FP8_REQUIRE(states != nullptr, FP8_ERR_INVALID_ARG, "states is NULL");
    for (int32_t i = 0; i < n; ++i) {
        const fp8_history_state& t = states[i];
        FP8_REQUIRE(t.history && t.pos && t.amax && t.bias && t.scale && t.scale_inv, FP8_ERR_INVALID_ARG,
                    "record %d: history, pos, amax, bias, scale and scale_inv are required", (int)i);
        FP8_REQUIRE(t.len >= 1 && t.len <= 65536, FP8_ERR_INVALID_ARG, "record %d: len must be in [1, 65536] (got %d)",
                    (int)i, (int)t.len);
        FP8_REQUIRE(valid_fmt(t.fmt), FP8_ERR_INVALID_ARG, "record %d: unknown format %d", (int)i, (int)t.fmt);
        FP8_REQUIRE(t.reserved == 0, FP8_ERR_INVALID_ARG, "record %d: reserved must be 0", (int)i);
        FP8_REQUIRE(aligned(t.pos, 8) && aligned(t.history, 4) && aligned(t.amax, 4) && aligned(t.bias, 4) &&
                        aligned(t.scale, 4) && aligned(t.scale_inv, 4) && (!t.status || aligned(t.status, 4)),
                    FP8_ERR_INVALID_ARG, "record %d: misaligned pointer (pos 8 bytes, the others 4)", (int)i);
    }
    return launch_history_batch(states, n, as_stream(stream));
}

}  // extern "C"

namespace fp8q {
namespace {

// The checks of one fp8_quantize call (shared with fp8_quantize_batch).
fp8_status check_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int gran,
                          const float* scale, const uint8_t* q_row, const uint8_t* q_col, const void* sf_row,
                          const void* sf_col, const float* amax) {
    fp8_status s = check_bf16_matrix(x, rows, cols, ld);
    if (s != FP8_OK) return s;
    s = check_tma_dims(rows, cols);
    if (s != FP8_OK) return s;
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(valid_gran(gran), FP8_ERR_INVALID_ARG, "unknown granularity %d", (int)gran);
    if (rows == 0 || cols == 0) return FP8_OK;
    FP8_REQUIRE(q_row || q_col, FP8_ERR_INVALID_ARG, "q_row and q_col are both NULL");
    if (gran == FP8_SCALE_TENSOR) {
        FP8_REQUIRE(scale != nullptr, FP8_ERR_INVALID_ARG, "per-tensor quantisation needs scale");
        FP8_REQUIRE(!sf_row && !sf_col, FP8_ERR_INVALID_ARG, "per-tensor quantisation takes no block scales");
    } else {
        FP8_REQUIRE(scale == nullptr, FP8_ERR_INVALID_ARG, "block quantisation takes no per-tensor scale");
        FP8_REQUIRE(!q_row || sf_row, FP8_ERR_INVALID_ARG, "q_row needs sf_row");
        FP8_REQUIRE(!q_col || sf_col, FP8_ERR_INVALID_ARG, "q_col needs sf_col");
        FP8_REQUIRE(!sf_row || q_row, FP8_ERR_INVALID_ARG, "sf_row given without q_row");
        FP8_REQUIRE(!sf_col || q_col, FP8_ERR_INVALID_ARG, "sf_col given without q_col");
        const uintptr_t sa = (gran == FP8_SCALE_MX_1x32 || gran == FP8_SCALE_MX_1x32_OCP) ? 1 : 4;
        FP8_REQUIRE((!sf_row || aligned(sf_row, sa)) && (!sf_col || aligned(sf_col, sa)), FP8_ERR_INVALID_ARG,
                    "block scale tensors must be aligned to their element size");
    }
    FP8_REQUIRE(!amax || aligned(amax, 4), FP8_ERR_INVALID_ARG, "amax must be 4-byte aligned");
    FP8_REQUIRE(!q_row || aligned(q_row, 8), FP8_ERR_UNSUPPORTED, "q_row must be 8-byte aligned");
    if (q_col) {
        FP8_REQUIRE(rows % 16 == 0, FP8_ERR_UNSUPPORTED, "column-wise output needs rows %% 16 == 0 (rows=%lld)",
                    (long long)rows);
        FP8_REQUIRE(aligned(q_col, 16), FP8_ERR_UNSUPPORTED, "q_col must be 16-byte aligned");
    }
    return FP8_OK;
}

}  // namespace
}  // namespace fp8q

extern "C" {

fp8_status fp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt, fp8_granularity gran,
                        int32_t margin, const float* scale, uint8_t* q_row, uint8_t* q_col, void* sf_row,
                        void* sf_col, float* amax, void* stream) {
    g_detail[0] = 0;
    fp8_status s = check_quantize(x, rows, cols, ld, fmt, gran, scale, q_row, q_col, sf_row, sf_col, amax);
    if (s != FP8_OK || rows == 0 || cols == 0) return s;
    return launch_quantize(x, rows, cols, ld, fmt, gran, margin, scale, q_row, q_col, sf_row, sf_col, amax,
                           as_stream(stream));
}

fp8_status fp8_quantize_batch(const fp8_quantize_desc* descs, int32_t n, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(n >= 0 && n <= FP8_QUANTIZE_BATCH_MAX, FP8_ERR_INVALID_ARG, "n = %d outside [0, %d]", (int)n,
                FP8_QUANTIZE_BATCH_MAX);
    if (n == 0) return FP8_OK;
    FP8_REQUIRE(descs != nullptr, FP8_ERR_INVALID_ARG, "descs is NULL");
    for (int i = 0; i < n; ++i) {
        const fp8_quantize_desc& d = descs[i];
        FP8_REQUIRE(d.reserved == 0, FP8_ERR_INVALID_ARG, "descriptor %d: reserved must be 0", i);
        fp8_status s = check_quantize(d.x, d.rows, d.cols, d.ld, d.fmt, d.gran, d.scale, d.q_row, d.q_col, d.sf_row,
                                      d.sf_col, d.amax);
        if (s != FP8_OK) {
            char why[sizeof g_detail];
            snprintf(why, sizeof why, "%s", g_detail);
            set_error_detail("descriptor %d: %s", i, why);
            return s;
        }
    }
    return launch_quantize_batch(descs, n, as_stream(stream));
}

fp8_status fp8_quantize_current(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt, int32_t margin,
                                uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias, float* scale,
                                float* scale_inv, void* workspace, int32_t* status, void* stream) {
    g_detail[0] = 0;
    fp8_status s = check_bf16_matrix(x, rows, cols, ld);
    if (s != FP8_OK) return s;
    s = check_tma_dims(rows, cols);
    if (s != FP8_OK) return s;
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(workspace != nullptr, FP8_ERR_INVALID_ARG, "workspace is NULL");
    FP8_REQUIRE(aligned(workspace, 16), FP8_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    FP8_REQUIRE((!amax || aligned(amax, 4)) && (!bias || aligned(bias, 4)) && (!scale || aligned(scale, 4)) &&
                    (!scale_inv || aligned(scale_inv, 4)) && (!status || aligned(status, 4)),
                FP8_ERR_INVALID_ARG, "amax, bias, scale, scale_inv and status must be 4-byte aligned");
    if (rows > 0 && cols > 0) {
        FP8_REQUIRE(q_row || q_col, FP8_ERR_INVALID_ARG, "q_row and q_col are both NULL");
        FP8_REQUIRE(!q_row || aligned(q_row, 8), FP8_ERR_UNSUPPORTED, "q_row must be 8-byte aligned");
        if (q_col) {
            FP8_REQUIRE(rows % 16 == 0, FP8_ERR_UNSUPPORTED,
                        "column-wise output needs rows %% 16 == 0 (rows=%lld)", (long long)rows);
            FP8_REQUIRE(aligned(q_col, 16), FP8_ERR_UNSUPPORTED, "q_col must be 16-byte aligned");
        }
    }
    return launch_quantize_current(x, rows, cols, ld, fmt, margin, q_row, q_col, amax, bias, scale, scale_inv,
                                   workspace, status, as_stream(stream));
}

fp8_status fp8_quantize_current_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt,
                                        int32_t margin, uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias,
                                        float* scale, float* scale_inv, int32_t* status, void* stream) {
    g_detail[0] = 0;
    fp8_status s = check_bf16_matrix(x, rows, cols, ld);
    if (s != FP8_OK) return s;
    s = check_tma_dims(rows, cols);
    if (s != FP8_OK) return s;
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE((!amax || aligned(amax, 4)) && (!bias || aligned(bias, 4)) && (!scale || aligned(scale, 4)) &&
                    (!scale_inv || aligned(scale_inv, 4)) && (!status || aligned(status, 4)),
                FP8_ERR_INVALID_ARG, "amax, bias, scale, scale_inv and status must be 4-byte aligned");
    if (rows > 0 && cols > 0) {
        FP8_REQUIRE(q_row || q_col, FP8_ERR_INVALID_ARG, "q_row and q_col are both NULL");
        FP8_REQUIRE(!q_row || aligned(q_row, 8), FP8_ERR_UNSUPPORTED, "q_row must be 8-byte aligned");
        if (q_col) {
            FP8_REQUIRE(rows % 16 == 0, FP8_ERR_UNSUPPORTED,
                        "column-wise output needs rows %% 16 == 0 (rows=%lld)", (long long)rows);
            FP8_REQUIRE(aligned(q_col, 16), FP8_ERR_UNSUPPORTED, "q_col must be 16-byte aligned");
        }
    }
    return launch_quantize_current_noalloc(x, rows, cols, ld, fmt, margin, q_row, q_col, amax, bias, scale,
                                           scale_inv, status, as_stream(stream));
}

fp8_status fp8_set_bias(int32_t e, int32_t* bias, float* scale, float* scale_inv, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(e >= -126 && e <= 127, FP8_ERR_INVALID_ARG, "bias %d outside [-126, 127]", (int)e);
    FP8_REQUIRE(bias || scale || scale_inv, FP8_ERR_INVALID_ARG, "bias, scale and scale_inv are all NULL");
    FP8_REQUIRE((!bias || aligned(bias, 4)) && (!scale || aligned(scale, 4)) && (!scale_inv || aligned(scale_inv, 4)),
                FP8_ERR_INVALID_ARG, "bias, scale and scale_inv must be 4-byte aligned");
    return launch_set_bias(e, bias, scale, scale_inv, as_stream(stream));
}

fp8_status fp8_cast_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, fp8_format fmt, const float* scales,
                          int32_t n, uint64_t* saturated, uint64_t* underflow, void* stream) {
    g_detail[0] = 0;
    fp8_status s = check_bf16_matrix(x, rows, cols, ld);
    if (s != FP8_OK) return s;
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    FP8_REQUIRE(n >= 1 && n <= 8, FP8_ERR_INVALID_ARG, "n = %d scales (1 to 8)", (int)n);
    FP8_REQUIRE(scales && saturated && underflow, FP8_ERR_INVALID_ARG, "scales, saturated and underflow are required");
    FP8_REQUIRE(aligned(scales, 4) && aligned(saturated, 8) && aligned(underflow, 8), FP8_ERR_INVALID_ARG,
                "scales must be 4-byte and the counters 8-byte aligned");
    if (rows == 0 || cols == 0) return FP8_OK;
    return launch_cast_stats(x, rows, cols, ld, fmt, scales, n, saturated, underflow, as_stream(stream));
}

fp8_status fp8_quantize_f32(const float* x, int64_t n, fp8_format fmt, const float* scale, uint8_t* q, float* amax,
                            void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(n >= 0, FP8_ERR_INVALID_ARG, "negative size");
    FP8_REQUIRE(valid_fmt(fmt), FP8_ERR_INVALID_ARG, "unknown format %d", (int)fmt);
    if (n == 0) return FP8_OK;
    FP8_REQUIRE(x && q, FP8_ERR_INVALID_ARG, "x and q are required");
    FP8_REQUIRE(aligned(x, 16), FP8_ERR_UNSUPPORTED, "x must be 16-byte aligned");
    FP8_REQUIRE(aligned(q, 8), FP8_ERR_UNSUPPORTED, "q must be 8-byte aligned");
    FP8_REQUIRE((!scale || aligned(scale, 4)) && (!amax || aligned(amax, 4)), FP8_ERR_INVALID_ARG,
                "scale and amax must be 4-byte aligned");
    return launch_quantize_f32(x, n, fmt, scale, q, amax, as_stream(stream));
}

fp8_status fp8_scaled_gemm(fp8_gemm_op op, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                           fp8_format fa, fp8_granularity ga, const void* sfa, const uint8_t* B, int64_t ldb,
                           fp8_format fb, fp8_granularity gb, const void* sfb, void* D, fp8_out_dtype out_dtype,
                           int64_t ldd, int32_t* status, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(op == FP8_GEMM_FPROP || op == FP8_GEMM_DGRAD || op == FP8_GEMM_WGRAD, FP8_ERR_INVALID_ARG,
                "unknown gemm op %d", (int)op);
    FP8_REQUIRE(M >= 0 && N >= 0 && K >= 0, FP8_ERR_INVALID_ARG, "negative size");
    FP8_REQUIRE(valid_fmt(fa) && valid_fmt(fb), FP8_ERR_INVALID_ARG, "unknown format");
    FP8_REQUIRE(valid_gran(ga) && valid_gran(gb), FP8_ERR_INVALID_ARG, "unknown granularity");
    FP8_REQUIRE(out_dtype == FP8_OUT_F32 || out_dtype == FP8_OUT_BF16, FP8_ERR_INVALID_ARG, "unknown output dtype");
    FP8_REQUIRE((ga == FP8_SCALE_TENSOR) == (gb == FP8_SCALE_TENSOR), FP8_ERR_INVALID_ARG,
                "per-tensor scaling must be used for both operands or for neither");
    FP8_REQUIRE(ldd >= N, FP8_ERR_INVALID_ARG, "ldd < N");
    if (M == 0 || N == 0) return FP8_OK;
    FP8_REQUIRE(D != nullptr, FP8_ERR_INVALID_ARG, "D is NULL");
    const int esz = out_dtype == FP8_OUT_F32 ? 4 : 2;
    FP8_REQUIRE(N % 16 == 0 && ldd % 16 == 0, FP8_ERR_UNSUPPORTED, "N and ldd must be multiples of 16");
    FP8_REQUIRE(aligned(D, 16), FP8_ERR_UNSUPPORTED, "D must be 16-byte aligned");
    FP8_REQUIRE(M < (1ll << 31) && N < (1ll << 31) && K < (1ll << 31), FP8_ERR_UNSUPPORTED, "dimension >= 2^31");
    if (K == 0) {
        cudaError_t e = cudaMemset2DAsync(D, (size_t)ldd * esz, 0, (size_t)N * esz, (size_t)M, as_stream(stream));
        FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cudaMemset2DAsync: %s", cudaGetErrorString(e));
        return FP8_OK;
    }
    FP8_REQUIRE(A != nullptr && B != nullptr, FP8_ERR_INVALID_ARG, "A or B is NULL");
    FP8_REQUIRE(sfa != nullptr && sfb != nullptr, FP8_ERR_INVALID_ARG, "sfa and sfb are required");
    FP8_REQUIRE(lda >= K && ldb >= K, FP8_ERR_INVALID_ARG, "lda/ldb < K");
    FP8_REQUIRE(K % 16 == 0 && lda % 16 == 0 && ldb % 16 == 0, FP8_ERR_UNSUPPORTED,
                "K, lda and ldb must be multiples of 16");
    FP8_REQUIRE(aligned(A, 16) && aligned(B, 16), FP8_ERR_UNSUPPORTED, "A and B must be 16-byte aligned");
    if (ga != FP8_SCALE_TENSOR) {
        FP8_REQUIRE(K % 128 == 0, FP8_ERR_UNSUPPORTED, "block-scaled GEMM needs K %% 128 == 0");
        FP8_REQUIRE(aligned(sfa, 4) && aligned(sfb, 4), FP8_ERR_UNSUPPORTED, "scale tensors must be 4-byte aligned");
    } else {
        FP8_REQUIRE(aligned(sfa, 4) && aligned(sfb, 4), FP8_ERR_INVALID_ARG, "sfa/sfb must be 4-byte aligned");
    }
    return launch_gemm(M, N, K, A, lda, fa, ga, sfa, B, ldb, fb, gb, sfb, D, out_dtype == FP8_OUT_BF16 ? 1 : 0, ldd,
                       nullptr, nullptr, status, as_stream(stream));
}

fp8_status fp8_scaled_gemm_quantize(fp8_gemm_op op, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                                    fp8_format fa, const float* sfa, const uint8_t* B, int64_t ldb, fp8_format fb,
                                    const float* sfb, uint8_t* Dq, int64_t ldd, fp8_format fd, const float* scale_d,
                                    float* amax_d, int32_t* status, void* stream) {
    g_detail[0] = 0;
    FP8_REQUIRE(op == FP8_GEMM_FPROP || op == FP8_GEMM_DGRAD || op == FP8_GEMM_WGRAD, FP8_ERR_INVALID_ARG,
                "unknown gemm op %d", (int)op);
    FP8_REQUIRE(M >= 0 && N >= 0 && K >= 0, FP8_ERR_INVALID_ARG, "negative size");
    FP8_REQUIRE(valid_fmt(fa) && valid_fmt(fb) && valid_fmt(fd), FP8_ERR_INVALID_ARG, "unknown format");
    FP8_REQUIRE(ldd >= N, FP8_ERR_INVALID_ARG, "ldd < N");
    if (M == 0 || N == 0) return FP8_OK;
    FP8_REQUIRE(Dq != nullptr && scale_d != nullptr, FP8_ERR_INVALID_ARG, "Dq or scale_d is NULL");
    FP8_REQUIRE(aligned(scale_d, 4) && (!amax_d || aligned(amax_d, 4)), FP8_ERR_INVALID_ARG,
                "scale_d and amax_d must be 4-byte aligned");
    FP8_REQUIRE(N % 16 == 0 && ldd % 16 == 0, FP8_ERR_UNSUPPORTED, "N and ldd must be multiples of 16");
    FP8_REQUIRE(aligned(Dq, 16), FP8_ERR_UNSUPPORTED, "Dq must be 16-byte aligned");
    FP8_REQUIRE(M < (1ll << 31) && N < (1ll << 31) && K < (1ll << 31), FP8_ERR_UNSUPPORTED, "dimension >= 2^31");
    if (K == 0) {  // D = 0: every code is +0 and max|D| = 0 leaves amax_d as it is
        cudaError_t e = cudaMemset2DAsync(Dq, (size_t)ldd, 0, (size_t)N, (size_t)M, as_stream(stream));
        FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cudaMemset2DAsync: %s", cudaGetErrorString(e));
        return FP8_OK;
    }
    FP8_REQUIRE(A != nullptr && B != nullptr, FP8_ERR_INVALID_ARG, "A or B is NULL");
    FP8_REQUIRE(sfa != nullptr && sfb != nullptr, FP8_ERR_INVALID_ARG, "sfa and sfb are required");
    FP8_REQUIRE(lda >= K && ldb >= K, FP8_ERR_INVALID_ARG, "lda/ldb < K");
    FP8_REQUIRE(K % 16 == 0 && lda % 16 == 0 && ldb % 16 == 0, FP8_ERR_UNSUPPORTED,
                "K, lda and ldb must be multiples of 16");
    FP8_REQUIRE(aligned(A, 16) && aligned(B, 16), FP8_ERR_UNSUPPORTED, "A and B must be 16-byte aligned");
    FP8_REQUIRE(aligned(sfa, 4) && aligned(sfb, 4), FP8_ERR_INVALID_ARG, "sfa/sfb must be 4-byte aligned");
    return launch_gemm(M, N, K, A, lda, fa, FP8_SCALE_TENSOR, sfa, B, ldb, fb, FP8_SCALE_TENSOR, sfb, Dq,
                       fd == FP8_E4M3 ? 2 : 3, ldd, scale_d, amax_d, status, as_stream(stream));
}

}  // extern "C"
