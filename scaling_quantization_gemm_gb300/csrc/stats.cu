// stats.cu -- fixed (FP8-CSCALE) biases and the statistics of a cast at given scales.
//
// FP8-CSCALE keeps a fixed, user-chosen exponent bias per tensor where FP8-AMAX
// derives it from the amax; fixed biases only work in a narrow range ("Training
// and inference of large language models using 8-bit floating point",
// "Proposed method" and "Key findings", the fixed-scaling sweep).
//
//   set_bias_kernel    bias = e, scale = 2^e, scale_inv = 2^-e (one thread).
//   cast_stats_kernel  for up to 8 scales s_j at once, counts the elements the
//                      cast saturates (|fl32(x s_j)| > fmax) and the non-zero
//                      elements it flushes to zero (Encode(fl32(x s_j)) = +-0);
//                      NaN elements count in neither.
//
// The cast is monotone in |x|, so for each scale both sets are ranges of bf16
// magnitudes: saturated iff |x| >= T_j, flushed iff 0 < |x| <= U_j.  Every CTA
// finds T_j and U_j by bisection over the 2^15 magnitudes with the same fp32
// product and conversion instruction the cast kernels use; the pass over x is
// then two integer compares per element and scale (one 16-byte load per
// thread per step, grid-stride).
#include "common.cuh"

namespace fp8q {

namespace {

constexpr int kStatsThreads = 256;
constexpr int kMaxScales = 8;
constexpr uint32_t kInfMag = 0x7F80u;  // bf16 +inf; larger magnitudes are NaN

__global__ void set_bias_kernel(int e, int32_t* bias, float* scale, float* scale_inv) {
    if (bias) *bias = e;
    if (scale) *scale = pow2_exact(e);
    if (scale_inv) *scale_inv = pow2_exact(-e);
}

template <int FMT>
__device__ __forceinline__ bool saturates(uint32_t mag, float s) {
    const float v = __fmul_rn(__uint_as_float(mag << 16), s);
    return fabsf(v) > (FMT == FP8_E4M3 ? 448.0f : 57344.0f);  // false for NaN
}

template <int FMT>
__device__ __forceinline__ bool flushes(uint32_t mag, float s) {
    if (mag == 0) return false;
    const float v = __fmul_rn(__uint_as_float(mag << 16), s);
    return (cvt_fp8x2<FMT>(v, 0.0f) & 0x7Fu) == 0;
}

// T: smallest magnitude that saturates (kInfMag + 1 if none); U: largest that flushes (0 if none).
template <int FMT>
__device__ void thresholds(float s, uint32_t& T, uint32_t& U) {
    if (!saturates<FMT>(kInfMag, s)) {
        T = kInfMag + 1;
    } else {
        uint32_t lo = 0, hi = kInfMag;  // !saturates(lo) (0 never saturates), saturates(hi)
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (saturates<FMT>(mid, s))
                hi = mid;
            else
                lo = mid;
        }
        T = hi;
    }
    if (!flushes<FMT>(1, s)) {
        U = 0;
    } else if (flushes<FMT>(kInfMag, s)) {
        U = kInfMag;
    } else {
        uint32_t lo = 1, hi = kInfMag;  // flushes(lo), !flushes(hi)
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (flushes<FMT>(mid, s))
                lo = mid;
            else
                hi = mid;
        }
        U = lo;
    }
}

template <int NS>
__device__ __forceinline__ void count2(uint32_t w, const uint32_t (&T)[NS], const uint32_t (&U)[NS],
                                       uint32_t (&cs)[NS], uint32_t (&cu)[NS]) {
    uint32_t m0 = w & 0x7FFFu, m1 = (w >> 16) & 0x7FFFu;
    m0 = m0 > kInfMag ? 0u : m0;  // NaN counts in neither
    m1 = m1 > kInfMag ? 0u : m1;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        cs[j] += (m0 >= T[j]) + (m1 >= T[j]);
        cu[j] += (m0 - 1u < U[j]) + (m1 - 1u < U[j]);  // 0 wraps to 2^32 - 1: never counted
    }
}

template <int FMT, int NS>
__global__ void __launch_bounds__(kStatsThreads)
    cast_stats_kernel(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                      unsigned long long* saturated, unsigned long long* underflow) {
    __shared__ uint32_t sT[NS], sU[NS];
    __shared__ uint32_t red[kStatsThreads / 32][2 * NS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < NS) {
        uint32_t t = kInfMag + 1, u = 0;  // padding slots match nothing
        if (tid < n) thresholds<FMT>(scales[tid], t, u);
        sT[tid] = t;
        sU[tid] = u;
    }
    __syncthreads();
    uint32_t T[NS], U[NS], cs[NS], cu[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        T[j] = sT[j];
        U[j] = sU[j];
        cs[j] = cu[j] = 0;
    }
    const int64_t cpr = cols >> 3;
    const int64_t total = rows * cpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < total; i += stride) {
        const uint16_t* p = (ld == cols) ? x + i * 8 : x + (i / cpr) * ld + (i % cpr) * 8;
        const uint4 v = ld_stream_v4(p);
        count2<NS>(v.x, T, U, cs, cu);
        count2<NS>(v.y, T, U, cs, cu);
        count2<NS>(v.z, T, U, cs, cu);
        count2<NS>(v.w, T, U, cs, cu);
    }
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        cs[j] = __reduce_add_sync(0xffffffffu, cs[j]);
        cu[j] = __reduce_add_sync(0xffffffffu, cu[j]);
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            red[warp][j] = cs[j];
            red[warp][NS + j] = cu[j];
        }
    }
    __syncthreads();
    if (tid < 2 * NS && (tid % NS) < n) {
        unsigned long long sum = 0;
        for (int w = 0; w < kStatsThreads / 32; ++w) sum += red[w][tid];
        if (sum) atomicAdd(tid < NS ? &saturated[tid] : &underflow[tid - NS], sum);
    }
}

template <int FMT, int NS>
fp8_status launch_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                        uint64_t* saturated, uint64_t* underflow, cudaStream_t st) {
    const int64_t chunks = rows * (cols / 8);
    int64_t grid = (chunks + kStatsThreads - 1) / kStatsThreads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cast_stats_kernel<FMT, NS><<<(int)grid, kStatsThreads, 0, st>>>(
        static_cast<const uint16_t*>(x), rows, cols, ld, scales, n, reinterpret_cast<unsigned long long*>(saturated),
        reinterpret_cast<unsigned long long*>(underflow));
    return check_launch("cast_stats kernel launch");
}

template <int FMT>
fp8_status launch_stats_fmt(const void* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                            uint64_t* saturated, uint64_t* underflow, cudaStream_t st) {
    if (n <= 1) return launch_stats<FMT, 1>(x, rows, cols, ld, scales, n, saturated, underflow, st);
    if (n <= 2) return launch_stats<FMT, 2>(x, rows, cols, ld, scales, n, saturated, underflow, st);
    if (n <= 4) return launch_stats<FMT, 4>(x, rows, cols, ld, scales, n, saturated, underflow, st);
    return launch_stats<FMT, kMaxScales>(x, rows, cols, ld, scales, n, saturated, underflow, st);
}

}  // namespace

fp8_status launch_set_bias(int e, int32_t* bias, float* scale, float* scale_inv, cudaStream_t st) {
    set_bias_kernel<<<1, 1, 0, st>>>(e, bias, scale, scale_inv);
    return check_launch("set_bias kernel launch");
}

fp8_status launch_cast_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, const float* scales,
                             int n, uint64_t* saturated, uint64_t* underflow, cudaStream_t st) {
    return fmt == FP8_E4M3 ? launch_stats_fmt<FP8_E4M3>(x, rows, cols, ld, scales, n, saturated, underflow, st)
                           : launch_stats_fmt<FP8_E5M2>(x, rows, cols, ld, scales, n, saturated, underflow, st);
}

}  // namespace fp8q
