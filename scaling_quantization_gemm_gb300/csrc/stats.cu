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
// product and conversion instruction the cast kernels use.  The pass over x
// (one 16-byte load per thread per step, grid-stride) then compares the two
// magnitudes of a 32-bit word with a threshold in one packed bf16x2 compare
// (a NaN compares false) and adds the two 0xFFFF / 0 lane masks into packed
// 16-bit counters that count down; flushed counts are |x| <= U_j less the
// zeros, counted once per word.
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

__device__ __forceinline__ uint32_t ge_mask2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t le_mask2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("set.le.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t eq_mask2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Lane-wise 16-bit add: adding a 0xFFFF mask lane takes one off that lane's count.
__device__ __forceinline__ uint32_t add_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Elements a packed count-down counter has seen in its two lanes.
__device__ __forceinline__ uint32_t down_count(uint32_t c) {
    return ((0x10000u - (c & 0xFFFFu)) & 0xFFFFu) + ((0x10000u - (c >> 16)) & 0xFFFFu);
}

// Both magnitudes of word w against every threshold pair (T2, U2: the bf16 threshold in both lanes).
template <int NS>
__device__ __forceinline__ void count2(uint32_t w, const uint32_t (&T2)[NS], const uint32_t (&U2)[NS],
                                       uint32_t (&ps)[NS], uint32_t (&pu)[NS], uint32_t& pz) {
    const uint32_t m = w & 0x7FFF7FFFu;
    pz = add_u16x2(pz, eq_mask2(m, 0u));
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        ps[j] = add_u16x2(ps[j], ge_mask2(m, T2[j]));
        pu[j] = add_u16x2(pu[j], le_mask2(m, U2[j]));
    }
}

template <int FMT, int NS>
__global__ void __launch_bounds__(kStatsThreads)
    cast_stats_kernel(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                      unsigned long long* saturated, unsigned long long* underflow) {
    __shared__ uint32_t sT[NS], sU[NS];
    // this CTA's counts: saturated per scale, |x| <= U_j per scale, zeros
    __shared__ unsigned long long cnt[2 * NS + 1];
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < NS) {
        uint32_t t = kInfMag + 1, u = 0;  // padding slots match nothing
        if (tid < n) thresholds<FMT>(scales[tid], t, u);
        sT[tid] = t;
        sU[tid] = u;
    }
    if (tid < 2 * NS + 1) cnt[tid] = 0;
    __syncthreads();
    uint32_t T2[NS], U2[NS], ps[NS], pu[NS], pz = 0;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        T2[j] = sT[j] * 0x10001u;
        U2[j] = sU[j] * 0x10001u;
        ps[j] = pu[j] = 0;
    }
    // a packed lane counts at most 16 per step (four 16-byte chunks): every 2048 steps a thread adds its
    // lanes into the CTA's counts (tensors of more than 2048 steps per thread only), and once at the end
    auto fold_thread = [&]() {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            const uint32_t a = down_count(ps[j]), b = down_count(pu[j]);
            if (a) atomicAdd(&cnt[j], (unsigned long long)a);
            if (b) atomicAdd(&cnt[NS + j], (unsigned long long)b);
            ps[j] = pu[j] = 0;
        }
        const uint32_t z = down_count(pz);
        if (z) atomicAdd(&cnt[2 * NS], (unsigned long long)z);
        pz = 0;
    };
    const int64_t cpr = cols >> 3;
    const int64_t total = rows * cpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    auto addr = [&](int64_t id) -> const uint16_t* {
        return (ld == cols) ? x + id * 8 : x + (id / cpr) * ld + (id % cpr) * 8;
    };
    auto count8 = [&](const uint4& v) {
        count2<NS>(v.x, T2, U2, ps, pu, pz);
        count2<NS>(v.y, T2, U2, ps, pu, pz);
        count2<NS>(v.z, T2, U2, ps, pu, pz);
        count2<NS>(v.w, T2, U2, ps, pu, pz);
    };
    int steps = 0;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + tid;
    for (; i + 3 * stride < total; i += 4 * stride) {  // four loads in flight per thread
        const uint4 v0 = ld_stream_v4(addr(i)), v1 = ld_stream_v4(addr(i + stride));
        const uint4 v2 = ld_stream_v4(addr(i + 2 * stride)), v3 = ld_stream_v4(addr(i + 3 * stride));
        count8(v0);
        count8(v1);
        count8(v2);
        count8(v3);
        if (++steps == 2048) {
            fold_thread();
            steps = 0;
        }
    }
    for (; i < total; i += stride) count8(ld_stream_v4(addr(i)));  // fewer than four steps: no fold needed
    // every lane is here: one sum per warp and count, one shared atomic
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const uint32_t a = __reduce_add_sync(0xffffffffu, down_count(ps[j]));
        const uint32_t b = __reduce_add_sync(0xffffffffu, down_count(pu[j]));
        if (lane == 0 && a) atomicAdd(&cnt[j], (unsigned long long)a);
        if (lane == 0 && b) atomicAdd(&cnt[NS + j], (unsigned long long)b);
    }
    const uint32_t z = __reduce_add_sync(0xffffffffu, down_count(pz));
    if (lane == 0 && z) atomicAdd(&cnt[2 * NS], (unsigned long long)z);
    __syncthreads();
    if (tid < 2 * NS && (tid % NS) < n) {
        // |x| <= U_j counted the zeros too
        const unsigned long long sum = tid < NS ? cnt[tid] : cnt[tid] - cnt[2 * NS];
        if (sum) atomicAdd(tid < NS ? &saturated[tid] : &underflow[tid - NS], sum);
    }
}

template <int FMT, int NS>
fp8_status launch_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                        uint64_t* saturated, uint64_t* underflow, cudaStream_t st) {
    auto k = cast_stats_kernel<FMT, NS>;
    int occ = 0;  // grid-stride CTAs: no more than fit at once (the thresholds are found once per CTA)
    fp8_status s = resident_ctas(reinterpret_cast<const void*>(k), kStatsThreads, 0, &occ);
    if (s != FP8_OK) return s;
    const int64_t chunks = rows * (cols / 8);
    int64_t grid = (chunks + kStatsThreads - 1) / kStatsThreads;
    const int64_t cap = (int64_t)device_sm_count() * occ;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    k<<<(int)grid, kStatsThreads, 0, st>>>(
        static_cast<const uint16_t*>(x), rows, cols, ld, scales, n, reinterpret_cast<unsigned long long*>(saturated),
        reinterpret_cast<unsigned long long*>(underflow));
    return check_launch("cast_stats kernel launch");
}

template <int FMT>
fp8_status launch_stats_fmt(const void* x, int64_t rows, int64_t cols, int64_t ld, const float* scales, int n,
                            uint64_t* saturated, uint64_t* underflow, cudaStream_t st) {
    // one instantiation per count: a padding slot would cost its compares and adds on every word
    switch (n) {
        case 1: return launch_stats<FMT, 1>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 2: return launch_stats<FMT, 2>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 3: return launch_stats<FMT, 3>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 4: return launch_stats<FMT, 4>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 5: return launch_stats<FMT, 5>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 6: return launch_stats<FMT, 6>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        case 7: return launch_stats<FMT, 7>(x, rows, cols, ld, scales, n, saturated, underflow, st);
        default: return launch_stats<FMT, kMaxScales>(x, rows, cols, ld, scales, n, saturated, underflow, st);
    }
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
