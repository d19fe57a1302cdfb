// quantize.cu -- amax reduction, scale selection (current and delayed) and the
// fused scaled cast to FP8 with row-wise and column-wise outputs.
//
// Method: multiply by 2^e, then cast to FP8, with a per-tensor bias from the
// tensor's amax, e = floor(log2(fmax/amax)) - margin
// ("Training and inference of large language models using 8-bit floating
// point", "Proposed method"); delayed scaling from an amax history and
// per-block / MXFP8 scales ("Per-Tensor and Per-Block Scaling Strategies for
// Effective FP8 Training", "Key Questions Answered").
//
// All of it is HBM-bound.  The cast kernel reads each bf16 element once with
// 16-byte coalesced loads, computes block maxima in registers (warp shuffles),
// writes the row-wise codes straight from registers, and stages the tile in
// shared memory to produce the transposed column-wise codes, so one read feeds
// both outputs.  Amax is reduced per warp, per CTA, then one atomic per CTA.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace fp8q {

namespace {

constexpr int kTile = 128;          // tile is kTile x kTile bf16 elements
constexpr int kThreads = 256;
constexpr int kPitch = kTile + 8;   // smem row pitch in bf16 (272 bytes: conflict-free column reads)

struct QuantArgs {
    const uint16_t* x;
    int64_t rows, cols, ld;
    int margin;
    const float* scale;
    uint8_t* q_row;
    uint8_t* q_col;
    void* sf_row;
    void* sf_col;
    float* amax;
    int64_t tiles_c, ntiles;
    int do_row, do_col;
};

__device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int FMT>
__device__ __forceinline__ uint2 encode8(const uint4& v, float s) {
    uint32_t c0 = cvt_fp8x2<FMT>(__fmul_rn(bf16_lo(v.x), s), __fmul_rn(bf16_hi(v.x), s));
    uint32_t c1 = cvt_fp8x2<FMT>(__fmul_rn(bf16_lo(v.y), s), __fmul_rn(bf16_hi(v.y), s));
    uint32_t c2 = cvt_fp8x2<FMT>(__fmul_rn(bf16_lo(v.z), s), __fmul_rn(bf16_hi(v.z), s));
    uint32_t c3 = cvt_fp8x2<FMT>(__fmul_rn(bf16_lo(v.w), s), __fmul_rn(bf16_hi(v.w), s));
    return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

// Encode the low (HALF = 0) or high (HALF = 1) bf16 of 32 words (32 rows of one
// column) into 32 codes packed in 8 words, row order.
template <int FMT, int HALF>
__device__ __forceinline__ void encode_column32(const uint32_t (&w)[32], float s, uint32_t (&o)[8]) {
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float a0 = HALF ? bf16_hi(w[4 * p + 0]) : bf16_lo(w[4 * p + 0]);
        float a1 = HALF ? bf16_hi(w[4 * p + 1]) : bf16_lo(w[4 * p + 1]);
        float a2 = HALF ? bf16_hi(w[4 * p + 2]) : bf16_lo(w[4 * p + 2]);
        float a3 = HALF ? bf16_hi(w[4 * p + 3]) : bf16_lo(w[4 * p + 3]);
        uint32_t lo = cvt_fp8x2<FMT>(__fmul_rn(a0, s), __fmul_rn(a1, s));
        uint32_t hi = cvt_fp8x2<FMT>(__fmul_rn(a2, s), __fmul_rn(a3, s));
        o[p] = lo | (hi << 16);
    }
}

__device__ __forceinline__ void store_col32(uint8_t* q_col, int64_t c, int64_t rows, int64_t row0,
                                            const uint32_t (&o)[8]) {
    uint8_t* dst = q_col + c * rows + row0;
    if (row0 < rows) *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    if (row0 + 16 < rows) *reinterpret_cast<uint4*>(dst + 16) = make_uint4(o[4], o[5], o[6], o[7]);
}

// One CTA walks 128x128 tiles (grid-stride).  Thread t loads the 16-byte chunk
// column j = t % 16 of rows t/16 + 16 i, i = 0..7.
template <int GRAN, int FMT>
__global__ void __launch_bounds__(kThreads) quantize_tile_kernel(QuantArgs a) {
    __shared__ __align__(16) uint16_t sx[kTile * kPitch];
    __shared__ uint32_t red[2][8];
    __shared__ uint32_t col_part[4][64];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = tid & 15;
    const int rsub = tid >> 4;

    float s_tensor = 1.0f;
    if constexpr (GRAN == FP8_SCALE_TENSOR) s_tensor = *a.scale;

    uint32_t amax_acc = 0;
    int parity = 0;

    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, parity ^= 1) {
        const int64_t r0 = (tile / a.tiles_c) * kTile, c0 = (tile % a.tiles_c) * kTile;
        const int64_t col = c0 + 8 * j;
        const bool col_ok = col < a.cols;

        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t r = r0 + rsub + 16 * i;
            v[i] = (col_ok && r < a.rows) ? ld_stream_v4(a.x + r * a.ld + col) : make_uint4(0, 0, 0, 0);
        }
        uint32_t cm[8];  // |x| max of each loaded chunk, bf16 bits
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            cm[i] = fold2(absmax2(absmax2(absmax2(absmax2(0u, v[i].x), v[i].y), v[i].z), v[i].w));
            amax_acc = max(amax_acc, cm[i]);
        }

        // 128x128 blocks: one exponent for the whole tile, shared by both outputs.
        int e_tile = 0;
        if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, cm[i]);
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == 0) red[parity][warp] = m;
            __syncthreads();
            m = red[parity][0];
#pragma unroll
            for (int w = 1; w < 8; ++w) m = max(m, red[parity][w]);
            bool nf = false;
            e_tile = bias_from_amax(bf16bits_to_float(m), FMT, a.margin, &nf);
            if (tid == 0) {
                const int64_t tr = r0 / kTile, tc = c0 / kTile;
                if (a.do_row) static_cast<float*>(a.sf_row)[tr * cdiv(a.cols, kTile) + tc] = pow2_exact(-e_tile);
                if (a.do_col) static_cast<float*>(a.sf_col)[tc * cdiv(a.rows, kTile) + tr] = pow2_exact(-e_tile);
            }
        }

        // ---------------------------------------------------------- row-wise
        if (a.do_row) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t r = r0 + rsub + 16 * i;
                const bool ok = col_ok && r < a.rows;
                float s;
                if constexpr (GRAN == FP8_SCALE_TENSOR) {
                    s = s_tensor;
                } else if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
                    s = pow2_exact(e_tile);
                } else if constexpr (GRAN == FP8_SCALE_MX_1x32) {
                    uint32_t m = cm[i];
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    bool nf = false;
                    const int e = bias_from_amax(bf16bits_to_float(m), FMT, a.margin, &nf);
                    s = pow2_exact(e);
                    if ((j & 3) == 0 && ok)
                        static_cast<uint8_t*>(a.sf_row)[r * cdiv(a.cols, 32) + (col >> 5)] = (uint8_t)(127 - e);
                } else {  // 1x128
                    uint32_t m = cm[i];
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    bool nf = false;
                    const int e = bias_from_amax(bf16bits_to_float(m), FMT, a.margin, &nf);
                    s = pow2_exact(e);
                    if (j == 0 && r < a.rows)
                        static_cast<float*>(a.sf_row)[r * cdiv(a.cols, kTile) + c0 / kTile] = pow2_exact(-e);
                }
                if (ok) *reinterpret_cast<uint2*>(a.q_row + r * a.cols + col) = encode8<FMT>(v[i], s);
            }
        }

        // ------------------------------------------------------- column-wise
        if (a.do_col) {
#pragma unroll
            for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(&sx[(rsub + 16 * i) * kPitch + 8 * j]) = v[i];
            __syncthreads();
            const int cp = lane + 32 * (warp & 1);  // column pair within the tile
            const int seg = warp >> 1;              // 32-row segment within the tile
            uint32_t w[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) w[r] = *reinterpret_cast<const uint32_t*>(&sx[(32 * seg + r) * kPitch + 2 * cp]);
            uint32_t mm = 0;
#pragma unroll
            for (int r = 0; r < 32; ++r) mm = absmax2(mm, w[r]);

            float sA, sB;
            const int64_t ca = c0 + 2 * cp, cb = ca + 1;
            const int64_t row0 = r0 + 32 * seg;
            if constexpr (GRAN == FP8_SCALE_TENSOR) {
                sA = sB = s_tensor;
            } else if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
                sA = sB = pow2_exact(e_tile);
            } else if constexpr (GRAN == FP8_SCALE_MX_1x32) {
                bool nf = false;
                const int eA = bias_from_amax(bf16bits_to_float(mm & 0xFFFFu), FMT, a.margin, &nf);
                const int eB = bias_from_amax(bf16bits_to_float(mm >> 16), FMT, a.margin, &nf);
                sA = pow2_exact(eA);
                sB = pow2_exact(eB);
                if (row0 < a.rows) {
                    uint8_t* sf = static_cast<uint8_t*>(a.sf_col);
                    const int64_t nb = cdiv(a.rows, 32);
                    if (ca < a.cols) sf[ca * nb + (row0 >> 5)] = (uint8_t)(127 - eA);
                    if (cb < a.cols) sf[cb * nb + (row0 >> 5)] = (uint8_t)(127 - eB);
                }
            } else {  // 1x128 -> 128x1 column blocks: combine the four 32-row segments
                col_part[seg][cp] = mm;
                __syncthreads();
                uint32_t m4 = __vmaxu2(__vmaxu2(col_part[0][cp], col_part[1][cp]), __vmaxu2(col_part[2][cp], col_part[3][cp]));
                bool nf = false;
                const int eA = bias_from_amax(bf16bits_to_float(m4 & 0xFFFFu), FMT, a.margin, &nf);
                const int eB = bias_from_amax(bf16bits_to_float(m4 >> 16), FMT, a.margin, &nf);
                sA = pow2_exact(eA);
                sB = pow2_exact(eB);
                if (seg == 0) {
                    float* sf = static_cast<float*>(a.sf_col);
                    const int64_t nb = cdiv(a.rows, kTile);
                    if (ca < a.cols) sf[ca * nb + r0 / kTile] = pow2_exact(-eA);
                    if (cb < a.cols) sf[cb * nb + r0 / kTile] = pow2_exact(-eB);
                }
            }
            uint32_t o[8];
            if (ca < a.cols) {
                encode_column32<FMT, 0>(w, sA, o);
                store_col32(a.q_col, ca, a.rows, row0, o);
            }
            if (cb < a.cols) {
                encode_column32<FMT, 1>(w, sB, o);
                store_col32(a.q_col, cb, a.rows, row0, o);
            }
            __syncthreads();  // sx / col_part are rewritten by the next tile
        }
    }

    if (a.amax) {
        uint32_t m = __reduce_max_sync(0xffffffffu, amax_acc);
        __shared__ uint32_t am[8];
        __syncthreads();
        if (lane == 0) am[warp] = m;
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int w = 1; w < 8; ++w) m = max(m, am[w]);
            m = max(m, am[0]);
            atomicMax(reinterpret_cast<unsigned int*>(a.amax), m << 16);
        }
    }
}

// Standalone amax: grid-stride over 16-byte chunks, four loads in flight per thread.
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, float* amax) {
    const int64_t cpr = cols >> 3;
    const int64_t total = rows * cpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t m = 0;
    auto addr = [&](int64_t id) -> const uint16_t* {
        return (ld == cols) ? x + id * 8 : x + (id / cpr) * ld + (id % cpr) * 8;
    };
    for (; i + 3 * stride < total; i += 4 * stride) {
        uint4 v0 = ld_stream_v4(addr(i)), v1 = ld_stream_v4(addr(i + stride));
        uint4 v2 = ld_stream_v4(addr(i + 2 * stride)), v3 = ld_stream_v4(addr(i + 3 * stride));
        m = absmax2(absmax2(absmax2(absmax2(m, v0.x), v0.y), v0.z), v0.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v1.x), v1.y), v1.z), v1.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v2.x), v2.y), v2.z), v2.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v3.x), v3.y), v3.z), v3.w);
    }
    for (; i < total; i += stride) {
        uint4 v = ld_stream_v4(addr(i));
        m = absmax2(absmax2(absmax2(absmax2(m, v.x), v.y), v.z), v.w);
    }
    m = __reduce_max_sync(0xffffffffu, fold2(m));
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w]);
        m = max(m, red[0]);
        atomicMax(reinterpret_cast<unsigned int*>(amax), m << 16);
    }
}

__global__ void compute_scale_kernel(const float* amax, int fmt, int margin, int32_t* bias, float* scale,
                                     float* scale_inv, int32_t* status) {
    bool nf = false;
    const int e = bias_from_amax(*amax, fmt, margin, &nf);
    if (bias) *bias = e;
    if (scale) *scale = pow2_exact(e);
    if (scale_inv) *scale_inv = pow2_exact(-e);
    if (nf && status) atomicOr(status, FP8_STATUS_NONFINITE_AMAX);
}

// One delayed-scaling step in one CTA: record, window max, bias, reset.
__global__ void __launch_bounds__(1024) history_kernel(float* hist, int len, int64_t* pos, float* amax, int fmt,
                                                       int margin, int32_t* bias, float* scale, float* scale_inv,
                                                       int32_t* status) {
    __shared__ int64_t p_s;
    __shared__ uint32_t red[32];
    if (threadIdx.x == 0) {
        const int64_t p = *pos;
        hist[p % len] = *amax;
        p_s = p;
    }
    __syncthreads();
    const int64_t n = min(p_s + 1, (int64_t)len);
    uint32_t m = 0;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) m = max(m, __float_as_uint(hist[i]) & 0x7FFFFFFFu);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w]);
        m = max(m, red[0]);
        bool nf = false;
        const int e = bias_from_amax(__uint_as_float(m), fmt, margin, &nf);
        *bias = e;
        *scale = pow2_exact(e);
        *scale_inv = pow2_exact(-e);
        *amax = 0.0f;
        *pos = p_s + 1;
        if (nf && status) atomicOr(status, FP8_STATUS_NONFINITE_AMAX);
    }
}

template <int GRAN, int FMT>
int quant_grid(int64_t ntiles) {
    static int occ = [] {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, quantize_tile_kernel<GRAN, FMT>, kThreads, 0);
        return o > 0 ? o : 1;
    }();
    const int64_t cap = (int64_t)device_sm_count() * occ;
    return (int)(ntiles < cap ? ntiles : cap);
}

template <int GRAN, int FMT>
fp8_status launch_quant(const QuantArgs& a, cudaStream_t st) {
    const int grid = quant_grid<GRAN, FMT>(a.ntiles);
    quantize_tile_kernel<GRAN, FMT><<<grid, kThreads, 0, st>>>(a);
    return check_launch("quantize kernel launch");
}

}  // namespace

// ------------------------------------------------------------------- host API

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    static int cache[64] = {0};
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

fp8_status launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, float* amax, cudaStream_t st) {
    const int64_t chunks = rows * (cols / 8);
    int64_t grid = (chunks + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    amax_kernel<<<(int)grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), rows, cols, ld, amax);
    return check_launch("amax kernel launch");
}

fp8_status launch_compute_scale(const float* amax, int fmt, int margin, int32_t* bias, float* scale,
                                float* scale_inv, int32_t* status, cudaStream_t st) {
    compute_scale_kernel<<<1, 1, 0, st>>>(amax, fmt, margin, bias, scale, scale_inv, status);
    return check_launch("compute_scale kernel launch");
}

fp8_status launch_history(float* hist, int len, int64_t* pos, float* amax, int fmt, int margin, int32_t* bias,
                          float* scale, float* scale_inv, int32_t* status, cudaStream_t st) {
    const int threads = len >= 1024 ? 1024 : ((len + 31) / 32) * 32;
    history_kernel<<<1, threads, 0, st>>>(hist, len, pos, amax, fmt, margin, bias, scale, scale_inv, status);
    return check_launch("history kernel launch");
}

fp8_status launch_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int gran, int margin,
                           const float* scale, uint8_t* q_row, uint8_t* q_col, void* sf_row, void* sf_col,
                           float* amax, cudaStream_t st) {
    QuantArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.rows = rows;
    a.cols = cols;
    a.ld = ld;
    a.margin = margin;
    a.scale = scale;
    a.q_row = q_row;
    a.q_col = q_col;
    a.sf_row = sf_row;
    a.sf_col = sf_col;
    a.amax = amax;
    a.tiles_c = (cols + kTile - 1) / kTile;
    a.ntiles = ((rows + kTile - 1) / kTile) * a.tiles_c;
    a.do_row = q_row != nullptr;
    a.do_col = q_col != nullptr;
#define FP8Q_QDISPATCH(G)                                                         \
    case G:                                                                       \
        return fmt == FP8_E4M3 ? launch_quant<G, FP8_E4M3>(a, st) : launch_quant<G, FP8_E5M2>(a, st);
    switch (gran) {
        FP8Q_QDISPATCH(FP8_SCALE_TENSOR)
        FP8Q_QDISPATCH(FP8_SCALE_BLOCK_1x128)
        FP8Q_QDISPATCH(FP8_SCALE_BLOCK_128x128)
        FP8Q_QDISPATCH(FP8_SCALE_MX_1x32)
    }
#undef FP8Q_QDISPATCH
    return FP8_ERR_UNSUPPORTED;
}

}  // namespace fp8q
