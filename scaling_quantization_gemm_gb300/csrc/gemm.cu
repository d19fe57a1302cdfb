// gemm.cu -- FP8 scaled GEMM on the 5th-generation tensor cores (tcgen05).
//
// D[m, n] = sum_k (A[m,k] sa) (B[n,k] sb): the FP8 product followed by the
// unscale ("Training and inference of large language models using 8-bit
// floating point", "Proposed method"), with per-tensor scales or with
// per-block / MXFP8 scales ("Per-Tensor and Per-Block Scaling Strategies for
// Effective FP8 Training", "Key Questions Answered").
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: 128x128-byte A tiles and 256x128-byte B tiles,
//               128-byte swizzle, into a 4-stage shared-memory ring.
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread); each
//               128-wide K tile is four K=32 MMAs.
//   warps 2-5   epilogue: TMEM -> registers (tcgen05.ld), unscale, convert,
//               store.  Each warp owns the 32 TMEM lanes (= tile rows) that
//               its warp index selects.
//   warps 6-9   (block-scaled kernel only) scale-factor writers: per K tile
//               they load the E8M0 (or power-of-two fp32) scales of the
//               tile's rows and store them into TMEM next to the accumulator.
// Per-tensor: two 128x256 fp32 accumulators in TMEM (512 columns), so the
// epilogue of one tile overlaps the main loop of the next; the unscale
// 2^-(ea+eb) is applied in the epilogue.  Block-scaled: the scales enter the
// MMA itself (kind::mxf8f6f4 with block_scale); one accumulator + scale
// columns.  Power-of-two fp32 block scales (1x128, 128x128) are re-encoded as
// E8M0 exactly and repeated over the four 32-wide K sub-blocks they cover.
//
// Every barrier wait is bounded (2 s); a wait that gives up raises a shared
// abort flag, every role leaves its loop, in-flight TMA loads and MMAs are
// drained, TMEM is released and FP8_STATUS_TIMEOUT is ORed into the status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"

namespace fp8q {

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;
constexpr int kBBytes = BN * BK;
constexpr int kGroupM = 16;  // tile raster: groups of 16 M-tiles walk N together (L2 reuse)

// TMEM layout of the block-scaled kernel.
constexpr int kSfColBase = 256;   // scale factors start after the 256 accumulator columns
constexpr int kSfColsPerStage = 16;  // 8 for A (4 used), 8 for B

// Scale-factor placement in TMEM for kind::mxf8f6f4, scale_vec::1X, M = 128:
// the scale of operand row r for the four 32-wide K sub-blocks of one K tile is
// one 32-bit word (byte i = sub-block i, selected by the MMA's scale-factor id)
// at lane 32*q + (r % 32) for every lane quarter q, column (r / 32) of the
// operand's scale region.
constexpr int kSfaCols = 4;  // 128 rows of A
constexpr int kSfbCols = 8;  // 256 rows of B

struct GemmArgs {
    int M, N, K;
    int tiles_m, tiles_n, k_tiles, num_tiles;
    void* D;
    int64_t ldd;
    const float* sa;  // per-tensor dequantisation factors
    const float* sb;
    const void* sfa;  // block scales
    const void* sfb;
    int ga, gb;
    int64_t sfa_ld, sfb_ld;  // row pitch of the scale tensors, in elements
    int32_t* status;
};

__device__ __forceinline__ void tile_coords(int t, const GemmArgs& g, int& tm, int& tn) {
    const int group = kGroupM * g.tiles_n;
    const int first_m = (t / group) * kGroupM;
    const int gsize = min(g.tiles_m - first_m, kGroupM);
    const int r = t % group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Store 32 consecutive fp32 accumulator values of one output row (16-column granularity).
template <int OUT_BF16>
__device__ __forceinline__ void store_row32(const GemmArgs& g, int64_t row, int64_t col0, const uint32_t (&r)[32],
                                            float sa, float sb) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (col0 + 16 * h >= g.N) break;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(__fmul_rn(__uint_as_float(r[16 * h + i]), sa), sb);
        if constexpr (OUT_BF16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.D) + row * g.ldd + col0 + 16 * h);
            dst[0] = make_uint4(cvt_bf16x2(v[0], v[1]), cvt_bf16x2(v[2], v[3]), cvt_bf16x2(v[4], v[5]), cvt_bf16x2(v[6], v[7]));
            dst[1] = make_uint4(cvt_bf16x2(v[8], v[9]), cvt_bf16x2(v[10], v[11]), cvt_bf16x2(v[12], v[13]),
                                cvt_bf16x2(v[14], v[15]));
        } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(g.D) + row * g.ldd + col0 + 16 * h);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    }
}

// Wait until the TMA loads last issued into each stage have landed (used only
// when the kernel is giving up, so that no copy writes shared memory after exit).
__device__ void drain_tma(uint64_t* full, const uint32_t* last_phase, const bool* used) {
    for (int s = 0; s < kStages; ++s) {
        if (!used[s]) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&full[s]), last_phase[s])) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
}

__device__ void drain_mma(uint64_t* bar) {
    tc_commit(smem_u32(bar));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(bar), 0)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
}

// ------------------------------------------------------------------ producer

__device__ __forceinline__ void producer_loop(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmArgs& g,
                                              uint8_t (*sa)[kABytes], uint8_t (*sb)[kBBytes], uint64_t* full,
                                              uint64_t* empty, volatile int* abort_flag) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t last_phase[kStages] = {0, 0, 0, 0};
    bool used[kStages] = {false, false, false, false};
    bool ok = true;
    for (int t = blockIdx.x; ok && t < g.num_tiles; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, g, tm, tn);
        for (int kt = 0; kt < g.k_tiles; ++kt) {
            if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(smem_u32(&full[stage]), kABytes + kBBytes);
            tma_load_2d(smem_u32(sa[stage]), tmA, smem_u32(&full[stage]), kt * BK, tm * BM);
            tma_load_2d(smem_u32(sb[stage]), tmB, smem_u32(&full[stage]), kt * BK, tn * BN);
            last_phase[stage] = phase;
            used[stage] = true;
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    if (!ok) drain_tma(full, last_phase, used);
}

// ============================================================ per-tensor GEMM

struct alignas(1024) SmemPT {
    uint8_t a[kStages][kABytes];
    uint8_t b[kStages][kBBytes];
    uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int OUT_BF16>
__global__ void __launch_bounds__(192, 1)
    gemm_tensor_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs g,
                       uint32_t idesc) {
    extern __shared__ uint8_t smem_raw[];
    SmemPT& S = *reinterpret_cast<SmemPT*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &S.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&S.tfull[a]), 1);
            mbar_init(smem_u32(&S.tempty[a]), 4);
        }
        mbar_init(smem_u32(&S.drain), 1);
        S.abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&S.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer_loop(&tmA, &tmB, g, S.a, S.b, S.full, S.empty, abort_flag);
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < g.num_tiles; t += gridDim.x) {
                if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), acc_phase ^ 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN);
                for (int kt = 0; kt < g.k_tiles; ++kt) {
                    if (!mbar_wait_bounded(smem_u32(&S.full[stage]), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(smem_u32(S.a[stage]));
                    const uint64_t bd = sdesc_kmajor_sw128(smem_u32(S.b[stage]));
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        tc_mma_f8f6f4(d, ad + 2 * k, bd + 2 * k, idesc, (kt | k) != 0 ? 1u : 0u);
                    tc_commit(smem_u32(&S.empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(smem_u32(&S.tfull[acc]));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            drain_mma(&S.drain);
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float sa = *g.sa, sb = *g.sb;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < g.num_tiles; t += gridDim.x) {
            bool ok = mbar_wait_bounded(smem_u32(&S.tfull[acc]), acc_phase, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            int tm, tn;
            tile_coords(t, g, tm, tn);
            const int64_t row = (int64_t)tm * BM + q * 32 + lane;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                const int64_t col0 = (int64_t)tn * BN + c * 32;
                if (row < g.M) store_row32<OUT_BF16>(g, row, col0, r, sa, sb);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0 && S.abort_flag && g.status) atomicOr(g.status, FP8_STATUS_TIMEOUT);
}

// ========================================================= block-scaled GEMM

struct alignas(1024) SmemBS {
    uint8_t a[kStages][kABytes];
    uint8_t b[kStages][kBBytes];
    uint64_t full[kStages], empty[kStages], tfull, tempty, drain;
    uint32_t tmem_base;
    int abort_flag;
    int bad_scale;
};

// fp32 power of two in [2^-127, 2^127] -> E8M0 code (its biased exponent).
__device__ __forceinline__ uint32_t e8m0_of_pow2(float f, bool& bad) {
    const uint32_t u = __float_as_uint(f);
    if (u == 0x00400000u) return 0;  // 2^-127 is the only subnormal power of two in range
    const uint32_t ex = (u >> 23) & 0xFFu;
    if ((u & 0x807FFFFFu) != 0 || ex == 0 || ex == 255) bad = true;
    return ex;
}

// The 32-bit scale word (four K sub-blocks of 32) of operand row `row` for K tile `kt`.
__device__ __forceinline__ uint32_t scale_word(const void* sf, int gran, int64_t ld, int64_t row, int64_t rows, int kt,
                                               bool& bad) {
    if (row >= rows) return 0x7F7F7F7Fu;  // rows past the edge hold zeros: any finite scale
    if (gran == FP8_SCALE_MX_1x32) return __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(sf) + row * ld) + kt);
    const float* f = static_cast<const float*>(sf);
    const float v = (gran == FP8_SCALE_BLOCK_1x128) ? __ldg(f + row * ld + kt) : __ldg(f + (row >> 7) * ld + kt);
    return e8m0_of_pow2(v, bad) * 0x01010101u;
}

template <int OUT_BF16>
__global__ void __launch_bounds__(320, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            GemmArgs g, uint32_t idesc) {
    extern __shared__ uint8_t smem_raw[];
    SmemBS& S = *reinterpret_cast<SmemBS*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &S.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1 + 4);  // TMA producer + four scale writers
            mbar_init(smem_u32(&S.empty[s]), 1);
        }
        mbar_init(smem_u32(&S.tfull), 1);
        mbar_init(smem_u32(&S.tempty), 4);
        mbar_init(smem_u32(&S.drain), 1);
        S.abort_flag = 0;
        S.bad_scale = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&S.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer_loop(&tmA, &tmB, g, S.a, S.b, S.full, S.empty, abort_flag);
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < g.num_tiles; t += gridDim.x) {
                if (!mbar_wait_bounded(smem_u32(&S.tempty), acc_phase ^ 1, abort_flag)) break;
                tc_fence_after();
                for (int kt = 0; kt < g.k_tiles; ++kt) {
                    if (!mbar_wait_bounded(smem_u32(&S.full[stage]), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(smem_u32(S.a[stage]));
                    const uint64_t bd = sdesc_kmajor_sw128(smem_u32(S.b[stage]));
                    const uint32_t sfa_t = tmem + (uint32_t)(kSfColBase + stage * kSfColsPerStage);
                    const uint32_t sfb_t = sfa_t + 8;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        tc_mma_mxf8f6f4(tmem, ad + 2 * k, bd + 2 * k, idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4),
                                        sfa_t, sfb_t, (kt | k) != 0 ? 1u : 0u);
                    tc_commit(smem_u32(&S.empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(smem_u32(&S.tfull));
                acc_phase ^= 1;
            }
            drain_mma(&S.drain);
        }
    } else if (warp < 6) {
        const int q = warp & 3;
        uint32_t acc_phase = 0;
        const float one = 1.0f;
        for (int t = blockIdx.x; t < g.num_tiles; t += gridDim.x) {
            bool ok = mbar_wait_bounded(smem_u32(&S.tfull), acc_phase, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            int tm, tn;
            tile_coords(t, g, tm, tn);
            const int64_t row = (int64_t)tm * BM + q * 32 + lane;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                const int64_t col0 = (int64_t)tn * BN + c * 32;
                if (row < g.M) store_row32<OUT_BF16>(g, row, col0, r, one, one);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.tempty));
            acc_phase ^= 1;
        }
    } else {
        // Scale-factor writers: warp (6..9) writes the lanes of quarter q = warp % 4.
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true, bad = false;
        for (int t = blockIdx.x; ok && t < g.num_tiles; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, g, tm, tn);
            const int64_t arow0 = (int64_t)tm * BM + lane, brow0 = (int64_t)tn * BN + lane;
            for (int kt0 = 0; ok && kt0 < g.k_tiles; kt0 += 4) {
                // Load four K tiles' worth of scale words at once (loads in flight together).
                uint32_t wa[4][kSfaCols], wb[4][kSfbCols];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int kt = min(kt0 + j, g.k_tiles - 1);
#pragma unroll
                    for (int c = 0; c < kSfaCols; ++c) wa[j][c] = scale_word(g.sfa, g.ga, g.sfa_ld, arow0 + 32 * c, g.M, kt, bad);
#pragma unroll
                    for (int c = 0; c < kSfbCols; ++c) wb[j][c] = scale_word(g.sfb, g.gb, g.sfb_ld, brow0 + 32 * c, g.N, kt, bad);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (kt0 + j >= g.k_tiles) break;
                    bool w = mbar_wait_bounded(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag);
                    w = __all_sync(0xffffffffu, w);
                    if (!w) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = tmem + lane_base + (uint32_t)(kSfColBase + stage * kSfColsPerStage);
                    tmem_st_32x32b_x4(col, wa[j][0], wa[j][1], wa[j][2], wa[j][3]);
                    tmem_st_32x32b_x4(col + 8, wb[j][0], wb[j][1], wb[j][2], wb[j][3]);
                    tmem_st_32x32b_x4(col + 12, wb[j][4], wb[j][5], wb[j][6], wb[j][7]);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&S.full[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&S.bad_scale, 1);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0 && g.status) {
        if (S.abort_flag) atomicOr(g.status, FP8_STATUS_TIMEOUT);
        if (S.bad_scale) atomicOr(g.status, FP8_STATUS_BAD_BLOCK_SCALE);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 2-D map over a K-major u8 matrix [rows x K] (row pitch ld bytes), box 128 bytes x box_rows, 128-byte swizzle.
fp8_status make_operand_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld, int box_rows) {
    auto fn = encode_fn();
    FP8_REQUIRE(fn != nullptr, FP8_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    FP8_REQUIRE(r == CUDA_SUCCESS, FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FP8_OK;
}

// Raise the dynamic shared-memory limit of `func` once per (function, device).
fp8_status prepare_kernel(const void* func, size_t smem) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({func, dev})) return FP8_OK;
    cudaError_t err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    FP8_REQUIRE(err == cudaSuccess, FP8_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(err));
    done.insert({func, dev});
    return FP8_OK;
}

}  // namespace

fp8_status launch_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int fa, int ga, const void* sfa,
                       const uint8_t* B, int64_t ldb, int fb, int gb, const void* sfb, void* D, int out_bf16,
                       int64_t ldd, int32_t* status, cudaStream_t st) {
    GemmArgs g;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    g.tiles_m = (int)((M + BM - 1) / BM);
    g.tiles_n = (int)((N + BN - 1) / BN);
    g.k_tiles = (int)((K + BK - 1) / BK);
    g.num_tiles = g.tiles_m * g.tiles_n;
    g.D = D;
    g.ldd = ldd;
    g.status = status;
    g.ga = ga;
    g.gb = gb;
    g.sa = g.sb = nullptr;
    g.sfa = g.sfb = nullptr;
    g.sfa_ld = g.sfb_ld = 0;

    CUtensorMap tmA, tmB;
    fp8_status s = make_operand_map(&tmA, A, M, K, lda, BM);
    if (s != FP8_OK) return s;
    s = make_operand_map(&tmB, B, N, K, ldb, BN);
    if (s != FP8_OK) return s;

    const int grid = std::min(g.num_tiles, device_sm_count());
    if (ga == FP8_SCALE_TENSOR) {
        g.sa = static_cast<const float*>(sfa);
        g.sb = static_cast<const float*>(sfb);
        const uint32_t idesc = idesc_f8f6f4(fa, fb, BM, BN);
        const size_t smem = sizeof(SmemPT) + 1024;
        if (out_bf16) {
            if ((s = prepare_kernel(reinterpret_cast<const void*>(gemm_tensor_kernel<1>), smem)) != FP8_OK) return s;
            gemm_tensor_kernel<1><<<grid, 192, smem, st>>>(tmA, tmB, g, idesc);
        } else {
            if ((s = prepare_kernel(reinterpret_cast<const void*>(gemm_tensor_kernel<0>), smem)) != FP8_OK) return s;
            gemm_tensor_kernel<0><<<grid, 192, smem, st>>>(tmA, tmB, g, idesc);
        }
        return check_launch("gemm_tensor_kernel launch");
    }
    g.sfa = sfa;
    g.sfb = sfb;
    const int64_t KT = (K + BK - 1) / BK;
    // row pitch of each scale tensor: MX in bytes-as-u32-words is handled by the word index (kt)
    g.sfa_ld = (ga == FP8_SCALE_MX_1x32) ? K / 32 : KT;
    g.sfb_ld = (gb == FP8_SCALE_MX_1x32) ? K / 32 : KT;
    const uint32_t idesc = idesc_mxf8f6f4(fa, fb, BM, BN, 0, 0);
    const size_t smem = sizeof(SmemBS) + 1024;
    if (out_bf16) {
        if ((s = prepare_kernel(reinterpret_cast<const void*>(gemm_blockscaled_kernel<1>), smem)) != FP8_OK) return s;
        gemm_blockscaled_kernel<1><<<grid, 320, smem, st>>>(tmA, tmB, g, idesc);
    } else {
        if ((s = prepare_kernel(reinterpret_cast<const void*>(gemm_blockscaled_kernel<0>), smem)) != FP8_OK) return s;
        gemm_blockscaled_kernel<0><<<grid, 320, smem, st>>>(tmA, tmB, g, idesc);
    }
    return check_launch("gemm_blockscaled_kernel launch");
}

}  // namespace fp8q
