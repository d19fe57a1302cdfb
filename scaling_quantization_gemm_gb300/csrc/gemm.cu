// gemm.cu -- FP8 scaled GEMM on the 5th-generation tensor cores (tcgen05).
//
// D[m, n] = sum_k (A[m,k] sa) (B[n,k] sb): the FP8 product followed by the
// unscale ("Training and inference of large language models using 8-bit
// floating point", "Proposed method"), with per-tensor scales or with
// per-block / MXFP8 scales ("Per-Tensor and Per-Block Scaling Strategies for
// Effective FP8 Training", "Key Questions Answered").
//
// Design (persistent, warp-specialised, one CTA per SM):
//   warp 0      TMA producer: A and B tiles (128-byte rows of a 128-wide K
//               tile, 128-byte swizzle) into a shared-memory ring.
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread); each
//               128-wide K tile is four K=32 MMAs.
//   warps 2-5   epilogue: TMEM -> registers (tcgen05.ld), unscale, convert
//               (fp32, bf16, or E4M3/E5M2 with a given scale and a fused amax),
//               store (the pair kernels stage 32x32 chunks in shared memory and
//               store them with TMA).  Each warp owns the 32 TMEM lanes (= tile
//               rows) that its warp index selects.
//   warps 6-9   (block-scaled kernels only) scale-factor writers.
// Two fp32 accumulators live in TMEM so the epilogue of one tile overlaps the
// main loop of the next.  M > 128 runs on CTA pairs (clusters of two, tcgen05
// cta_group::2: the even CTA issues the MMAs for both SMs); M <= 128 runs the
// one-CTA kernels.
// Per-tensor: 256x256 tiles per pair (128x256 per CTA), 6 stages of one K
// tile; the unscale 2^-(ea+eb) is applied in the epilogue.
// Block-scaled: the scales enter the MMA itself (kind::mxf8f6f4 with
// block_scale, E8M0 scale per 32 K).  Tiles are 256x224 per pair so that two
// accumulators (448 columns) and four 16-column scale slots fit the 512 TMEM
// columns; stages hold two K tiles.  Power-of-two fp32 block scales (1x128,
// 128x128) are re-encoded as E8M0 exactly and repeated over the four 32-wide K
// sub-blocks they cover.  The scale writers store into TMEM the cells the MMA
// reads: the scale of A row m at lane m, column m/32; the scale of B row n at
// lane 32q + n%32, column n/32, in every lane quarter q (each quarter of the
// tensor core reads its own copy); byte = K sub-block.
//
// Every barrier wait is bounded (2 s); a wait that gives up raises a shared
// abort flag, every role leaves its loop, in-flight TMA loads and MMAs are
// drained, TMEM is released and FP8_STATUS_TIMEOUT is ORed into the status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <map>
#include <utility>

#include "common.cuh"

namespace fp8q {

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;
constexpr int kBBytes = BN * BK;
constexpr int kGroupM = 16;  // tile raster: groups of 16 M-tiles walk N together (L2 reuse)

// Block-scaled kernel: tile width, TMEM layout.
constexpr int BN_BS = 224;
constexpr int kBBytesBS = BN_BS * BK;
constexpr int kSfColBase = 2 * BN_BS;  // scale slots start after the two accumulators (448)
constexpr int kSfColsPerStage = 16;    // A scales at +0 (4 columns), B scales at +8 (up to 8 columns)
constexpr int kSfbCols = (BN_BS + 31) / 32;
static_assert(kSfbCols <= 8, "B scales of a tile fill at most eight TMEM columns");

// Block-scaled CTA-pair kernel: pair tile width and TMEM layout (accumulators, then scale slots).
// Measured on the MXFP8 and per-block shapes: 224 columns with two accumulators beat 192 with eight
// scale slots and 256 with one accumulator (a stage costs about the same beyond its arithmetic
// whatever the width -- the tensor core waits on the kernel's other traffic, not on the MMA -- so
// narrower tiles lose, and one accumulator exposes the epilogue).
constexpr int kBnPair = 224;   // output columns (B rows) of a pair tile
constexpr int kAccBufs = 2;    // accumulators: with two, a tile's epilogue overlaps the next tile's MMAs
constexpr int kSfColBasePair = kAccBufs * kBnPair;
constexpr int kSfbColsPair = (kBnPair + 31) / 32;
static_assert(kSfbColsPair <= 8, "B scales of a tile fill at most eight TMEM columns");

enum { SF_MX = 0, SF_ROW = 1, SF_BLOCK = 2 };  // E8M0 1x32 | fp32 per row (1x128) | fp32 per 128 rows (128x128)

struct GemmArgs {
    int M, N, K;
    int tiles_m, tiles_n, k_tiles, num_tiles;
    void* D;
    int64_t ldd;
    const float* sa;  // per-tensor dequantisation factors
    const float* sb;
    const void* sfa;  // block scales
    const void* sfb;
    int64_t sfa_ld, sfb_ld;  // row pitch of the scale tensors in elements (bytes for E8M0, floats for fp32)
    int vec_a, vec_b;        // scale rows allow 16-byte loads of four K tiles
    int pair;                // CTA-pair kernel (256-row tiles)
    int32_t* status;
    const float* sd;  // FP8 output: scale 2^e applied before the cast
    float* amax_d;    // FP8 output: max |D| before that scale is accumulated here (or NULL)
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

// FP8 output (the next layer's cast fused into this epilogue): 32 values of one row
// v = (acc sa) sb, code = RNE_sat(v sd), max |v| folded into `amax` (as bits, so a NaN wins).
template <int FMT>
__device__ __forceinline__ void store_row32_fp8(const GemmArgs& g, int64_t row, int64_t col0, const uint32_t (&r)[32],
                                                float sa, float sb, float sd, uint32_t& amax) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (col0 + 16 * h >= g.N) break;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v0 = __fmul_rn(__fmul_rn(__uint_as_float(r[16 * h + 2 * i]), sa), sb);
            const float v1 = __fmul_rn(__fmul_rn(__uint_as_float(r[16 * h + 2 * i + 1]), sa), sb);
            amax = max(amax, max(__float_as_uint(v0) & 0x7FFFFFFFu, __float_as_uint(v1) & 0x7FFFFFFFu));
            const uint32_t c = cvt_fp8x2<FMT>(__fmul_rn(v0, sd), __fmul_rn(v1, sd));
            if (i & 1)
                w[i >> 1] |= c << 16;
            else
                w[i >> 1] = c;
        }
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.D) + row * g.ldd + col0 + 16 * h) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Store one accumulator row chunk for output kind OUT: 0 fp32, 1 bf16, 2 E4M3, 3 E5M2.
template <int OUT>
__device__ __forceinline__ void store_out(const GemmArgs& g, int64_t row, int64_t col0, const uint32_t (&r)[32],
                                          float sa, float sb, float sd, uint32_t& amax) {
    if constexpr (OUT >= 2)
        store_row32_fp8<OUT - 2>(g, row, col0, r, sa, sb, sd, amax);
    else
        store_row32<OUT>(g, row, col0, r, sa, sb);
}

// Epilogue through TMA stores.  Each epilogue warp owns a 4 KB staging buffer in shared memory; a
// 32-row x 32-column output chunk (row `lane` from each lane) is written into it in the swizzle of the
// output tensor map (fp32 rows of 128 bytes: 128-byte swizzle; bf16, 64 bytes: 64-byte swizzle; FP8,
// 32 bytes: 32-byte swizzle -- 16-byte chunk j of row r at j ^ (r % 8), j ^ (r / 2 % 4), j ^ (r / 4 % 2),
// which puts a warp's 16-byte stores in distinct bank groups), then one thread issues one
// cp.async.bulk.tensor store of the chunk, which the tensor map clips at the edges of D.  Chunks
// rotate through the buffer's 4096 / chunk-bytes slots; before a slot is reused the store that last
// read it must be done reading (cp.async.bulk.wait_group.read).
constexpr int kOutStageBytes = 4096;
template <int OUT>
__host__ __device__ constexpr int out_chunk_bytes() { return OUT == 0 ? 4096 : OUT == 1 ? 2048 : 1024; }
template <int OUT>
__host__ __device__ constexpr int out_slots() { return kOutStageBytes / out_chunk_bytes<OUT>(); }

// Stage row `lane` of a chunk: values v = (acc sa) sb (SCALED) or acc; FP8 outputs hold the codes of
// v sd, and fold max |v| into `amax` (as bits, so a NaN wins).
template <int OUT, bool SCALED>
__device__ __forceinline__ void stage_out_row(uint32_t slot, int lane, const uint32_t (&r)[32], float sa, float sb,
                                              float sd, uint32_t& amax) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = SCALED ? __fmul_rn(__fmul_rn(__uint_as_float(r[i]), sa), sb) : __uint_as_float(r[i]);
    if constexpr (OUT == 0) {
        const uint32_t line = slot + (uint32_t)lane * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(line + ((uint32_t)(j ^ (lane & 7)) << 4), __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                         __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
    } else if constexpr (OUT == 1) {
        const uint32_t line = slot + (uint32_t)lane * 64u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_shared_v4(line + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4), cvt_bf16x2(v[8 * j], v[8 * j + 1]),
                         cvt_bf16x2(v[8 * j + 2], v[8 * j + 3]), cvt_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                         cvt_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            amax = max(amax, max(__float_as_uint(v[2 * i]) & 0x7FFFFFFFu, __float_as_uint(v[2 * i + 1]) & 0x7FFFFFFFu));
            const uint32_t c = cvt_fp8x2<OUT - 2>(__fmul_rn(v[2 * i], sd), __fmul_rn(v[2 * i + 1], sd));
            if (i & 1)
                w[i >> 1] |= c << 16;
            else
                w[i >> 1] = c;
        }
        const uint32_t line = slot + (uint32_t)lane * 32u;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            st_shared_v4(line + ((uint32_t)(j ^ ((lane >> 2) & 1)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
}

// One chunk through the warp's staging buffer: `nchunk` counts the warp's chunks (slot rotation).
// Rows row0 .. row0 + 31 of D, columns col0 .. col0 + 31; nothing is stored when all lie outside D.
template <int OUT, bool SCALED>
__device__ __forceinline__ void store_chunk_tma(const CUtensorMap* tmD, uint32_t buf, uint32_t& nchunk, int lane,
                                                const uint32_t (&r)[32], float sa, float sb, float sd, uint32_t& amax,
                                                int64_t row0, int64_t col0, const GemmArgs& g) {
    const uint32_t slot = buf + (nchunk % (uint32_t)out_slots<OUT>()) * (uint32_t)out_chunk_bytes<OUT>();
    ++nchunk;
    if (lane == 0) bulk_wait_read<out_slots<OUT>() - 1>();  // the store that last read `slot` is done reading
    __syncwarp();
    stage_out_row<OUT, SCALED>(slot, lane, r, sa, sb, sd, amax);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row0 < g.M && col0 < g.N) tma_store_2d(tmD, slot, (int)col0, (int)row0);
        bulk_commit();
    }
}

// End of an epilogue warp: fold the warp's amax into the caller's accumulator.
template <int OUT>
__device__ __forceinline__ void flush_amax(const GemmArgs& g, uint32_t amax) {
    if constexpr (OUT >= 2) {
        amax = __reduce_max_sync(0xffffffffu, amax);
        if ((threadIdx.x & 31) == 0 && g.amax_d != nullptr) atomicMax(reinterpret_cast<unsigned int*>(g.amax_d), amax);
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

template <int BN_>
__device__ __forceinline__ void producer_loop(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmArgs& g,
                                              uint8_t (*sa)[kABytes], uint8_t (*sb)[BN_ * BK], uint64_t* full,
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
            mbar_arrive_expect_tx(smem_u32(&full[stage]), kABytes + BN_ * BK);
            tma_load_2d(smem_u32(sa[stage]), tmA, smem_u32(&full[stage]), kt * BK, tm * BM);
            tma_load_2d(smem_u32(sb[stage]), tmB, smem_u32(&full[stage]), kt * BK, tn * BN_);
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

template <int OUT>
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
        if (lane == 0) producer_loop<BN>(&tmA, &tmB, g, S.a, S.b, S.full, S.empty, abort_flag);
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
        const float sd = OUT >= 2 ? *g.sd : 1.0f;
        uint32_t amax = 0;
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
                if (row < g.M) store_out<OUT>(g, row, col0, r, sa, sb, sd, amax);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        flush_amax<OUT>(g, amax);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0 && S.abort_flag && g.status) atomicOr(g.status, FP8_STATUS_TIMEOUT);
}

// ======================================================= per-tensor GEMM, CTA pair

// Two CTAs on two SMs compute one 256x256 tile with tcgen05.mma.cta_group::2:
// each CTA holds 128 rows of A and 128 rows of B per K tile (32 KB per stage,
// 6 stages) and 128 rows of the accumulator in its own TMEM.  The even CTA of
// the pair issues the MMAs for both.  Both producers signal the even CTA's
// `full` barrier; the MMA commits arrive on the `empty` / `tfull` barriers of
// both CTAs; both epilogues release an accumulator on the even CTA's `tempty`.
constexpr int kPairStages = 6;
constexpr int kPairRows = 128;                      // rows of A and of B per CTA per tile
constexpr int kPairTile = 2 * kPairRows;            // 256 x 256 output tile per pair
constexpr int kPairHalfBytes = kPairRows * BK;      // 16 KB
constexpr int kPairStageBytes = 2 * kPairHalfBytes; // A half + B half, per CTA

struct alignas(1024) SmemPair {
    uint8_t a[kPairStages][kPairHalfBytes];
    uint8_t b[kPairStages][kPairHalfBytes];
    alignas(1024) uint8_t out[4][kOutStageBytes];  // per epilogue warp: staged output chunks for TMA stores
    uint64_t full[kPairStages], empty[kPairStages], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};

static_assert(sizeof(SmemPair) + 1024 <= 232448, "the pair kernel's shared memory fits one SM (227 KB)");

template <int OUT>
__global__ void __launch_bounds__(192, 1)
    gemm_tensor_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmD, GemmArgs g, uint32_t idesc) {
    extern __shared__ uint8_t smem_raw[];
    SmemPair& S = *reinterpret_cast<SmemPair*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs of the pair
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    volatile int* abort_flag = &S.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(smem_u32(&S.full[s]), 2);   // one expect_tx arrival from each producer of the pair
            mbar_init(smem_u32(&S.empty[s]), 1);  // the MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&S.tfull[a]), 1);
            mbar_init(smem_u32(&S.tempty[a]), 8);  // four epilogue warps in each CTA
        }
        mbar_init(smem_u32(&S.drain), 1);
        S.abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&S.tmem_base), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = cid; ok && t < g.num_tiles; t += ncl) {
                int tm, tn;
                tile_coords(t, g, tm, tn);
                for (int kt = 0; kt < g.k_tiles; ++kt) {
                    if (!mbar_wait_bounded(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = map_to_cta(smem_u32(&S.full[stage]), 0);
                    mbar_arrive_expect_tx_cluster(full_leader, kPairStageBytes);
                    tma_load_2d_pair(smem_u32(S.a[stage]), &tmA, full_leader, kt * BK, tm * kPairTile + (int)rank * kPairRows);
                    tma_load_2d_pair(smem_u32(S.b[stage]), &tmB, full_leader, kt * BK, tn * kPairTile + (int)rank * kPairRows);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {  // giving up: the loads signal the other CTA's barrier, so just let them land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = cid; ok && t < g.num_tiles; t += ncl) {
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
                        tc_mma_f8f6f4_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kt | k) != 0 ? 1u : 0u);
                    tc_commit_pair_multicast(smem_u32(&S.empty[stage]), 0x3);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit_pair_multicast(smem_u32(&S.tfull[acc]), 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            tc_commit_pair(smem_u32(&S.drain));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&S.drain), 0))
                if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    } else {
        const int q = warp & 3;
        const float sa = *g.sa, sb = *g.sb;
        const float sd = OUT >= 2 ? *g.sd : 1.0f;
        uint32_t amax = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t obuf = smem_u32(S.out[q]);
        uint32_t nchunk = 0;  // chunks this warp has staged
        for (int t = cid; t < g.num_tiles; t += ncl) {
            bool ok = mbar_wait_bounded(smem_u32(&S.tfull[acc]), acc_phase, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            int tm, tn;
            tile_coords(t, g, tm, tn);
            const int64_t row0 = (int64_t)tm * kPairTile + (int64_t)rank * kPairRows + q * 32;  // this warp's rows
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                const int64_t col0 = (int64_t)tn * kPairTile + c * 32;
                store_chunk_tma<OUT, true>(&tmD, obuf, nchunk, lane, r, sa, sb, sd, amax, row0, col0, g);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&S.tempty[acc]), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) bulk_wait_all();  // this warp's stores are complete before the CTA exits
        flush_amax<OUT>(g, amax);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may still signal its barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
    if (threadIdx.x == 0 && S.abort_flag && g.status) atomicOr(g.status, FP8_STATUS_TIMEOUT);
}

// ========================================================= block-scaled GEMM

struct alignas(1024) SmemBS {
    uint8_t a[kStages][kABytes];
    uint8_t b[kStages][kBBytesBS];
    uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int bad_scale;
};

// fp32 power of two in [2^-127, 2^127] -> E8M0 code (its biased exponent), branch-free.  Any other
// value ORs a non-zero bit into `bad` (a register, not a flag in memory).
__device__ __forceinline__ uint32_t e8m0_of_pow2(float f, uint32_t& bad) {
    const uint32_t u = __float_as_uint(f);
    const uint32_t ex = (u >> 23) & 0xFFu;
    const uint32_t sub = (u == 0x00400000u);  // 2^-127, the only subnormal power of two in range
    bad |= (1u - sub) & (uint32_t)(((u & 0x807FFFFFu) != 0) | (ex == 0) | (ex == 255));
    return sub ? 0u : ex;
}

template <int KIND>
__device__ __forceinline__ uint32_t sf_neutral() {
    return KIND == SF_MX ? 0x7F7F7F7Fu : 0x3F800000u;  // scale 1.0 (rows past the edge hold zeros)
}

// Raw scale data of operand row `row` for the four K tiles kt0 .. kt0+3: E8M0
// words (four bytes = four 32-wide K sub-blocks each) or fp32 bit patterns.
template <int KIND>
__device__ __forceinline__ uint4 sf_load_group(const void* sf, int64_t ld, int64_t row, int64_t rows, int kt0,
                                               int k_tiles, bool vec) {
    const uint32_t z = sf_neutral<KIND>();
    uint4 r = make_uint4(z, z, z, z);
    if (row >= rows) return r;
    const uint32_t* p;
    if constexpr (KIND == SF_MX)
        p = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(sf) + row * ld) + kt0;
    else
        p = reinterpret_cast<const uint32_t*>(static_cast<const float*>(sf) + (KIND == SF_ROW ? row : (row >> 7)) * ld) +
            kt0;
    if (vec && kt0 + 4 <= k_tiles) return __ldg(reinterpret_cast<const uint4*>(p));
    r.x = __ldg(p);
    if (kt0 + 1 < k_tiles) r.y = __ldg(p + 1);
    if (kt0 + 2 < k_tiles) r.z = __ldg(p + 2);
    if (kt0 + 3 < k_tiles) r.w = __ldg(p + 3);
    return r;
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

template <int KIND>
__device__ __forceinline__ uint32_t sf_word(uint32_t raw, uint32_t& bad) {
    if constexpr (KIND == SF_MX) return raw;
    return e8m0_of_pow2(__uint_as_float(raw), bad) * 0x01010101u;
}

struct SfGroup {
    uint4 a;
    uint4 b[kSfbCols];
};

template <int OUT_BF16, int KA, int KB>
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
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&S.tfull[a]), 1);
            mbar_init(smem_u32(&S.tempty[a]), 4);
        }
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
        if (lane == 0) producer_loop<BN_BS>(&tmA, &tmB, g, S.a, S.b, S.full, S.empty, abort_flag);
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < g.num_tiles; t += gridDim.x) {
                if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), acc_phase ^ 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN_BS);
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
                        tc_mma_mxf8f6f4(d, ad + 2 * k, bd + 2 * k, idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4),
                                        sfa_t, sfb_t, (kt | k) != 0 ? 1u : 0u);
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
    } else if (warp < 6) {
        const int q = warp & 3;
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
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN_BS);
#pragma unroll 1
            for (int c = 0; c < BN_BS / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                const int64_t col0 = (int64_t)tn * BN_BS + c * 32;
                if (row < g.M) store_row32<OUT_BF16>(g, row, col0, r, 1.0f, 1.0f);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    } else {
        // Scale-factor writers: warp 6..9 owns TMEM lane quarter q = warp % 4.  Each quarter of the
        // tensor core reads scales from its own 32 lanes: the A scale of its rows 32q + l (column q of
        // the slot) and the B scales of all tile columns n (columns 8 + n/32 at lane 32q + n % 32), so
        // every writer stores its A column and a full copy of the B columns.  Scales are loaded one
        // group of four K tiles ahead of use.
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int groups = (g.k_tiles + 3) / 4;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t bad = 0;

        auto load = [&](int t, int grp, SfGroup& dst) {
            int tm, tn;
            tile_coords(t, g, tm, tn);
            dst.a = sf_load_group<KA>(g.sfa, g.sfa_ld, (int64_t)tm * BM + q * 32 + lane, g.M, 4 * grp, g.k_tiles,
                                      g.vec_a);
#pragma unroll
            for (int j = 0; j < kSfbCols; ++j)
                dst.b[j] = sf_load_group<KB>(g.sfb, g.sfb_ld, (int64_t)tn * BN_BS + 32 * j + lane, g.N, 4 * grp,
                                             g.k_tiles, g.vec_b);
        };
        auto emit = [&](const SfGroup& src, int grp) -> bool {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                if (4 * grp + jj >= g.k_tiles) break;
                bool w = mbar_wait_bounded(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag);
                if (!__all_sync(0xffffffffu, w)) return false;
                tc_fence_after();
                const uint32_t slot = tmem + lane_base + (uint32_t)(kSfColBase + stage * kSfColsPerStage);
                tmem_st_32x32b_x1(slot + q, sf_word<KA>(comp(src.a, jj), bad));
                uint32_t wb[8];
#pragma unroll
                for (int j = 0; j < kSfbCols; ++j) wb[j] = sf_word<KB>(comp(src.b[j], jj), bad);
#pragma unroll
                for (int j = kSfbCols; j < 8; ++j) wb[j] = 0x7F7F7F7Fu;
                tmem_st_32x32b_x8(slot + 8, wb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.full[stage]));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            return true;
        };
        // walk this CTA's (tile, group) pairs, loading one group ahead
        auto advance = [&](int& t, int& grp) -> bool {
            if (++grp == groups) {
                grp = 0;
                t += gridDim.x;
            }
            return t < g.num_tiles;
        };
        int t = blockIdx.x, grp = 0;
        if (t < g.num_tiles && groups > 0) {
            SfGroup b0, b1;
            load(t, grp, b0);
            while (true) {
                int t1 = t, g1 = grp;
                const bool has1 = advance(t1, g1);
                if (has1) load(t1, g1, b1);
                if (!emit(b0, grp) || !has1) break;
                t = t1;
                grp = g1;
                int t2 = t, g2 = grp;
                const bool has2 = advance(t2, g2);
                if (has2) load(t2, g2, b0);
                if (!emit(b1, grp) || !has2) break;
                t = t2;
                grp = g2;
            }
        }
        if (__any_sync(0xffffffffu, bad != 0) && lane == 0) atomicOr(&S.bad_scale, 1);
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

// ================================================== block-scaled GEMM, CTA pair

// A pair computes a 256x224 tile with tcgen05.mma.cta_group::2 ... block_scale:
// each CTA holds 128 rows of A and 112 rows of B per 128-wide K tile, two K
// tiles per stage (60 KB, 3 stages), and 128 rows of the accumulator.  Each CTA's tensor core reads the
// scales of its own A rows and of all 224 B rows from its own TMEM, so both
// CTAs' scale writers fill their own scale slots (A row m: lane m, column m/32;
// B row n: lane 32q + n%32, column 8 + n/32, every quarter q).  The producer
// TMA-loads the scales of each pair of groups of four K tiles (32 bytes per
// row: the A rows of this CTA and all B rows of the tile) into a two-slot
// shared-memory ring, one slot ahead.  When a group lands, each writer thread reads the
// words of its rows for the group's four K tiles into registers -- E8M0 words
// as they are; power-of-two fp32 block scales (1x128, 128x128) re-encoded as
// E8M0 and repeated over the four 32-wide sub-blocks -- and frees the slot, so
// what a writer does after waiting for a TMEM slot is the same few stores for
// every scale kind.  With 224-column tiles and two accumulators TMEM has room for four
// scale slots (64 columns beside the two 224-column accumulators): K tile i
// (counted over all of a pair's tiles) uses stage i / 2 % 3 and scale slot
// i % 4.  The even CTA's `full[stage]` completes when both producers' loads
// have landed and all eight scale writers of the pair have written the slots
// of both K tiles, so the issuing thread waits once and commits once per two K
// tiles (its per-K-tile waits and commits, not the tensor core, set the pace
// with one K tile per stage).  A writer may overwrite slot i % 4 once the MMAs
// of K tile i - 4, its last reader, are done, which is completion s / 3 of
// `empty[s % 3]`, s = (i - 4) / 2; that barrier cannot run a completion
// further ahead, because the MMAs of stage s + 3 wait for the writers of K
// tiles past i.
constexpr int kBsKPerStage = 2;  // 128-wide K tiles per operand stage
constexpr int kBsPairStages = 3;
constexpr int kSfSlots = (512 - kSfColBasePair) / kSfColsPerStage;  // TMEM scale slots beside the accumulators
constexpr int kSfRing = kSfSlots / kBsKPerStage;                     // stage steps the scale slots hold
static_assert(kSfSlots % kBsKPerStage == 0 && kSfRing >= 2, "scale slots hold whole stage steps");
// The writers of stage step s wait until the MMAs of step s - kSfAhead are done: by then the slots of
// step s are free (their last reader, step s - kSfRing, is done) and `full[s % kBsPairStages]` has
// completed the phase of step s - kBsPairStages, so their arrivals count toward step s.  Running them
// further ahead than the operand ring would let an arrival land on a phase still open, one more than the
// barrier's count (undefined behaviour; on the GPU, a fault).  With the constants above kSfAhead = 2.
constexpr int kSfAhead = kSfRing < kBsPairStages ? kSfRing : kBsPairStages;
constexpr int kBsPairB = kBnPair / 2;                    // rows of B per CTA
constexpr int kBsPairABytes = kPairRows * BK;          // 16 KB per K tile
constexpr int kBsPairBBytes = kBsPairB * BK;           // B bytes per K tile and CTA
constexpr int kBsPairStageBytes = kBsKPerStage * (kBsPairABytes + kBsPairBBytes);
// Scale ring: each slot holds the scales of two groups of four K tiles (32 bytes per row), so a TMA
// box of 128 (A) or 224 (B) rows carries twice the bytes per row request; two slots.
constexpr int kScaleGroupsPerSlot = 2;
constexpr int kScaleRowBytes = 16 * kScaleGroupsPerSlot;
constexpr int kScaleSlots = 2;
constexpr int kScaleBlockRowsB = 3;                    // a tile's B rows touch at most three 128-row blocks

static_assert(kBnPair <= 2 * 128 + 1, "a tile's B rows span at most three 128-row blocks");

struct alignas(1024) SmemBsPair {
    uint8_t a[kBsPairStages][kBsKPerStage * kBsPairABytes];
    uint8_t b[kBsPairStages][kBsKPerStage * kBsPairBBytes];
    alignas(128) uint8_t sa[kScaleSlots][kPairRows * kScaleRowBytes];  // per row and group: four K tiles x 4 bytes
    alignas(128) uint8_t sb[kScaleSlots][kBnPair * kScaleRowBytes];
    alignas(1024) uint8_t out[4][kOutStageBytes];  // per epilogue warp: staged output chunks for TMA stores
    uint64_t full[kBsPairStages], empty[kBsPairStages], tfull[2], tempty[2], drain;
    uint64_t scale_full[kScaleSlots], scale_empty[kScaleSlots];
    uint32_t tmem_base;
    int abort_flag;
    int bad_scale;
};

static_assert(sizeof(SmemBsPair) + 1024 <= 232448, "the pair kernel's shared memory fits one SM (227 KB)");

// Scale-tensor TMA box of one group for an operand of kind KIND: the rows of the box and its bytes.
template <int KIND>
__host__ __device__ constexpr int scale_box_rows(int rows) {
    return KIND == SF_BLOCK ? (rows == kPairRows ? 1 : kScaleBlockRowsB) : rows;
}

// Validity of fp32 block scales, accumulated without branches: a power of two in range is, after
// 2^-127 (the only subnormal one) is mapped to the bit pattern of 2^-126, a pattern with sign and
// mantissa clear between those of 2^-126 and 2^127.
struct ScaleCheck {
    uint32_t bits = 0, lo = 0xFFFFFFFFu, hi = 0;
    __device__ __forceinline__ void add(uint32_t raw) {
        const uint32_t u = raw == 0x00400000u ? 0x00800000u : raw;
        bits |= u;
        lo = min(lo, u);
        hi = max(hi, u);
    }
    // true if some word added was not a power of two in [2^-127, 2^127]
    __device__ __forceinline__ bool any_bad() const {
        return (bits & 0x807FFFFFu) != 0 || lo < 0x00800000u || hi > 0x7F000000u;
    }
};

// E8M0 code of an fp32 block scale that is a power of two in [2^-127, 2^127]: its biased exponent (0 for
// 2^-127).  Other values give an unspecified code; they are found by the epilogue warps' check.
__device__ __forceinline__ uint32_t e8m0_code(uint32_t raw) {
    return raw == 0x00400000u ? 0u : (raw >> 23) & 0xFFu;
}

// The scale words of one operand row for the four K tiles of a scale group (word jj: four E8M0 bytes,
// one per 32-wide K sub-block of K tile jj), from the group's shared-memory slot: MX words as they
// are, fp32 block scales as their E8M0 code.  Local row r of the slot, or for 128x128 scales the
// block row of `row` counted from `block_base`; rows past the edge get the neutral scale 1.
template <int KIND>
__device__ __forceinline__ void sf_group_words(const uint8_t* slot, int half, int r, int block_base, int64_t row,
                                               int64_t rows, uint32_t (&w)[4]) {
    if (row >= rows) {
        w[0] = w[1] = w[2] = w[3] = 0x7F7F7F7Fu;
        return;
    }
    const int sr = KIND == SF_BLOCK ? (int)(row >> 7) - block_base : r;
    const uint4 v = *reinterpret_cast<const uint4*>(slot + sr * kScaleRowBytes + half * 16);
    const uint32_t raw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) w[jj] = KIND == SF_MX ? raw[jj] : e8m0_code(raw[jj]) * 0x01010101u;
}

// The epilogue warps' check of the fp32 block scales of pair tile (tm, tn), made from global memory
// (L2) while they wait for the tile's accumulator: warp q of CTA `rank` checks the A scales of its 32
// rows (1x128) or, warp 0, the CTA's one 128-row block (128x128), and the B scales of a quarter of the
// CTA's half of the tile's rows (1x128) or, CTA 0's warps 0..2, the tile's 128-row blocks (128x128),
// over all K tiles.  MX scales need no check (every E8M0 code but 255 is a scale).
template <int KA, int KB>
__device__ __forceinline__ bool tile_scales_bad(const GemmArgs& g, int tm, int tn, uint32_t rank, int q, int lane) {
    ScaleCheck chk;
    const int64_t arow0 = (int64_t)tm * kPairTile + (int64_t)rank * kPairRows;
    if constexpr (KA == SF_ROW) {
        const int64_t row = arow0 + 32 * q + lane;
        if (row < g.M) {
            const uint32_t* p = static_cast<const uint32_t*>(g.sfa) + row * g.sfa_ld;
            for (int k = 0; k < g.k_tiles; ++k) chk.add(__ldg(p + k));
        }
    } else if constexpr (KA == SF_BLOCK) {
        if (q == 0 && arow0 < g.M) {
            const uint32_t* p = static_cast<const uint32_t*>(g.sfa) + (arow0 >> 7) * g.sfa_ld;
            for (int k = lane; k < g.k_tiles; k += 32) chk.add(__ldg(p + k));
        }
    }
    if constexpr (KB == SF_ROW) {
        const int local = 32 * q + lane;  // of this CTA's kBsPairB rows
        const int64_t row = (int64_t)tn * kBnPair + (int64_t)rank * kBsPairB + local;
        if (local < kBsPairB && row < g.N) {
            const uint32_t* p = static_cast<const uint32_t*>(g.sfb) + row * g.sfb_ld;
            for (int k = 0; k < g.k_tiles; ++k) chk.add(__ldg(p + k));
        }
    } else if constexpr (KB == SF_BLOCK) {
        const int64_t b0 = ((int64_t)tn * kBnPair) >> 7, brow = b0 + q;
        const int64_t last = ((int64_t)tn * kBnPair + kBnPair - 1) >> 7;
        if (rank == 0 && q < kScaleBlockRowsB && brow <= last && (brow << 7) < g.N) {
            const uint32_t* p = static_cast<const uint32_t*>(g.sfb) + brow * g.sfb_ld;
            for (int k = lane; k < g.k_tiles; k += 32) chk.add(__ldg(p + k));
        }
    }
    return chk.any_bad();
}

template <int OUT_BF16, int KA, int KB>
__global__ void __launch_bounds__(320, 1)
    gemm_blockscaled_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                 const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                                 const __grid_constant__ CUtensorMap tmD, GemmArgs g, uint32_t idesc) {
    extern __shared__ uint8_t smem_raw[];
    SmemBsPair& S = *reinterpret_cast<SmemBsPair*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int groups = (g.k_tiles + 3) / 4;
    volatile int* abort_flag = &S.abort_flag;
    constexpr int kSaBytes = scale_box_rows<KA>(kPairRows) * kScaleRowBytes;
    constexpr int kSbBytes = scale_box_rows<KB>(kBnPair) * kScaleRowBytes;
    const int pairs = (groups + kScaleGroupsPerSlot - 1) / kScaleGroupsPerSlot;  // scale slots per tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBsPairStages; ++s) {
            mbar_init(smem_u32(&S.full[s]), 2 + 8);  // both producers + the eight scale writers of the pair
            mbar_init(smem_u32(&S.empty[s]), 1);     // the MMA commit
        }
        for (int s = 0; s < kScaleSlots; ++s) {
            mbar_init(smem_u32(&S.scale_full[s]), 1);
            mbar_init(smem_u32(&S.scale_empty[s]), 4);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(smem_u32(&S.tfull[a]), 1);
            mbar_init(smem_u32(&S.tempty[a]), 8);
        }
        mbar_init(smem_u32(&S.drain), 1);
        S.abort_flag = 0;
        S.bad_scale = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmD);
    }
    cluster_sync_all();
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&S.tmem_base), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int issued = 0;                    // scale slots issued so far (flattened over this pair's tiles)
            int nt = cid, npair = 0;           // the next (tile, pair of groups) whose scales to load
            auto issue_next_scales = [&]() -> bool {
                if (nt >= g.num_tiles || groups == 0) return true;
                const int slot = issued % kScaleSlots;
                if (issued >= kScaleSlots &&
                    !mbar_wait_bounded(smem_u32(&S.scale_empty[slot]), (uint32_t)((issued / kScaleSlots - 1) & 1),
                                       abort_flag))
                    return false;
                int tm, tn;
                tile_coords(nt, g, tm, tn);
                const int xa = (KA == SF_MX ? 16 : 4) * kScaleGroupsPerSlot * npair;
                const int xb = (KB == SF_MX ? 16 : 4) * kScaleGroupsPerSlot * npair;
                const int arow = tm * kPairTile + (int)rank * kPairRows, brow = tn * kBnPair;
                mbar_arrive_expect_tx(smem_u32(&S.scale_full[slot]), kSaBytes + kSbBytes);
                tma_load_2d(smem_u32(S.sa[slot]), &tmSA, smem_u32(&S.scale_full[slot]), xa, KA == SF_BLOCK ? arow >> 7 : arow);
                tma_load_2d(smem_u32(S.sb[slot]), &tmSB, smem_u32(&S.scale_full[slot]), xb, KB == SF_BLOCK ? brow >> 7 : brow);
                ++issued;
                if (++npair == pairs) {
                    npair = 0;
                    nt += ncl;
                }
                return true;
            };
            ok = issue_next_scales();  // one slot ahead of the slot being consumed
            for (int t = cid; ok && t < g.num_tiles; t += ncl) {
                int tm, tn;
                tile_coords(t, g, tm, tn);
                for (int kt = 0; kt < g.k_tiles; kt += kBsKPerStage) {  // k_tiles is a multiple of 4 here
                    // entering a slot's first group: load the next slot
                    if ((kt % (4 * kScaleGroupsPerSlot)) == 0 && !(ok = issue_next_scales())) break;
                    if (!mbar_wait_bounded(smem_u32(&S.empty[stage]), phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = map_to_cta(smem_u32(&S.full[stage]), 0);
#pragma unroll
                    for (int h = 0; h < kBsKPerStage; ++h) {
                        tma_load_2d_pair(smem_u32(S.a[stage] + h * kBsPairABytes), &tmA, full_leader, (kt + h) * BK,
                                         tm * kPairTile + (int)rank * kPairRows);
                        tma_load_2d_pair(smem_u32(S.b[stage] + h * kBsPairBBytes), &tmB, full_leader, (kt + h) * BK,
                                         tn * kBnPair + (int)rank * kBsPairB);
                    }
                    mbar_arrive_expect_tx_cluster(full_leader, kBsPairStageBytes);
                    if (++stage == kBsPairStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int stage = 0, acc = 0, slot = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = cid; ok && t < g.num_tiles; t += ncl) {
                if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), acc_phase ^ 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kBnPair);
                for (int kt = 0; kt < g.k_tiles; kt += kBsKPerStage) {
                    if (!mbar_wait_bounded(smem_u32(&S.full[stage]), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < kBsKPerStage; ++h) {
                        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(S.a[stage] + h * kBsPairABytes));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(S.b[stage] + h * kBsPairBBytes));
                        const uint32_t sfa_t = tmem + (uint32_t)(kSfColBasePair + slot * kSfColsPerStage);
                        const uint32_t sfb_t = sfa_t + 8;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            tc_mma_mxf8f6f4_pair(d, ad + 2 * k, bd + 2 * k,
                                                 idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4), sfa_t, sfb_t,
                                                 ((kt + h) | k) != 0 ? 1u : 0u);
                        if (++slot == kSfSlots) slot = 0;
                    }
                    tc_commit_pair_multicast(smem_u32(&S.empty[stage]), 0x3);
                    if (++stage == kBsPairStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit_pair_multicast(smem_u32(&S.tfull[acc]), 0x3);
                if (++acc == kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            tc_commit_pair(smem_u32(&S.drain));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&S.drain), 0))
                if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    } else if (warp < 6) {
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool bad = false;
        const uint32_t obuf = smem_u32(S.out[q]);
        uint32_t nchunk = 0;  // chunks this warp has staged
        for (int t = cid; t < g.num_tiles; t += ncl) {
            int tm, tn;
            tile_coords(t, g, tm, tn);
            // fp32 block scales: checked here, off the MMAs' path, while the tile accumulates
            if constexpr (KA != SF_MX || KB != SF_MX) bad |= tile_scales_bad<KA, KB>(g, tm, tn, rank, q, lane);
            bool ok = mbar_wait_bounded(smem_u32(&S.tfull[acc]), acc_phase, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int64_t row0 = (int64_t)tm * kPairTile + (int64_t)rank * kPairRows + q * 32;  // this warp's rows
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBnPair);
#pragma unroll 1
            for (int c = 0; c < kBnPair / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                const int64_t col0 = (int64_t)tn * kBnPair + c * 32;
                uint32_t unused_amax = 0;
                store_chunk_tma<OUT_BF16, false>(&tmD, obuf, nchunk, lane, r, 1.0f, 1.0f, 1.0f, unused_amax, row0, col0, g);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&S.tempty[acc]), 0));
            if (++acc == kAccBufs) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's stores are complete before the CTA exits
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&S.bad_scale, 1);
    } else {
        // Scale writers of this CTA (warp 6..9 = lane quarter q): for every K tile, the A scale of row
        // 32q + lane (column q of the K tile's slot) and the scales of all 224 B rows (columns 8 + j).
        // When a group's scales land, each thread reads the words of its rows for the group's four K
        // tiles into registers (re-encoding fp32 block scales there) and frees the ring slot; after
        // each slot wait only the TMEM stores remain, the same for every scale kind.
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int kcount = 0;  // K tiles written so far (over all of this pair's tiles)
        int consumed = 0;
        uint32_t bad = 0;
        bool ok = true;
        for (int t = cid; ok && t < g.num_tiles; t += ncl) {
            int tm, tn;
            tile_coords(t, g, tm, tn);
            const int64_t arow = (int64_t)tm * kPairTile + (int64_t)rank * kPairRows + q * 32 + lane;
            const int ablock = (tm * kPairTile + (int)rank * kPairRows) >> 7;
            const int bblock = (tn * kBnPair) >> 7;
            for (int grp = 0; ok && grp < groups; ++grp) {  // k_tiles is a multiple of 4 on this path
                const int slot = consumed % kScaleSlots, half = grp % kScaleGroupsPerSlot;
                bool w = true;
                if (half == 0) {
                    w = mbar_wait_bounded(smem_u32(&S.scale_full[slot]), (uint32_t)((consumed / kScaleSlots) & 1),
                                          abort_flag);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                }
                uint32_t wa[4], wb[kSfbColsPair][4];
                sf_group_words<KA>(S.sa[slot], half, q * 32 + lane, ablock, arow, g.M, wa);
#pragma unroll
                for (int j = 0; j < kSfbColsPair; ++j)
                    sf_group_words<KB>(S.sb[slot], half, 32 * j + lane, bblock, (int64_t)tn * kBnPair + 32 * j + lane,
                                       g.N, wb[j]);
                if (half == kScaleGroupsPerSlot - 1 || grp == groups - 1) {  // the slot's last group of this tile
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&S.scale_empty[slot]));  // the producer may refill the slot
                    ++consumed;
                }
#pragma unroll
                for (int u = 0; u < 4 / kBsKPerStage; ++u) {  // one stage (two K tiles) per arrival
                    if (kcount >= kSfAhead * kBsKPerStage) {
                        const int prev = kcount / kBsKPerStage - kSfAhead;  // its MMAs must be done
                        w = mbar_wait_bounded(smem_u32(&S.empty[prev % kBsPairStages]),
                                              (uint32_t)((prev / kBsPairStages) & 1), abort_flag);
                        if (!__all_sync(0xffffffffu, w)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const int stage = (kcount / kBsKPerStage) % kBsPairStages;
#pragma unroll
                    for (int h = 0; h < kBsKPerStage; ++h) {
                        const int jj = kBsKPerStage * u + h;
                        const uint32_t tslot =
                            tmem + lane_base + (uint32_t)(kSfColBasePair + ((kcount + h) % kSfSlots) * kSfColsPerStage);
                        tmem_st_32x32b_x1(tslot + q, wa[jj]);
                        uint32_t v8[8];
#pragma unroll
                        for (int j = 0; j < kSfbColsPair; ++j) v8[j] = wb[j][jj];
#pragma unroll
                        for (int j = kSfbColsPair; j < 8; ++j) v8[j] = 0x7F7F7F7Fu;
                        tmem_st_32x32b_x8(tslot + 8, v8);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&S.full[stage]), 0));
                    kcount += kBsKPerStage;
                }
            }
        }
        if (__any_sync(0xffffffffu, bad != 0) && lane == 0) atomicOr(&S.bad_scale, 1);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
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

// 2-D map over the output D [M x N] (row pitch ldd elements) of output kind `out` (0 fp32, 1 bf16, 2/3
// FP8) for the pair epilogues' TMA stores: box 32 x 32, rows of the box in the swizzle whose span is
// the box row (128, 64 or 32 bytes), as the epilogue stages them.
fp8_status make_out_map(CUtensorMap* map, void* ptr, int64_t M, int64_t N, int64_t ldd, int out) {
    auto fn = encode_fn();
    FP8_REQUIRE(fn != nullptr, FP8_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const int64_t es = out == 0 ? 4 : out == 1 ? 2 : 1;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(ldd * es)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = out == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw = out == 0   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : out == 1 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = fn(map, dt, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    FP8_REQUIRE(r == CUDA_SUCCESS, FP8_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
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

// Number of pair tiles: the GemmArgs among the kernel arguments.
template <typename... Rest>
int pair_tiles_of(const GemmArgs& g, const Rest&...) { return g.num_tiles; }
template <typename T, typename... Rest>
int pair_tiles_of(const T&, const Rest&... rest) { return pair_tiles_of(rest...); }

// 2-D map over a scale tensor for two groups of four K tiles per row: 32 bytes per row (eight E8M0
// words' bytes, or eight fp32), `box_rows` rows (or 128-row blocks for 128x128 scales).
template <int KIND>
fp8_status make_scale_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t ld, int tile_rows) {
    auto fn = encode_fn();
    FP8_REQUIRE(fn != nullptr, FP8_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const bool mx = KIND == SF_MX;
    const int64_t srows = KIND == SF_BLOCK ? (rows + 127) / 128 : rows;
    cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)srows};
    cuuint64_t strides[1] = {(cuuint64_t)(mx ? ld : 4 * ld)};
    cuuint32_t box[2] = {(cuuint32_t)((mx ? 16 : 4) * kScaleGroupsPerSlot), (cuuint32_t)scale_box_rows<KIND>(tile_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    FP8_REQUIRE(r == CUDA_SUCCESS, FP8_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", (int)r);
    return FP8_OK;
}

// Launch a CTA-pair kernel: clusters of 2, as many resident pairs as fit, never more pairs than tiles.
template <typename Kernel, typename... Args>
fp8_status launch_pair_kernel(Kernel k, size_t smem, int threads, cudaStream_t st, const Args&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> max_pairs;  // (kernel, device) -> resident pairs
    int dev = 0;
    cudaGetDevice(&dev);
    int mc;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair(reinterpret_cast<const void*>(k), dev);
        auto it = max_pairs.find(key);
        if (it == max_pairs.end()) {
            cfg.gridDim = dim3(2 * (device_sm_count() / 2));
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(k), &cfg) != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = device_sm_count() / 2;
            }
            it = max_pairs.emplace(key, n).first;
        }
        mc = it->second;
    }
    const int pairs = std::max(1, std::min(pair_tiles_of(args...), mc));
    cfg.gridDim = dim3(2 * pairs);
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "CTA-pair GEMM launch: %s", cudaGetErrorString(e));
    return check_launch("CTA-pair GEMM launch");
}

template <int OUT>
fp8_status launch_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g, uint32_t idesc,
                       cudaStream_t st) {
    CUtensorMap tmD;  // D is 16-byte aligned with 16-byte aligned rows (checked by the API)
    fp8_status s = make_out_map(&tmD, g.D, g.M, g.N, g.ldd, OUT);
    if (s != FP8_OK) return s;
    s = prepare_kernel(reinterpret_cast<const void*>(gemm_tensor_pair_kernel<OUT>), sizeof(SmemPair) + 1024);
    if (s != FP8_OK) return s;
    return launch_pair_kernel(gemm_tensor_pair_kernel<OUT>, sizeof(SmemPair) + 1024, 192, st, tmA, tmB, tmD, g, idesc);
}

template <int OUT>
fp8_status launch_single(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g, uint32_t idesc, int grid,
                         cudaStream_t st) {
    const size_t smem = sizeof(SmemPT) + 1024;
    fp8_status s = prepare_kernel(reinterpret_cast<const void*>(gemm_tensor_kernel<OUT>), smem);
    if (s != FP8_OK) return s;
    gemm_tensor_kernel<OUT><<<grid, 192, smem, st>>>(tmA, tmB, g, idesc);
    return check_launch("gemm_tensor_kernel launch");
}

bool is_mx(int gran) { return gran == FP8_SCALE_MX_1x32 || gran == FP8_SCALE_MX_1x32_OCP; }  // same E8M0 storage
int sf_kind(int gran) { return is_mx(gran) ? SF_MX : gran == FP8_SCALE_BLOCK_1x128 ? SF_ROW : SF_BLOCK; }

template <int OUT_BF16, int KA, int KB>
fp8_status launch_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g, uint32_t idesc, int grid,
                     cudaStream_t st) {
    if (g.pair) {
        CUtensorMap tmSA, tmSB;
        fp8_status s = make_scale_map<KA>(&tmSA, g.sfa, g.M, g.sfa_ld, kPairRows);
        if (s != FP8_OK) return s;
        s = make_scale_map<KB>(&tmSB, g.sfb, g.N, g.sfb_ld, kBnPair);
        if (s != FP8_OK) return s;
        CUtensorMap tmD;  // D is 16-byte aligned with 16-byte aligned rows (checked by the API)
        s = make_out_map(&tmD, g.D, g.M, g.N, g.ldd, OUT_BF16);
        if (s != FP8_OK) return s;
        auto kp = gemm_blockscaled_pair_kernel<OUT_BF16, KA, KB>;
        const size_t smem_p = sizeof(SmemBsPair) + 1024;
        s = prepare_kernel(reinterpret_cast<const void*>(kp), smem_p);
        if (s != FP8_OK) return s;
        return launch_pair_kernel(kp, smem_p, 320, st, tmA, tmB, tmSA, tmSB, tmD, g, idesc);
    }
    const size_t smem = sizeof(SmemBS) + 1024;
    auto k = gemm_blockscaled_kernel<OUT_BF16, KA, KB>;
    fp8_status s = prepare_kernel(reinterpret_cast<const void*>(k), smem);
    if (s != FP8_OK) return s;
    k<<<grid, 320, smem, st>>>(tmA, tmB, g, idesc);
    return check_launch("gemm_blockscaled_kernel launch");
}

template <int OUT_BF16>
fp8_status dispatch_bs(int ka, int kb, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                       uint32_t idesc, int grid, cudaStream_t st) {
#define FP8Q_BS(A, B) \
    if (ka == A && kb == B) return launch_bs<OUT_BF16, A, B>(tmA, tmB, g, idesc, grid, st);
    FP8Q_BS(SF_MX, SF_MX)
    FP8Q_BS(SF_ROW, SF_BLOCK)
    FP8Q_BS(SF_ROW, SF_ROW)
    FP8Q_BS(SF_BLOCK, SF_BLOCK)
    FP8Q_BS(SF_BLOCK, SF_ROW)
    FP8Q_BS(SF_MX, SF_ROW)
    FP8Q_BS(SF_MX, SF_BLOCK)
    FP8Q_BS(SF_ROW, SF_MX)
    FP8Q_BS(SF_BLOCK, SF_MX)
#undef FP8Q_BS
    return FP8_ERR_UNSUPPORTED;
}

}  // namespace

// out: 0 fp32, 1 bf16, 2 E4M3, 3 E5M2 (the FP8 outputs take the per-tensor path only, with sd / amax_d).
fp8_status launch_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int fa, int ga, const void* sfa,
                       const uint8_t* B, int64_t ldb, int fb, int gb, const void* sfb, void* D, int out,
                       int64_t ldd, const float* sd, float* amax_d, int32_t* status, cudaStream_t st) {
    const int out_bf16 = out == 1;
    const bool blockscaled = ga != FP8_SCALE_TENSOR;
    // two-SM tiles once the second half of a 256-row tile has work; block-scaled pairs TMA-load 16-byte
    // scale rows, which needs K % 512 == 0 and 16-byte aligned scale tensors
    const bool pair = M > BM && (!blockscaled || (K % 512 == 0 && (reinterpret_cast<uintptr_t>(sfa) & 15) == 0 &&
                                                  (reinterpret_cast<uintptr_t>(sfb) & 15) == 0));
    const int bn = blockscaled ? (pair ? kBnPair : BN_BS) : BN;
    GemmArgs g;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    const int bm = pair ? kPairTile : BM;
    g.tiles_m = (int)((M + bm - 1) / bm);
    g.tiles_n = (int)((N + bn - 1) / bn);
    g.k_tiles = (int)((K + BK - 1) / BK);
    g.num_tiles = g.tiles_m * g.tiles_n;
    g.D = D;
    g.ldd = ldd;
    g.status = status;
    g.sa = g.sb = nullptr;
    g.sfa = g.sfb = nullptr;
    g.sfa_ld = g.sfb_ld = 0;
    g.vec_a = g.vec_b = 0;
    g.sd = sd;
    g.amax_d = amax_d;

    CUtensorMap tmA, tmB;
    fp8_status s = make_operand_map(&tmA, A, M, K, lda, BM);
    if (s != FP8_OK) return s;
    s = make_operand_map(&tmB, B, N, K, ldb, pair ? bn / 2 : bn);
    if (s != FP8_OK) return s;
    g.pair = pair;
    if (pair && !blockscaled) {
        g.sa = static_cast<const float*>(sfa);
        g.sb = static_cast<const float*>(sfb);
        const uint32_t idesc = idesc_f8f6f4(fa, fb, kPairTile, BN);
        switch (out) {
            case 0: return launch_pair<0>(tmA, tmB, g, idesc, st);
            case 1: return launch_pair<1>(tmA, tmB, g, idesc, st);
            case 2: return launch_pair<2>(tmA, tmB, g, idesc, st);
            default: return launch_pair<3>(tmA, tmB, g, idesc, st);
        }
    }

    const int grid = std::min(g.num_tiles, device_sm_count());
    if (!blockscaled) {
        g.sa = static_cast<const float*>(sfa);
        g.sb = static_cast<const float*>(sfb);
        const uint32_t idesc = idesc_f8f6f4(fa, fb, BM, BN);
        switch (out) {
            case 0: return launch_single<0>(tmA, tmB, g, idesc, grid, st);
            case 1: return launch_single<1>(tmA, tmB, g, idesc, grid, st);
            case 2: return launch_single<2>(tmA, tmB, g, idesc, grid, st);
            default: return launch_single<3>(tmA, tmB, g, idesc, grid, st);
        }
    }
    g.sfa = sfa;
    g.sfb = sfb;
    const int64_t KT = (K + BK - 1) / BK;
    // row pitch of each scale tensor: E8M0 rows are K/32 bytes, fp32 rows are ceil(K/128) floats
    g.sfa_ld = is_mx(ga) ? K / 32 : KT;
    g.sfb_ld = is_mx(gb) ? K / 32 : KT;
    auto vec_ok = [](const void* p, int gran, int64_t ld) {
        const int64_t row_bytes = is_mx(gran) ? ld : 4 * ld;
        return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && row_bytes % 16 == 0;
    };
    g.vec_a = vec_ok(sfa, ga, g.sfa_ld);
    g.vec_b = vec_ok(sfb, gb, g.sfb_ld);
    const uint32_t idesc = idesc_mxf8f6f4(fa, fb, pair ? kPairTile : BM, pair ? kBnPair : BN_BS, 0, 0);
    return out_bf16 ? dispatch_bs<1>(sf_kind(ga), sf_kind(gb), tmA, tmB, g, idesc, grid, st)
                    : dispatch_bs<0>(sf_kind(ga), sf_kind(gb), tmA, tmB, g, idesc, grid, st);
}

}  // namespace fp8q
