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
// All of it is HBM-bound.  The cast kernel streams 128x128 bf16 tiles through
// a two-deep TMA ring per CTA, three CTAs per SM (each CTA works on one tile
// while the next one loads), computes block maxima in registers (warp
// shuffles), writes the row-wise codes, and reads the same tile down its
// columns for the transposed column-wise codes, so one HBM read feeds both
// outputs.  The column-wise codes of a tile are staged (128B-swizzled) in the
// tile's own shared-memory stage once every warp has read it, and leave as one
// TMA store of whole 128-byte lines; the stage is refilled after that store has
// read it.  The fused amax is reduced per warp, per CTA, then one atomic per
// CTA.  Current scaling runs the amax pass and the cast in one cooperative
// launch with a grid barrier between them.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace fp8q {

namespace {

constexpr int kTile = 128;     // tile is kTile x kTile bf16 elements (32 KB)
constexpr int kThreads = 256;
constexpr int kQStages = 2;    // TMA ring depth (3 CTAs per SM)
constexpr uint32_t kHalfBytes = kTile * 64 * 2;  // a tile is loaded as two 64-column halves (16 KB each)

struct QuantArgs {
    int64_t rows, cols;
    int margin;
    const float* scale;
    uint8_t* q_row;
    uint8_t* q_col;
    void* sf_row;
    void* sf_col;
    float* amax;
    int64_t tiles_c, ntiles;
    int do_row, do_col;
    int32_t* status;
};

// Tensor maps of a cast launch: the bf16 input x and the column-wise output (u8 [cols x rows]; unused
// without one).
struct QuantMaps {
    CUtensorMap x;
    CUtensorMap qc;
};

struct alignas(1024) QuantSmem {
    uint16_t tile[kQStages][kTile * kTile];
    uint64_t full[kQStages];
    uint64_t empty[kQStages];  // one arrival per warp when it is done with the stage
    uint32_t red[2][8];
    uint32_t col_part[4][64];
    uint32_t col_sf[2][128];  // MX column scales of a tile: four 32-row segments (bytes) per column
    uint32_t am[8];
    int abort_flag;
};

__device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Bias of a block from the bf16 bit pattern m of its amax (|x| bits): for a
// normal finite m the exponent and the top mantissa bits are read directly
// (m > 1.75 <=> the 7 fraction bits exceed 0x60); other m take the general path.
__device__ __forceinline__ int bias_bf16(uint32_t m, int fmt, int margin) {
    if (m - 0x80u < 0x7F00u) {
        // floor(log2(fmax / amax)) with fmax = 1.75 * 2^ef and amax = (1 + f) 2^(E - 127): ef + 127 - E, one
        // less when f > 0.75 (a mantissa above 0x60), and adding 0x1F to the bits carries into the
        // exponent field exactly then
        const int ef = fmt == FP8_E4M3 ? 8 : 15;
        const int e = ef + 127 - margin - (int)((m + 0x1Fu) >> 7);
        return min(max(e, -126), 127);
    }
    bool nf = false;
    return bias_from_amax(bf16bits_to_float(m), fmt, margin, &nf);
}

// The OCP MX alternative for 1x32 blocks: e = emax - floor(log2(amax)) - margin, no mantissa term.
__device__ __forceinline__ int bias_bf16_ocp(uint32_t m, int fmt, int margin) {
    if (m - 0x80u < 0x7F00u) {
        const int ef = fmt == FP8_E4M3 ? 8 : 15;
        const int e = ef + 127 - (int)(m >> 7) - margin;
        return min(max(e, -126), 127);
    }
    bool nf = false;
    return bias_from_amax_ocp(bf16bits_to_float(m), fmt, margin, &nf);
}

// Block bias of granularity GRAN.
template <int GRAN>
__device__ __forceinline__ int block_bias(uint32_t m, int fmt, int margin) {
    if constexpr (GRAN == FP8_SCALE_MX_1x32_OCP)
        return bias_bf16_ocp(m, fmt, margin);
    else
        return bias_bf16(m, fmt, margin);
}

// Running |x| maximum of bf16 pairs: one instruction per word.  max.xorsign.abs
// keeps the larger magnitude (its sign bit is meaningless and masked off at the
// end); .NaN makes a NaN win, so a NaN input yields a NaN amax.
__device__ __forceinline__ uint32_t absmax_acc(uint32_t acc, uint32_t w) {
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t absmax_fold(uint32_t acc) { return fold2(acc & 0x7FFF7FFFu); }

// 2^e as a bf16x2 pair, e in [-126, 127].
__device__ __forceinline__ uint32_t pow2_bf16x2(int e) {
    const uint32_t b = (uint32_t)(e + 127) << 7;
    return b | (b << 16);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Scaled cast of the two bf16 in word w: x * 2^e is exact in bf16 whenever it
// is a normal number, and when it is not its magnitude is below 2^-126 and
// encodes to a signed zero either way, so the codes equal those of the fp32
// product.  Low byte = low element.
template <int FMT>
__device__ __forceinline__ uint32_t encode2(uint32_t w, uint32_t s2) {
    const uint32_t p = mul_bf16x2(w, s2);
    return cvt_fp8x2<FMT>(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
}

template <int FMT>
__device__ __forceinline__ uint2 encode8(const uint4& v, uint32_t s2) {
    return make_uint2(encode2<FMT>(v.x, s2) | (encode2<FMT>(v.y, s2) << 16),
                      encode2<FMT>(v.z, s2) | (encode2<FMT>(v.w, s2) << 16));
}

// Same with an arbitrary fp32 scale (per-tensor scales that are not powers of two).
template <int FMT>
__device__ __forceinline__ uint32_t encode2_f32(uint32_t w, float s) {
    return cvt_fp8x2<FMT>(__fmul_rn(bf16_lo(w), s), __fmul_rn(bf16_hi(w), s));
}
template <int FMT>
__device__ __forceinline__ uint2 encode8_f32(const uint4& v, float s) {
    return make_uint2(encode2_f32<FMT>(v.x, s) | (encode2_f32<FMT>(v.y, s) << 16),
                      encode2_f32<FMT>(v.z, s) | (encode2_f32<FMT>(v.w, s) << 16));
}

// Both columns of a word column at once: w[r] holds rows r of columns A (low) and B (high); s2
// holds the bf16 scales of A (low) and B (high).  One bf16x2 multiply per row scales both
// columns, then each column's rows 2p, 2p+1 are converted together.
template <int FMT>
__device__ __forceinline__ void encode_column_pair32(const uint32_t (&w)[32], uint32_t s2, uint32_t (&oA)[8],
                                                     uint32_t (&oB)[8]) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const uint32_t a = mul_bf16x2(w[2 * p], s2), b = mul_bf16x2(w[2 * p + 1], s2);
        const uint32_t cA = cvt_fp8x2<FMT>(__uint_as_float(a << 16), __uint_as_float(b << 16));
        const uint32_t cB = cvt_fp8x2<FMT>(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u));
        if (p & 1) {
            oA[p >> 1] |= cA << 16;
            oB[p >> 1] |= cB << 16;
        } else {
            oA[p >> 1] = cA;
            oB[p >> 1] = cB;
        }
    }
}

// Column-wise with an arbitrary fp32 scale: the low (HALF = 0) or high (HALF = 1) bf16 of 32 words
// (32 rows of one column) -> 32 codes in 8 words, row order.
template <int FMT, int HALF>
__device__ __forceinline__ void encode_column32_f32(const uint32_t (&w)[32], float s, uint32_t (&o)[8]) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const uint32_t pair = HALF ? __byte_perm(w[2 * p], w[2 * p + 1], 0x7632) : __byte_perm(w[2 * p], w[2 * p + 1], 0x5410);
        const uint32_t c = encode2_f32<FMT>(pair, s);
        if (p & 1) o[p >> 1] |= c << 16; else o[p >> 1] = c;
    }
}

// The 32 codes of column c (0..127 in the tile), rows 32 seg .. 32 seg + 31, into the staged
// column-wise tile: 128 bytes per column, 16-byte chunks in the 128B swizzle of the TMA store
// (chunk k of line c sits at chunk k ^ (c % 8); the stage is 1024-byte aligned).
__device__ __forceinline__ void stage_col32(uint32_t base, int c, int seg, const uint32_t (&o)[8]) {
    const uint32_t line = base + (uint32_t)c * kTile;
    st_shared_v4(line + ((uint32_t)((2 * seg) ^ (c & 7)) << 4), o[0], o[1], o[2], o[3]);
    st_shared_v4(line + ((uint32_t)((2 * seg + 1) ^ (c & 7)) << 4), o[4], o[5], o[6], o[7]);
}

// Persistent CTAs walk 128x128 tiles (grid-stride).  Thread 0 keeps the next
// tile's TMA load in flight; each warp releases a stage on its own (an mbarrier
// arrival).  Row-wise only, warps never wait for one another except where a
// tile needs a cross-warp reduction (128x128 blocks); with the column-wise copy
// the CTA works in lock step (the codes are staged in the stage all warps read).
// A tile arrives as two 64-column halves (two TMA loads), each 128 rows of 128
// bytes in the 128-byte swizzle: 16-byte chunk k of row r is stored at chunk
// k ^ (r % 8).  Row pass: each thread casts 16 columns of four rows 32 apart
// (the mapping is spelled out below); a warp instruction covers four whole
// rows.  Column pass: warp w covers column pairs lane + 32 (w & 1) over the
// 32-row segment w / 2.  Both passes' shared-memory reads are free of bank
// conflicts.
// The tile loop (shared by the cast kernel and the fused current-scaling kernel).  For
// per-tensor scaling `s_given` is the scale; block granularities compute their own.  With
// `from_end` (the fused kernel, whose amax pass has just read x front to back) the CTAs walk the
// tiles from the last one back, so that the tiles read last, the likeliest to be still in L2, come
// first, and the codes are stored with an L2 evict-first policy, so that they do not push the rest
// of x out of L2 before it is read again (measured: 92.2 -> 88.1 us at 16384x5120 row+col).  The
// plain casts store without the hint: their codes are the next GEMM's operands (measured: the hint
// made the benchmark step's casts 1 % slower).
template <int GRAN, int FMT>
__device__ __forceinline__ void quantize_tiles(const QuantMaps* maps, const QuantArgs& a, float s_given, int cta,
                                               int ctas, bool from_end = false) {
    const CUtensorMap* tmX = &maps->x;
    extern __shared__ uint8_t smem_raw[];
    QuantSmem& S = *reinterpret_cast<QuantSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Row pass: in visit v (0..3) the thread casts 16 columns (two 16-byte chunks) of tile row
    // 32 v + rl: half h = bit 3 of the lane, chunk pair cp = lane % 4 of that half, rl = 4 warp +
    // 2 (lane / 16) + (lane / 4) % 2.  A warp instruction covers 4 whole rows (128 bytes each: full
    // lines for the row-wise stores); the 8 lanes of a quarter warp read one half of two adjacent rows,
    // whose swizzled chunks fall in 8 different bank groups.  A 1x32 block is two neighbouring lanes
    // (lane ^ 1), a 1x128 row block the 8 lanes that differ in bits 0, 1 and 3.
    const int rh = (lane >> 3) & 1, rcp = lane & 3;
    const int rl = 4 * warp + 2 * (lane >> 4) + ((lane >> 2) & 1);
    uint32_t row_off[2];  // byte offsets of the thread's two chunks within row rl of its half
#pragma unroll
    for (int c = 0; c < 2; ++c)
        row_off[c] = (uint32_t)rh * kHalfBytes + (uint32_t)rl * 128u + ((uint32_t)((2 * rcp + c) ^ (rl & 7)) << 4);
    const int64_t n_my = (a.ntiles - cta + ctas - 1) / ctas;

    // tiles that need a block-wide reduction, and the staged column-wise copy, keep the CTA in lock step
    constexpr bool kMX = GRAN == FP8_SCALE_MX_1x32 || GRAN == FP8_SCALE_MX_1x32_OCP;
    const bool lockstep = GRAN == FP8_SCALE_BLOCK_128x128 || a.do_col;
    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), kThreads / 32);
        }
        S.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // x is read once.  Per-tensor casts mark its lines evict-first in L2, which leaves L2 to the
    // outputs (measured: row+col per-tensor cast 6 % faster); the block granularities measured
    // slower with the hint and load without it.
    const uint64_t policy = GRAN == FP8_SCALE_TENSOR && tid == 0 ? l2_policy_evict_first() : 0;
    const uint64_t out_policy = from_end ? l2_policy_evict_first() : 0;
    // Tile coordinates (tile row, tile column) advance by the grid size each step, with a carry: one
    // division per CTA instead of a 64-bit division per tile in every thread.
    const int tiles_c = (int)a.tiles_c;
    const int step_r = (int)(ctas / a.tiles_c), step_c = (int)(ctas % a.tiles_c);
    const int64_t first = from_end ? a.ntiles - 1 - cta : cta;
    auto advance = [&](int& tr, int& tc) {
        if (from_end) {
            tr -= step_r;
            tc -= step_c;
            if (tc < 0) {
                tc += tiles_c;
                --tr;
            }
        } else {
            tr += step_r;
            tc += step_c;
            if (tc >= tiles_c) {
                tc -= tiles_c;
                ++tr;
            }
        }
    };
    int ld_tr = (int)(first / a.tiles_c), ld_tc = (int)(first % a.tiles_c);  // next tile to load (thread 0)
    auto issue = [&](int64_t i) {  // TMA load of this CTA's i-th tile (the next one in order) into stage i % kQStages
        const int st = (int)(i % kQStages);
        const int x0 = ld_tc * kTile, y0 = ld_tr * kTile;
        advance(ld_tr, ld_tc);
        mbar_arrive_expect_tx(smem_u32(&S.full[st]), kTile * kTile * 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two 64-column halves, 128-byte rows in the 128B swizzle
            if constexpr (GRAN == FP8_SCALE_TENSOR)
                tma_load_2d_hint(smem_u32(S.tile[st]) + h * kHalfBytes, tmX, smem_u32(&S.full[st]), x0 + 64 * h, y0,
                                 policy);
            else
                tma_load_2d(smem_u32(S.tile[st]) + h * kHalfBytes, tmX, smem_u32(&S.full[st]), x0 + 64 * h, y0);
        }
    };
    int64_t issued = 0;  // meaningful in thread 0
    if (tid == 0) {
        tma_prefetch_desc(tmX);
        for (; issued < kQStages && issued < n_my; ++issued) issue(issued);
    }

    uint32_t s2_tensor = 0;
    float s_tensor = 1.0f;
    bool pow2_tensor = true;
    if constexpr (GRAN == FP8_SCALE_TENSOR) {
        // a positive normal power of two 2^e is exact as a bf16x2 pair; any other scale takes the fp32 path
        s_tensor = s_given;
        const uint32_t u = __float_as_uint(s_tensor);
        pow2_tensor = (u & 0x807FFFFFu) == 0 && (u >> 23) - 1u < 254u;
        const uint32_t sb = u >> 16;
        s2_tensor = sb | (sb << 16);
    }
    uint32_t amax_acc = 0;
    int cur_tr = (int)(first / a.tiles_c), cur_tc = (int)(first % a.tiles_c);  // tile being cast
    const int64_t sf32_ld = cdiv(a.cols, 32), sf128_ld = a.tiles_c;  // row pitch of 1x32 / 1x128 row scales
    // every row's 16-column chunks are 16-byte aligned when the rows are (q_row is 8-byte aligned)
    const bool rows16 = a.do_row && (a.cols % 16 == 0) && ((reinterpret_cast<uintptr_t>(a.q_row) & 15) == 0);

    for (int64_t i = 0; i < n_my; ++i, advance(cur_tr, cur_tc)) {
        if (tid == 0 && i >= 1 && i + 1 < n_my) {
            // stage (i+1) % 2 held tile i-1: wait until every warp has released it and the TMA store
            // of its column-wise codes has read it, then refill
            const int64_t u = i - 1;
            if (mbar_wait_bounded(smem_u32(&S.empty[u % kQStages]), (uint32_t)((u / kQStages) & 1), &S.abort_flag)) {
                if (a.do_col) bulk_wait_read_all();
                issue(i + 1);
                issued = i + 2;
            }
        }
        const int st = (int)(i % kQStages);
        bool ok = mbar_wait_bounded(smem_u32(&S.full[st]), (uint32_t)((i / kQStages) & 1), &S.abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (lockstep) {
            if (__syncthreads_or(!ok)) break;
        } else if (!ok) {
            break;
        }
        const uint32_t Tb = smem_u32(S.tile[st]);
        const int64_t r0 = (int64_t)cur_tr * kTile, c0 = (int64_t)cur_tc * kTile;
        const int parity = (int)(i & 1);

        // row pass, loads: visit v reads row 32 v + rl (rows 32 apart keep the swizzle phase: rl % 8)
        uint4 v[4][2];
#pragma unroll
        for (int vi = 0; vi < 4; ++vi)
#pragma unroll
            for (int c = 0; c < 2; ++c) v[vi][c] = ld_shared_v4(Tb + (uint32_t)(32 * vi) * 128u + row_off[c]);
        uint32_t pm[4] = {0, 0, 0, 0};  // |x| max of the thread's 16 columns in each visit, bf16 bits
        if (GRAN != FP8_SCALE_TENSOR || a.amax != nullptr) {
#pragma unroll
            for (int vi = 0; vi < 4; ++vi) {
                const uint4 x0 = v[vi][0], x1 = v[vi][1];
                pm[vi] = absmax_fold(absmax_acc(absmax_acc(absmax_acc(x0.x, x0.y), absmax_acc(x0.z, x0.w)),
                                                absmax_acc(absmax_acc(x1.x, x1.y), absmax_acc(x1.z, x1.w))));
                amax_acc = max(amax_acc, pm[vi]);
            }
        }

        int e_tile = 0;
        if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
            uint32_t m = __reduce_max_sync(0xffffffffu, max(max(pm[0], pm[1]), max(pm[2], pm[3])));
            if (lane == 0) S.red[parity][warp] = m;
            __syncthreads();
            m = S.red[parity][0];
#pragma unroll
            for (int w = 1; w < 8; ++w) m = max(m, S.red[parity][w]);
            e_tile = bias_bf16(m, FMT, a.margin);
            if (tid == 0) {
                const int64_t tr = r0 / kTile, tc = c0 / kTile;
                if (a.do_row) static_cast<float*>(a.sf_row)[tr * cdiv(a.cols, kTile) + tc] = pow2_exact(-e_tile);
                if (a.do_col) static_cast<float*>(a.sf_col)[tc * cdiv(a.rows, kTile) + tr] = pow2_exact(-e_tile);
            }
        }

        // ---------------------------------------------------------- row-wise
        if (a.do_row) {
            const int64_t cc = c0 + 64 * rh + 16 * rcp;  // the thread's first column
            const int64_t r_first = r0 + rl;
            uint8_t* dst_row = a.q_row + r_first * a.cols + cc;  // advances 32 rows per visit
            // MX: the E8M0 byte of the thread's 32-column block (lanes with even rcp store it)
            uint8_t* sf_mx = kMX ? static_cast<uint8_t*>(a.sf_row) + r_first * sf32_ld + (cc >> 5) : nullptr;
#pragma unroll
            for (int vi = 0; vi < 4; ++vi, dst_row += 32 * a.cols, sf_mx += kMX ? 32 * sf32_ld : 0) {
                const int64_t r = r_first + 32 * vi;
                const bool row_ok = r < a.rows;
                uint32_t s2;
                if constexpr (GRAN == FP8_SCALE_TENSOR) {
                    s2 = s2_tensor;
                } else if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
                    s2 = pow2_bf16x2(e_tile);
                } else if constexpr (kMX) {
                    const uint32_t m = max(pm[vi], __shfl_xor_sync(0xffffffffu, pm[vi], 1));
                    const int e = block_bias<GRAN>(m, FMT, a.margin);
                    s2 = pow2_bf16x2(e);
                    if ((rcp & 1) == 0 && row_ok && cc < a.cols) *sf_mx = (uint8_t)(127 - e);
                } else {  // 1x128
                    uint32_t m = max(pm[vi], __shfl_xor_sync(0xffffffffu, pm[vi], 1));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    const int e = bias_bf16(m, FMT, a.margin);
                    s2 = pow2_bf16x2(e);
                    if (rh == 0 && rcp == 0 && row_ok)
                        static_cast<float*>(a.sf_row)[r * sf128_ld + cur_tc] = pow2_exact(-e);
                }
                if (row_ok) {
                    uint2 q0, q1;
                    if (GRAN != FP8_SCALE_TENSOR || pow2_tensor) {
                        q0 = encode8<FMT>(v[vi][0], s2);
                        q1 = encode8<FMT>(v[vi][1], s2);
                    } else {
                        q0 = encode8_f32<FMT>(v[vi][0], s_tensor);
                        q1 = encode8_f32<FMT>(v[vi][1], s_tensor);
                    }
                    uint8_t* dst = dst_row;
                    if (cc + 16 <= a.cols && rows16) {
                        if (from_end)
                            st_global_v4_hint(dst, q0.x, q0.y, q1.x, q1.y, out_policy);
                        else
                            *reinterpret_cast<uint4*>(dst) = make_uint4(q0.x, q0.y, q1.x, q1.y);
                    } else {
                        if (cc < a.cols) *reinterpret_cast<uint2*>(dst) = q0;
                        if (cc + 8 < a.cols) *reinterpret_cast<uint2*>(dst + 8) = q1;
                    }
                }
            }
        }

        // ------------------------------------------------------- column-wise
        if (a.do_col) {
            const int cp = lane + 32 * (warp & 1);  // column pair within the tile
            const int seg = warp >> 1;              // 32-row segment within the tile
            // word (rows 32 seg + rr, columns 2 cp, 2 cp + 1): half cp / 32, 16-byte chunk (cp % 32) / 4 of the
            // row's 128 bytes, stored at chunk ((cp % 32) / 4) ^ (row % 8); row % 8 = rr % 8
            const uint32_t cbase = Tb + (uint32_t)(warp & 1) * kHalfBytes + (uint32_t)(32 * seg) * 128u + 4u * (lane & 3);
            uint32_t w[32];
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
                w[rr] = ld_shared_u32(cbase + (uint32_t)rr * 128u + ((uint32_t)((lane >> 2) ^ (rr & 7)) << 4));
            uint32_t mm = w[0];
#pragma unroll
            for (int r = 1; r < 32; ++r) mm = absmax_acc(mm, w[r]);
            mm &= 0x7FFF7FFFu;

            uint32_t sA, sB;
            const int64_t ca = c0 + 2 * cp, cb = ca + 1;
            if constexpr (GRAN == FP8_SCALE_TENSOR) {
                sA = sB = s2_tensor;
            } else if constexpr (GRAN == FP8_SCALE_BLOCK_128x128) {
                sA = sB = pow2_bf16x2(e_tile);
            } else if constexpr (kMX) {
                const int eA = block_bias<GRAN>(mm & 0xFFFFu, FMT, a.margin);
                const int eB = block_bias<GRAN>(mm >> 16, FMT, a.margin);
                sA = pow2_bf16x2(eA);
                sB = pow2_bf16x2(eB);
                uint8_t* cs = reinterpret_cast<uint8_t*>(S.col_sf[parity]);
                cs[4 * (2 * cp) + seg] = (uint8_t)(127 - eA);
                cs[4 * (2 * cp + 1) + seg] = (uint8_t)(127 - eB);
                __syncthreads();
                if (tid < kTile) {  // column c0 + tid: its four segment scales, rows r0 .. r0 + 127
                    const int64_t c = c0 + tid;
                    const int64_t nb = cdiv(a.rows, 32);
                    uint8_t* sf = static_cast<uint8_t*>(a.sf_col) + c * nb + (r0 >> 5);
                    const uint32_t word = S.col_sf[parity][tid];
                    if (c < a.cols) {
                        if (r0 + kTile <= a.rows && ((reinterpret_cast<uintptr_t>(sf) & 3) == 0)) {
                            *reinterpret_cast<uint32_t*>(sf) = word;
                        } else {
                            for (int q = 0; q < 4 && r0 + 32 * q < a.rows; ++q) sf[q] = (uint8_t)(word >> (8 * q));
                        }
                    }
                }
            } else {  // 1x128 -> 128x1 column blocks: combine the four 32-row segments
                S.col_part[seg][cp] = mm;
                __syncthreads();
                const uint32_t m4 = __vmaxu2(__vmaxu2(S.col_part[0][cp], S.col_part[1][cp]),
                                             __vmaxu2(S.col_part[2][cp], S.col_part[3][cp]));
                const int eA = bias_bf16(m4 & 0xFFFFu, FMT, a.margin);
                const int eB = bias_bf16(m4 >> 16, FMT, a.margin);
                sA = pow2_bf16x2(eA);
                sB = pow2_bf16x2(eB);
                if (seg == 0) {
                    float* sf = static_cast<float*>(a.sf_col);
                    const int64_t nb = cdiv(a.rows, kTile);
                    if (ca < a.cols) sf[ca * nb + r0 / kTile] = pow2_exact(-eA);
                    if (cb < a.cols) sf[cb * nb + r0 / kTile] = pow2_exact(-eB);
                }
            }
            uint32_t o[8], oB[8];
            if (GRAN == FP8_SCALE_TENSOR && !pow2_tensor) {
                encode_column32_f32<FMT, 0>(w, s_tensor, o);
                encode_column32_f32<FMT, 1>(w, s_tensor, oB);
            } else {
                encode_column_pair32<FMT>(w, (sA & 0xFFFFu) | (sB & 0xFFFF0000u), o, oB);
            }
            // every warp has read the tile (row pass and column loads; the block granularities' barrier
            // above already says so): the codes go into its stage and leave as one TMA store, which clips
            // the rows and columns past the tensor's edge
            if constexpr (!(kMX || GRAN == FP8_SCALE_BLOCK_1x128)) __syncthreads();
            stage_col32(Tb, 2 * cp, seg, o);
            stage_col32(Tb, 2 * cp + 1, seg, oB);
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                if (from_end)
                    tma_store_2d_hint(&maps->qc, Tb, (int)r0, (int)c0, out_policy);
                else
                    tma_store_2d(&maps->qc, Tb, (int)r0, (int)c0);
                bulk_commit();
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.empty[st]));  // this warp is done with the stage
    }
    if (tid == 0 && a.do_col) bulk_wait_all();  // the column-wise stores complete before the CTA exits

    __syncthreads();
    if (S.abort_flag) {
        // giving up: let the loads already issued land before the CTA exits
        if (tid == 0) {
            for (int64_t i = issued > kQStages ? issued - kQStages : 0; i < issued; ++i) {
                const int st = (int)(i % kQStages);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_u32(&S.full[st]), (uint32_t)((i / kQStages) & 1)))
                    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
            }
            if (a.status) atomicOr(a.status, FP8_STATUS_TIMEOUT);
        }
        return;
    }
    if (a.amax) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, amax_acc);
        if (lane == 0) S.am[warp] = m;
        __syncthreads();
        if (tid == 0) {
            uint32_t mx = S.am[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) mx = max(mx, S.am[w]);
            atomicMax(reinterpret_cast<unsigned int*>(a.amax), mx << 16);
        }
    }
}

template <int GRAN>
__device__ __forceinline__ float tensor_scale(const QuantArgs& a) {
    if constexpr (GRAN == FP8_SCALE_TENSOR)
        return *a.scale;
    else
        return 1.0f;
}

template <int GRAN, int FMT>
__global__ void __launch_bounds__(kThreads, 3) quantize_tile_kernel(const __grid_constant__ QuantMaps maps, QuantArgs a) {
    quantize_tiles<GRAN, FMT>(&maps, a, tensor_scale<GRAN>(a), blockIdx.x, gridDim.x);
}

// ----------------------------------------------------------- batched casts
//
// Several casts in one launch (fp8_quantize_batch): the grid is split among the tensors in
// proportion to their tiles, and each CTA runs the tile loop of one tensor with its own granularity
// and format, as a CTA of that tensor's own launch would, over its share of the grid.  The batch
// pays one launch, one fill and one tail instead of one per tensor.
constexpr int kMaxBatch = FP8_QUANTIZE_BATCH_MAX;

struct QuantBatch {
    QuantMaps maps[kMaxBatch];
    QuantArgs a[kMaxBatch];
    int cta0[kMaxBatch + 1];  // tensor k's CTAs are cta0[k] .. cta0[k + 1] - 1
    int kind[kMaxBatch];      // granularity * 2 + format
    int n;
};

__global__ void __launch_bounds__(kThreads, 3) quantize_batch_kernel(const __grid_constant__ QuantBatch b) {
    int k = 0;
    while (k + 1 < b.n && (int)blockIdx.x >= b.cta0[k + 1]) ++k;
    const int cta = (int)blockIdx.x - b.cta0[k], ctas = b.cta0[k + 1] - b.cta0[k];
    const QuantMaps* m = &b.maps[k];
    const QuantArgs& a = b.a[k];
    switch (b.kind[k]) {
#define FP8Q_BATCH_CASE(G)                                                                    \
    case 2 * (G) + FP8_E4M3:                                                                  \
        quantize_tiles<G, FP8_E4M3>(m, a, tensor_scale<G>(a), cta, ctas);                    \
        break;                                                                                \
    case 2 * (G) + FP8_E5M2:                                                                  \
        quantize_tiles<G, FP8_E5M2>(m, a, tensor_scale<G>(a), cta, ctas);                    \
        break;
        FP8Q_BATCH_CASE(FP8_SCALE_TENSOR)
        FP8Q_BATCH_CASE(FP8_SCALE_BLOCK_1x128)
        FP8Q_BATCH_CASE(FP8_SCALE_BLOCK_128x128)
        FP8Q_BATCH_CASE(FP8_SCALE_MX_1x32)
        FP8Q_BATCH_CASE(FP8_SCALE_MX_1x32_OCP)
#undef FP8Q_BATCH_CASE
        default:
            break;
    }
}

// ------------------------------------------------- fused current scaling

// Per-tensor current scaling in one cooperative launch: amax of x, the
// compute_bias rule, and the cast with 2^e.  Phase 1 reduces max|x| per CTA and
// folds it into one workspace word with an atomic max; the last CTA to reach
// the grid barrier reads that word, derives e, writes the caller's amax / bias /
// scale / scale_inv, publishes 2^e and releases the others (a generation
// counter; it zeroes the max and the count, so the workspace is left ready for
// the next call); phase 2 is the tile loop of the cast kernel.  One word instead
// of a slot per CTA that the last CTA reads one by one: 10-12 us less per call.
struct CurrentWorkspace {
    unsigned count;      // CTAs arrived at the barrier of the current call
    unsigned gen;        // barrier generation
    float scale;         // 2^e of the current call
    unsigned amax_bits;  // max |x| of the current call (bf16 magnitude bits, NaN above inf); 0 at rest
};
constexpr int kCurrentWsHeader = 16;
static_assert(sizeof(CurrentWorkspace) == kCurrentWsHeader, "barrier header layout");

struct CurrentOut {
    float* amax;
    int32_t* bias;
    float* scale;
    float* scale_inv;
    int32_t* status;
    int margin;
};

template <int FMT>
__global__ void __launch_bounds__(kThreads, 3)
    quantize_current_kernel(const __grid_constant__ QuantMaps maps, QuantArgs a, const uint16_t* x, int64_t ld,
                            CurrentOut out, CurrentWorkspace* ws) {
    __shared__ uint32_t red[kThreads / 32];
    __shared__ float s_scale;
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // phase 1: max |x| of this CTA's share of 16-byte chunks
    const int64_t cpr = a.cols >> 3;
    const int64_t total = a.rows * cpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    auto addr = [&](int64_t id) -> const uint16_t* {
        return (ld == a.cols) ? x + id * 8 : x + (id / cpr) * ld + (id % cpr) * 8;
    };
    uint32_t m = 0;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + tid;
    for (; i + 3 * stride < total; i += 4 * stride) {
        const uint4 v0 = ld_stream_v4(addr(i)), v1 = ld_stream_v4(addr(i + stride));
        const uint4 v2 = ld_stream_v4(addr(i + 2 * stride)), v3 = ld_stream_v4(addr(i + 3 * stride));
        m = absmax2(absmax2(absmax2(absmax2(m, v0.x), v0.y), v0.z), v0.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v1.x), v1.y), v1.z), v1.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v2.x), v2.y), v2.z), v2.w);
        m = absmax2(absmax2(absmax2(absmax2(m, v3.x), v3.y), v3.z), v3.w);
    }
    for (; i < total; i += stride) {
        const uint4 v = ld_stream_v4(addr(i));
        m = absmax2(absmax2(absmax2(absmax2(m, v.x), v.y), v.z), v.w);
    }
    m = __reduce_max_sync(0xffffffffu, fold2(m));
    if (lane == 0) red[warp] = m;
    __syncthreads();

    // grid barrier (bounded wait), scale selection by the last CTA
    if (tid == 0) {
        uint32_t mx = red[0];
        for (int w = 1; w < kThreads / 32; ++w) mx = max(mx, red[w]);
        volatile CurrentWorkspace* vws = ws;
        const unsigned gen0 = vws->gen;
        atomicMax(&ws->amax_bits, mx);  // before this CTA counts itself in
        __threadfence();
        s_abort = 0;
        if (atomicAdd(&ws->count, 1u) == gridDim.x - 1) {
            __threadfence();
            const uint32_t all = vws->amax_bits;  // every CTA's max arrived before its count
            vws->amax_bits = 0;
            const float amax = bf16bits_to_float(all);
            bool nf = false;
            const int e = bias_from_amax(amax, FMT, out.margin, &nf);
            if (out.amax) *out.amax = amax;
            if (out.bias) *out.bias = e;
            if (out.scale) *out.scale = pow2_exact(e);
            if (out.scale_inv) *out.scale_inv = pow2_exact(-e);
            if (nf && out.status) atomicOr(out.status, FP8_STATUS_NONFINITE_AMAX);
            vws->scale = pow2_exact(e);
            vws->count = 0;
            __threadfence();
            atomicAdd(&ws->gen, 1u);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (vws->gen == gen0) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    s_abort = 1;
                    if (out.status) atomicOr(out.status, FP8_STATUS_TIMEOUT);
                    break;
                }
            }
            __threadfence();
        }
        s_scale = vws->scale;
    }
    __syncthreads();
    if (s_abort) return;

    // phase 2: the cast
    quantize_tiles<FP8_SCALE_TENSOR, FMT>(&maps, a, s_scale, blockIdx.x, gridDim.x, /*from_end=*/true);
}

// Per-tensor scaled cast of an fp32 tensor: q = Encode(fl32(x s)), grid-stride over 8-element
// chunks (two 16-byte loads, one 8-byte store); the n % 8 tail is cast by the first threads of
// CTA 0.  The fused amax takes the largest |x| bit pattern, so a NaN wins.
template <int FMT>
__global__ void __launch_bounds__(256) cast_f32_kernel(const float* x, int64_t n, const float* scale, uint8_t* q,
                                                       float* amax) {
    const float s = scale ? *scale : 1.0f;
    const int64_t n8 = n >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 a = ld_stream_v4(x + 8 * i), b = ld_stream_v4(x + 8 * i + 4);
        const uint32_t lo = cvt_fp8x2<FMT>(__fmul_rn(__uint_as_float(a.x), s), __fmul_rn(__uint_as_float(a.y), s)) |
                            (cvt_fp8x2<FMT>(__fmul_rn(__uint_as_float(a.z), s), __fmul_rn(__uint_as_float(a.w), s)) << 16);
        const uint32_t hi = cvt_fp8x2<FMT>(__fmul_rn(__uint_as_float(b.x), s), __fmul_rn(__uint_as_float(b.y), s)) |
                            (cvt_fp8x2<FMT>(__fmul_rn(__uint_as_float(b.z), s), __fmul_rn(__uint_as_float(b.w), s)) << 16);
        *reinterpret_cast<uint2*>(q + 8 * i) = make_uint2(lo, hi);
        m = max(m, max(max(max(a.x & 0x7FFFFFFFu, a.y & 0x7FFFFFFFu), max(a.z & 0x7FFFFFFFu, a.w & 0x7FFFFFFFu)),
                       max(max(b.x & 0x7FFFFFFFu, b.y & 0x7FFFFFFFu), max(b.z & 0x7FFFFFFFu, b.w & 0x7FFFFFFFu))));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
        const int64_t i = 8 * n8 + threadIdx.x;
        const uint32_t u = __float_as_uint(x[i]);
        q[i] = (uint8_t)cvt_fp8x2<FMT>(__fmul_rn(__uint_as_float(u), s), 0.0f);
        m = max(m, u & 0x7FFFFFFFu);
    }
    if (amax) {
        m = __reduce_max_sync(0xffffffffu, m);
        if ((threadIdx.x & 31) == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(amax), m);
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

// The ratio alternative: scale = fmax / amax, scale_inv = 1 / scale, each rounded to nearest.
__global__ void compute_scale_ratio_kernel(const float* amax, int fmt, float* scale, float* scale_inv,
                                           int32_t* status) {
    const float a = fabsf(*amax);
    const bool nf = !(a <= 3.402823466e38f);  // NaN or Inf
    const float s = (nf || a == 0.0f) ? 1.0f : __fdiv_rn(fmt == FP8_E4M3 ? 448.0f : 57344.0f, a);
    if (scale) *scale = s;
    if (scale_inv) *scale_inv = __fdiv_rn(1.0f, s);
    if (nf && status) atomicOr(status, FP8_STATUS_NONFINITE_AMAX);
}

// One delayed-scaling step in one CTA: record, window max, bias, reset.
__device__ __forceinline__ void history_step(float* hist, int len, int64_t* pos, float* amax, int fmt, int margin,
                                             int32_t* bias, float* scale, float* scale_inv, int32_t* status) {
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

__global__ void __launch_bounds__(1024) history_kernel(float* hist, int len, int64_t* pos, float* amax, int fmt,
                                                       int margin, int32_t* bias, float* scale, float* scale_inv,
                                                       int32_t* status) {
    history_step(hist, len, pos, amax, fmt, margin, bias, scale, scale_inv, status);
}

// Many independent delayed-scaling states in one launch: CTA b runs the step of state b.
constexpr int kHistBatch = 48;  // records per launch (48 x 72 bytes of kernel parameters)
struct HistBatch {
    fp8_history_state s[kHistBatch];
};

__global__ void __launch_bounds__(1024) history_batch_kernel(const __grid_constant__ HistBatch b) {
    const fp8_history_state& st = b.s[blockIdx.x];
    history_step(st.history, st.len, st.pos, st.amax, st.fmt, st.margin, st.bias, st.scale, st.scale_inv, st.status);
}

PFN_cuTensorMapEncodeTiled_v12000 q_encode_fn() {
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

template <int GRAN, int FMT>
fp8_status launch_quant(const QuantMaps& tm, const QuantArgs& a, cudaStream_t st) {
    auto k = quantize_tile_kernel<GRAN, FMT>;
    const size_t smem = sizeof(QuantSmem) + 1024;
    int occ = 0;
    fp8_status s = resident_ctas(reinterpret_cast<const void*>(k), kThreads, smem, &occ);
    if (s != FP8_OK) return s;
    const int64_t cap = (int64_t)device_sm_count() * occ;
    const int grid = (int)(a.ntiles < cap ? a.ntiles : cap);
    k<<<grid, kThreads, smem, st>>>(tm, a);
    return check_launch("quantize kernel launch");
}

}  // namespace

// ------------------------------------------------------------------- host API

// Resident CTAs per SM of `kernel` (`threads` threads, `smem` bytes of dynamic shared memory) on the
// current device.  The first call for a kernel on a device raises its shared-memory limit and queries
// the occupancy; the answer is kept in a fixed table (no heap allocation), so later calls, including
// those made while a stream is being captured, make neither CUDA call.
fp8_status resident_ctas(const void* kernel, int threads, size_t smem, int* occ) {
    struct Entry {
        const void* kernel;
        int dev, occ;
    };
    constexpr int kEntries = 256;  // 12 cast and 8 statistics kernels per device
    static std::mutex mu;
    static Entry table[kEntries];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].kernel == kernel && table[i].dev == dev) {
            *occ = table[i].occ;
            return FP8_OK;
        }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, smem);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
    FP8_REQUIRE(o > 0, FP8_ERR_CUDA, "a %d-thread CTA with %zu bytes of shared memory does not fit on an SM", threads,
                smem);
    if (used < kEntries) table[used++] = Entry{kernel, dev, o};
    *occ = o;
    return FP8_OK;
}

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    static std::atomic<int> cache[64];  // zero until the first query on that device
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
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

fp8_status launch_quantize_f32(const float* x, int64_t n, int fmt, const float* scale, uint8_t* q, float* amax,
                               cudaStream_t st) {
    int64_t grid = ((n >> 3) + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (fmt == FP8_E4M3)
        cast_f32_kernel<FP8_E4M3><<<(int)grid, 256, 0, st>>>(x, n, scale, q, amax);
    else
        cast_f32_kernel<FP8_E5M2><<<(int)grid, 256, 0, st>>>(x, n, scale, q, amax);
    return check_launch("fp32 cast kernel launch");
}

fp8_status launch_compute_scale(const float* amax, int fmt, int margin, int32_t* bias, float* scale,
                                float* scale_inv, int32_t* status, cudaStream_t st) {
    compute_scale_kernel<<<1, 1, 0, st>>>(amax, fmt, margin, bias, scale, scale_inv, status);
    return check_launch("compute_scale kernel launch");
}

fp8_status launch_compute_scale_ratio(const float* amax, int fmt, float* scale, float* scale_inv, int32_t* status,
                                      cudaStream_t st) {
    compute_scale_ratio_kernel<<<1, 1, 0, st>>>(amax, fmt, scale, scale_inv, status);
    return check_launch("compute_scale_ratio kernel launch");
}

fp8_status launch_history(float* hist, int len, int64_t* pos, float* amax, int fmt, int margin, int32_t* bias,
                          float* scale, float* scale_inv, int32_t* status, cudaStream_t st) {
    const int threads = len >= 1024 ? 1024 : ((len + 31) / 32) * 32;
    history_kernel<<<1, threads, 0, st>>>(hist, len, pos, amax, fmt, margin, bias, scale, scale_inv, status);
    return check_launch("history kernel launch");
}

fp8_status launch_history_batch(const fp8_history_state* states, int n, cudaStream_t st) {
    for (int first = 0; first < n; first += kHistBatch) {
        const int cnt = n - first < kHistBatch ? n - first : kHistBatch;
        HistBatch b;
        memset(&b, 0, sizeof(b));
        int longest = 1;
        for (int i = 0; i < cnt; ++i) {
            b.s[i] = states[first + i];
            longest = b.s[i].len > longest ? b.s[i].len : longest;
        }
        const int threads = longest >= 1024 ? 1024 : ((longest + 31) / 32) * 32;
        history_batch_kernel<<<cnt, threads, 0, st>>>(b);
        fp8_status s = check_launch("history batch kernel launch");
        if (s != FP8_OK) return s;
    }
    return FP8_OK;
}

namespace {

// bf16 [rows x cols] (row stride ld) in 128 x 128 boxes, no swizzle.
fp8_status make_x_map(const void* x, int64_t rows, int64_t cols, int64_t ld, CUtensorMap* tm) {
    auto fn = q_encode_fn();
    FP8_REQUIRE(fn != nullptr, FP8_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kTile};  // one 64-column half of a tile: 128-byte rows
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    FP8_REQUIRE(r == CUDA_SUCCESS, FP8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FP8_OK;
}

// The launch's maps: x as above; the column-wise output u8 [cols x rows] (rows a multiple of 16, base
// 16-byte aligned, both checked by the API) in 128 (rows) x 128 (columns) boxes with the 128B swizzle
// the kernel stages them in.  Without a column-wise output the second map is left zero and unused.
fp8_status make_maps(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q_col, QuantMaps* m) {
    fp8_status s = make_x_map(x, rows, cols, ld, &m->x);
    if (s != FP8_OK) return s;
    memset(&m->qc, 0, sizeof(m->qc));
    if (!q_col) return FP8_OK;
    auto fn = q_encode_fn();
    FP8_REQUIRE(fn != nullptr, FP8_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)rows, (cuuint64_t)cols};
    cuuint64_t strides[1] = {(cuuint64_t)rows};
    cuuint32_t box[2] = {(cuuint32_t)kTile, (cuuint32_t)kTile};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&m->qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_col, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    FP8_REQUIRE(r == CUDA_SUCCESS, FP8_ERR_CUDA, "cuTensorMapEncodeTiled (column-wise output) failed (%d)", (int)r);
    return FP8_OK;
}

__global__ void current_empty_kernel(CurrentOut out) {
    if (out.amax) *out.amax = 0.0f;
    if (out.bias) *out.bias = 0;
    if (out.scale) *out.scale = 1.0f;
    if (out.scale_inv) *out.scale_inv = 1.0f;
}

template <int FMT>
fp8_status launch_current(const QuantMaps& tm, const QuantArgs& a, const void* x, int64_t ld, const CurrentOut& out,
                          void* workspace, cudaStream_t st) {
    auto k = quantize_current_kernel<FMT>;
    const size_t smem = sizeof(QuantSmem) + 1024;
    int occ = 0;
    fp8_status s = resident_ctas(reinterpret_cast<const void*>(k), kThreads, smem, &occ);
    if (s != FP8_OK) return s;
    // every CTA must be resident at once (grid barrier): at most SMs x occupancy
    int64_t grid = (int64_t)device_sm_count() * occ;
    if (grid > a.ntiles) grid = a.ntiles;
    if (grid < 1) grid = 1;
    QuantMaps tm_arg = tm;
    QuantArgs a_arg = a;
    const uint16_t* x_arg = static_cast<const uint16_t*>(x);
    int64_t ld_arg = ld;
    CurrentOut out_arg = out;
    CurrentWorkspace* ws_arg = static_cast<CurrentWorkspace*>(workspace);
    void* args[] = {&tm_arg, &a_arg, &x_arg, &ld_arg, &out_arg, &ws_arg};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k), dim3((unsigned)grid),
                                                dim3(kThreads), args, smem, st);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cooperative launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

QuantArgs quant_args(int64_t rows, int64_t cols, int margin, const float* scale, uint8_t* q_row, uint8_t* q_col,
                     void* sf_row, void* sf_col, float* amax) {
    QuantArgs a;
    a.rows = rows;
    a.cols = cols;
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
    a.status = nullptr;
    return a;
}

}  // namespace

fp8_status launch_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int gran, int margin,
                           const float* scale, uint8_t* q_row, uint8_t* q_col, void* sf_row, void* sf_col,
                           float* amax, cudaStream_t st) {
    QuantMaps tm;
    fp8_status s = make_maps(x, rows, cols, ld, q_col, &tm);
    if (s != FP8_OK) return s;
    const QuantArgs a = quant_args(rows, cols, margin, scale, q_row, q_col, sf_row, sf_col, amax);
#define FP8Q_QDISPATCH(G)                                                         \
    case G:                                                                       \
        return fmt == FP8_E4M3 ? launch_quant<G, FP8_E4M3>(tm, a, st) : launch_quant<G, FP8_E5M2>(tm, a, st);
    switch (gran) {
        FP8Q_QDISPATCH(FP8_SCALE_TENSOR)
        FP8Q_QDISPATCH(FP8_SCALE_BLOCK_1x128)
        FP8Q_QDISPATCH(FP8_SCALE_BLOCK_128x128)
        FP8Q_QDISPATCH(FP8_SCALE_MX_1x32)
        FP8Q_QDISPATCH(FP8_SCALE_MX_1x32_OCP)
    }
#undef FP8Q_QDISPATCH
    return FP8_ERR_UNSUPPORTED;
}

fp8_status launch_quantize_batch(const fp8_quantize_desc* descs, int n, cudaStream_t st) {
    QuantBatch b;
    memset(&b, 0, sizeof b);
    int64_t tiles[kMaxBatch];
    int m = 0;  // non-empty casts
    for (int i = 0; i < n; ++i) {
        const fp8_quantize_desc& d = descs[i];
        if (d.rows == 0 || d.cols == 0) continue;
        fp8_status s = make_maps(d.x, d.rows, d.cols, d.ld, d.q_col, &b.maps[m]);
        if (s != FP8_OK) return s;
        b.a[m] = quant_args(d.rows, d.cols, d.margin, d.scale, d.q_row, d.q_col, d.sf_row, d.sf_col, d.amax);
        b.kind[m] = 2 * d.gran + d.fmt;
        tiles[m] = b.a[m].ntiles;
        ++m;
    }
    if (m == 0) return FP8_OK;
    b.n = m;
    const size_t smem = sizeof(QuantSmem) + 1024;
    int occ = 0;
    fp8_status s = resident_ctas(reinterpret_cast<const void*>(quantize_batch_kernel), kThreads, smem, &occ);
    if (s != FP8_OK) return s;
    int64_t total = 0;
    for (int k = 0; k < m; ++k) total += tiles[k];
    const int64_t cap = (int64_t)device_sm_count() * occ;
    const int grid = (int)(total < cap ? total : cap);  // >= m: every tensor has a tile
    // one CTA per tensor, then each further CTA to the tensor whose share has the most rounds of tiles
    // left: the launch lasts as long as its slowest share
    int share[kMaxBatch];
    for (int k = 0; k < m; ++k) share[k] = 1;
    for (int used = m; used < grid; ++used) {
        int best = -1;
        int64_t best_rounds = 0;
        for (int k = 0; k < m; ++k) {
            const int64_t rounds = (tiles[k] + share[k] - 1) / share[k];
            if (share[k] < tiles[k] && rounds > best_rounds) {
                best = k;
                best_rounds = rounds;
            }
        }
        if (best < 0) break;
        ++share[best];
    }
    b.cta0[0] = 0;
    for (int k = 0; k < m; ++k) b.cta0[k + 1] = b.cta0[k] + share[k];
    quantize_batch_kernel<<<b.cta0[m], kThreads, smem, st>>>(b);
    return check_launch("batched quantize kernel launch");
}

fp8_status launch_quantize_current(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int margin,
                                   uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias, float* scale,
                                   float* scale_inv, void* workspace, int32_t* status, cudaStream_t st) {
    const CurrentOut out{amax, bias, scale, scale_inv, status, margin};
    if (rows == 0 || cols == 0) {
        current_empty_kernel<<<1, 1, 0, st>>>(out);
        return check_launch("current-scaling kernel launch");
    }
    QuantMaps tm;
    fp8_status s = make_maps(x, rows, cols, ld, q_col, &tm);
    if (s != FP8_OK) return s;
    QuantArgs a = quant_args(rows, cols, margin, nullptr, q_row, q_col, nullptr, nullptr, nullptr);
    a.status = status;
    return fmt == FP8_E4M3 ? launch_current<FP8_E4M3>(tm, a, x, ld, out, workspace, st)
                           : launch_current<FP8_E5M2>(tm, a, x, ld, out, workspace, st);
}

// ------------------------------------------- fused current scaling, no allocation
//
// fp8_quantize_current_noalloc runs the same kernel as fp8_quantize_current, with
// its barrier header in the library's own static device array instead of a
// caller workspace.  It is for callers that cannot allocate
// device memory at the point of the call: a plugin or callback that a host
// framework hands only its input and output buffers, code whose device memory is
// planned once at start-up against a fixed budget, and latency-bound loops that
// cannot take the device-wide synchronisation cudaMalloc / cudaFree may cause.
//
// The array is kNoAllocScratchBytes (256 bytes) on every GPU that loads the
// library, held until the process exits; the kernel uses its 16-byte header
// (arrival count, generation, scale, the atomic max).  Every call shares the
// array and finds the previous call's contents there; the call clears the header
// on its stream before the kernel.  Calls whose kernels overlap on the GPU (other
// streams, other host threads) race on the array.
constexpr int kNoAllocScratchBytes = 256;
static_assert(kNoAllocScratchBytes >= kCurrentWsHeader, "scratch holds the barrier header");
static __device__ __align__(256) unsigned char g_current_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_current_scratch on the current device.  In host code the
// array's name only stands for the symbol; the first call on each device looks
// its address up, with that device current, and caches it.
fp8_status noalloc_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    FP8_REQUIRE(dev >= 0 && dev < 64, FP8_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
    // read without a lock once cached; the mutex only serialises the first lookup on a device
    static std::atomic<void*> addr[64];
    static std::mutex mu;
    void* p = addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(mu);
        p = addr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            e = cudaGetSymbolAddress(&p, g_current_scratch);
            FP8_REQUIRE(e == cudaSuccess && p != nullptr, FP8_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                        cudaGetErrorString(e));
            addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return FP8_OK;
}

template <int FMT>
fp8_status launch_current_noalloc(const QuantMaps& tm, const QuantArgs& a, const void* x, int64_t ld,
                                  const CurrentOut& out, void* scratch, cudaStream_t st) {
    auto k = quantize_current_kernel<FMT>;
    const size_t smem = sizeof(QuantSmem) + 1024;
    int occ = 0;
    fp8_status s = resident_ctas(reinterpret_cast<const void*>(k), kThreads, smem, &occ);
    if (s != FP8_OK) return s;
    int64_t grid = (int64_t)device_sm_count() * occ;  // all CTAs resident at once (grid barrier)
    if (grid > a.ntiles) grid = a.ntiles;
    if (grid < 1) grid = 1;
    cudaError_t e = cudaMemsetAsync(scratch, 0, kCurrentWsHeader, st);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cudaMemsetAsync(scratch header): %s", cudaGetErrorString(e));
    QuantMaps tm_arg = tm;
    QuantArgs a_arg = a;
    const uint16_t* x_arg = static_cast<const uint16_t*>(x);
    int64_t ld_arg = ld;
    CurrentOut out_arg = out;
    CurrentWorkspace* ws_arg = static_cast<CurrentWorkspace*>(scratch);
    void* args[] = {&tm_arg, &a_arg, &x_arg, &ld_arg, &out_arg, &ws_arg};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k), dim3((unsigned)grid), dim3(kThreads), args,
                                    smem, st);
    FP8_REQUIRE(e == cudaSuccess, FP8_ERR_CUDA, "cooperative launch: %s", cudaGetErrorString(e));
    return FP8_OK;
}

}  // namespace

fp8_status launch_quantize_current_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt,
                                           int margin, uint8_t* q_row, uint8_t* q_col, float* amax, int32_t* bias,
                                           float* scale, float* scale_inv, int32_t* status, cudaStream_t st) {
    const CurrentOut out{amax, bias, scale, scale_inv, status, margin};
    if (rows == 0 || cols == 0) {
        current_empty_kernel<<<1, 1, 0, st>>>(out);
        return check_launch("current-scaling kernel launch");
    }
    void* scratch = nullptr;
    fp8_status s = noalloc_scratch(&scratch);
    if (s != FP8_OK) return s;
    QuantMaps tm;
    s = make_maps(x, rows, cols, ld, q_col, &tm);
    if (s != FP8_OK) return s;
    QuantArgs a = quant_args(rows, cols, margin, nullptr, q_row, q_col, nullptr, nullptr, nullptr);
    a.status = status;
    return fmt == FP8_E4M3 ? launch_current_noalloc<FP8_E4M3>(tm, a, x, ld, out, scratch, st)
                           : launch_current_noalloc<FP8_E5M2>(tm, a, x, ld, out, scratch, st);
}

}  // namespace fp8q
