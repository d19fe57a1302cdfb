// common.cuh -- device helpers shared by the kernels of libfp8q (sm_103a).
//
// Inline PTX wrappers for mbarriers, TMA, tcgen05 (TMEM allocation, MMA,
// commit, loads), the FP8 conversion instruction and the exact integer form of
// the FP8-AMAX bias rule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q.h"

namespace fp8q {

// --------------------------------------------------------------- host status

// Thread-local detail text for the last error (returned by fp8_last_error_detail).
void set_error_detail(const char* fmt, ...);

#define FP8_REQUIRE(cond, code, ...)          \
    do {                                      \
        if (!(cond)) {                        \
            ::fp8q::set_error_detail(__VA_ARGS__); \
            return (code);                    \
        }                                     \
    } while (0)

inline fp8_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error_detail("%s: %s", what, cudaGetErrorString(e));
        return FP8_ERR_CUDA;
    }
    return FP8_OK;
}

int device_sm_count();
// Resident CTAs per SM of `kernel` on the current device (cached per kernel and device; no heap).
fp8_status resident_ctas(const void* kernel, int threads, size_t smem, int* occ);

// ------------------------------------------------------------ bias / scales

// FP8-AMAX bias: e = floor(log2(fmax / amax)) - margin, exactly, from the bits.
// Write amax = m 2^Ea with m in [1, 2) and fmax = 1.75 2^Ef (Ef = 8 for E4M3's
// 448, 15 for E5M2's 57344).  fmax / amax = (1.75 / m) 2^(Ef - Ea) and
// 1.75 / m lies in (0.875, 1.75], so floor(log2) = Ef - Ea - [m > 1.75].
// m > 1.75 <=> the 23 fraction bits exceed 0.75 * 2^23 = 0x600000.
// amax == 0 -> 0; non-finite -> 0 with *nonfinite set; clamp to [-126, 127].
__host__ __device__ __forceinline__ int bias_from_amax(float amax, int fmt, int margin, bool* nonfinite) {
    uint32_t u;
#ifdef __CUDA_ARCH__
    u = __float_as_uint(amax) & 0x7FFFFFFFu;
#else
    __builtin_memcpy(&u, &amax, 4);
    u &= 0x7FFFFFFFu;
#endif
    if (u >= 0x7F800000u) {
        *nonfinite = true;
        return 0;
    }
    if (u == 0) return 0;
    int biased = (int)(u >> 23);
    uint32_t frac = u & 0x7FFFFFu;
    int ea;
    if (biased == 0) {  // fp32 subnormal: value = frac 2^-149; normalise
#ifdef __CUDA_ARCH__
        int msb = 31 - __clz(frac);
#else
        int msb = 31 - __builtin_clz(frac);
#endif
        ea = msb - 149;
        frac = (frac << (23 - msb)) & 0x7FFFFFu;
    } else {
        ea = biased - 127;
    }
    const int ef = (fmt == FP8_E4M3) ? 8 : 15;
    long long e = (long long)ef - ea - (frac > 0x600000u ? 1 : 0) - (long long)margin;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return (int)e;
}

// 2^e as an exact fp32 for e in [-149, 127].
// The OCP MX alternative, e = emax - floor(log2(amax)) - margin (emax = 8 for
// E4M3, 15 for E5M2), from the exponent bits; same special cases and clamping.
__host__ __device__ __forceinline__ int bias_from_amax_ocp(float amax, int fmt, int margin, bool* nonfinite) {
    uint32_t u;
#ifdef __CUDA_ARCH__
    u = __float_as_uint(amax) & 0x7FFFFFFFu;
#else
    __builtin_memcpy(&u, &amax, 4);
    u &= 0x7FFFFFFFu;
#endif
    if (u >= 0x7F800000u) {
        *nonfinite = true;
        return 0;
    }
    if (u == 0) return 0;
    int ea = (int)(u >> 23) - 127;
    if ((u >> 23) == 0) {  // subnormal: floor(log2) from the leading mantissa bit
        ea = -127;
        for (uint32_t m = u; m < 0x00400000u; m <<= 1) --ea;
    }
    int e = (fmt == FP8_E4M3 ? 8 : 15) - ea - margin;
    return e < -126 ? -126 : (e > 127 ? 127 : e);
}

__host__ __device__ __forceinline__ float pow2_exact(int e) {
    uint32_t u = (e >= -126) ? ((uint32_t)(e + 127) << 23) : (1u << (e + 149));
#ifdef __CUDA_ARCH__
    return __uint_as_float(u);
#else
    float f;
    __builtin_memcpy(&f, &u, 4);
    return f;
#endif
}

#ifdef __CUDACC__

// ------------------------------------------------------------ conversions

// Two fp32 -> two FP8 codes, round-to-nearest-even with saturation to the
// largest finite value (NaN stays NaN).  Low byte = `lo`.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == FP8_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Low / high bf16 of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Per-halfword max of |bf16| bit patterns: for non-negative bf16 (and NaN) the
// unsigned order of the bits is the numeric order, NaN above Inf.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }
__device__ __forceinline__ uint32_t fold2(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }
// bf16 magnitude bits -> fp32 value
__device__ __forceinline__ float bf16bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// --------------------------------------------------------------- memory

// 16-byte global store with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void st_global_v4_hint(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                  uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Longest time a kernel thread waits on one barrier phase before it gives up.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Bounded wait on `parity` of an mbarrier.  Returns false if *abort is raised
// by another role, or if the wait exceeds kWaitLimitNs (then it raises *abort).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Same, with an L2 cache policy (from createpolicy) attached to the load.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
        "[%4], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// TMA store of a shared-memory box to global memory (bulk-group completion).  Elements outside the
// tensor's extent are not written.  The generic-proxy writes that filled the box must be made
// visible to the async proxy first (fence_proxy_async_smem by every writer, then a barrier).
__device__ __forceinline__ void tma_store_2d(const void* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"((uint64_t)map),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
// Same, with an L2 cache policy (from createpolicy) attached to the store.
__device__ __forceinline__ void tma_store_2d_hint(const void* map, uint32_t src, int x, int y, uint64_t policy) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
                     (uint64_t)map),
                 "r"(x), "r"(y), "r"(src), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// at most N committed bulk groups are still reading their shared-memory sources
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// every committed bulk store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// D(tmem) (+)= A(smem) . B(smem)^T, FP8 operands, fp32 accumulate.
__device__ __forceinline__ void tc_mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled variant: per-32-K E8M0 scale factors of A and B read from TMEM.
__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit TMEM columns -> 32 registers per thread; waits for completion.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 4 consecutive 32-bit TMEM columns <- 4 registers per thread (no wait).
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t a) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------ CTA pairs (clusters of 2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrivals on a barrier of either CTA of the pair.  Relaxed: they publish no
// memory writes of the arriving thread (TMA data is tracked by the transaction
// count; TMEM reads are complete before an epilogue arrives), and a release at
// cluster scope would cost a memory fence on every K tile.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier that may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t cluster_bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (M = 256 across the pair) (+)= A . B^T, issued by the even CTA for both.
__device__ __forceinline__ void tc_mma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Block-scaled pair MMA: each CTA's TMEM holds the scales of its own 128 rows of A and of all N rows of B.
__device__ __forceinline__ void tc_mma_mxf8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                     uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask` when the pair MMAs issued so far complete.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(cta_mask)
                 : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// 128-byte swizzle: 8-row groups of 128-byte rows, 1024 bytes apart.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4 bits 46-48 fixed 0b001
//   bits 49-51 base offset (0: tiles are 1024-byte aligned)   bits 61-63 swizzle (2 = 128B)
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

#endif  // __CUDACC__

// Instruction descriptor of tcgen05.mma kind::f8f6f4 (dense, K-major A and B):
//   bits 4-5 D type (1 = f32), 7-9 A type, 10-12 B type (0 = E4M3, 1 = E5M2),
//   15/16 transpose A/B (0 = K-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(int fa, int fb, int m, int n) {
    return (1u << 4) | ((uint32_t)fa << 7) | ((uint32_t)fb << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor of kind::mxf8f6f4 with E8M0 scale factors:
//   bits 4-5 B scale-factor id, 7-9 A type, 10-12 B type, 17-22 N >> 3,
//   23 scale type (1 = UE8M0), 24-28 M >> 4, 29-30 A scale-factor id.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(int fa, int fb, int m, int n, int sfa_id, int sfb_id) {
    return ((uint32_t)sfb_id << 4) | ((uint32_t)fa << 7) | ((uint32_t)fb << 10) | ((uint32_t)(n >> 3) << 17) |
           (1u << 23) | ((uint32_t)(m >> 4) << 24) | ((uint32_t)sfa_id << 29);
}

}  // namespace fp8q
