// Shared device helpers of the nvfp4rl library (sm_103a).
//
// Contents: the NVFP4 element/scale conversions used by both quantizers, the
// bounded mbarrier wait every pipelined kernel uses, and thin inline-PTX
// wrappers for TMA, mbarrier and the tcgen05 tensor-core instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "nvfp4rl.h"

namespace nvfp4rl {

// ----------------------------------------------------------------- host side

constexpr int kMaxDevices = 64;

struct LaunchCtx {
    cudaStream_t stream;
    int* status;      // device status word (NVFP4_ERR_TIMEOUT is recorded here)
    int num_sms;
    int device;       // current device ordinal, < kMaxDevices
};

// Launch-time occupancy of one kernel, cached per device: the count (co-resident CTAs
// per SM, or clusters per device) for the dynamic shared-memory size it was last
// computed for.  Filling an entry also raises the kernel's opt-in shared-memory limit
// on that device, so a hit needs neither runtime call again.  The cache assumes the
// device's primary context lives as long as the process.
struct OccupancyCache {
    std::atomic<uint64_t> entry[kMaxDevices];  // (smem bytes << 32) | count; 0 = empty
    int lookup(int dev, size_t smem) const {
        const uint64_t v = entry[dev].load(std::memory_order_acquire);
        return (v >> 32) == (uint64_t)smem ? (int)(uint32_t)v : 0;
    }
    void store(int dev, size_t smem, int count) {
        entry[dev].store(((uint64_t)smem << 32) | (uint32_t)count, std::memory_order_release);
    }
};

// Co-resident CTAs per SM of `kern` (at least 1) with `threads` threads and `smem` bytes.
template <typename Kern>
cudaError_t blocks_per_sm(OccupancyCache& cache, const LaunchCtx& ctx, Kern kern, int threads,
                          size_t smem, int* out) {
    int n = cache.lookup(ctx.device, smem);
    if (n == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem);
        if (e != cudaSuccess) return e;
        if (n < 1) n = 1;
        cache.store(ctx.device, smem, n);
    }
    *out = n;
    return cudaSuccess;
}

// Co-resident clusters of `kern` for the launch configuration `cfg` (its grid is
// ignored by the query; block size, shared memory and cluster size count).
template <typename Kern>
cudaError_t clusters_per_device(OccupancyCache& cache, const LaunchCtx& ctx, Kern kern,
                                const cudaLaunchConfig_t& cfg, int* out) {
    int n = cache.lookup(ctx.device, cfg.dynamicSmemBytes);
    if (n == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        cache.store(ctx.device, cfg.dynamicSmemBytes, n);
    }
    *out = n;
    return cudaSuccess;
}

// Implemented per translation unit; each returns cudaSuccess or the launch error.
cudaError_t launch_act_quant(const LaunchCtx&, const __nv_bfloat16* X, int64_t M, int64_t K,
                             uint8_t* codes, uint8_t* sf, float* s_row);
cudaError_t launch_act_quant_prescaled(const LaunchCtx&, const __nv_bfloat16* X, int64_t M, int64_t K,
                                       const float* row_amax, uint8_t* codes, uint8_t* sf, float* s_row);
cudaError_t launch_requant(const LaunchCtx&, const void* W, int w_dtype, const float* A,
                           const float* B, int r, float c, int64_t N, int64_t K, uint8_t* codes,
                           uint8_t* sf, float* s_t);
// Tensor-core merge (merge_tc.cu): bf16 W, rank 32, 16-byte aligned A and B, and a
// workspace of requant_tc_workspace_bytes (0 when the path does not apply) laid out by
// requant_tc_layout: A' [K, 128] bf16, rnorm [N rounded up to 256], cnorm [K / 128
// rounded up][4], two CTA counters (the grid barrier between the amax and quantize
// phases; the last CTA, which finishes the per-tensor scale).
struct RequantTcLayout {
    uint8_t* ap;
    float* rnorm;
    float* cnorm;
    unsigned int* counter;
    size_t bytes;
};
inline RequantTcLayout requant_tc_layout(void* base, int64_t N, int64_t K) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const uintptr_t p = reinterpret_cast<uintptr_t>(base);
    RequantTcLayout l;
    size_t off = 0;
    l.ap = reinterpret_cast<uint8_t*>(p + off);
    off += up((size_t)K * 256);
    l.rnorm = reinterpret_cast<float*>(p + off);
    off += up((size_t)((N + 255) / 256 * 256) * 4);
    l.cnorm = reinterpret_cast<float*>(p + off);
    off += up((size_t)((K + 127) / 128) * 16);
    l.counter = reinterpret_cast<unsigned int*>(p + off);
    off += 256;
    l.bytes = off;
    return l;
}
// Tensor maps of the merge kernel: W [N, K] bf16 (64 x 128 boxes) and A' [K, 128] bf16
// (64 x 64 boxes), both with the 128-byte swizzle.
struct RequantTcMaps {
    CUtensorMap w, ap;
};
size_t requant_tc_workspace_bytes(int w_dtype, int r, int64_t N, int64_t K);
cudaError_t launch_requant_tc(const LaunchCtx&, const RequantTcMaps& maps, const void* W,
                              const float* A, const float* B, void* workspace, float c, int64_t N,
                              int64_t K, uint8_t* codes, uint8_t* sf, float* s_t);
cudaError_t launch_test_merge(const LaunchCtx&, const void* W, int w_dtype, const float* A,
                              const float* B, int r, float c, int64_t N, int64_t K, float* out);
cudaError_t launch_select(const LaunchCtx&, const float* rewards, int P, int N, int K,
                          int global_std, int32_t* idx, float* r_out);
cudaError_t launch_test_e2m1(const LaunchCtx&, const float* q, uint8_t* codes, int64_t n);
cudaError_t launch_test_e4m3(const LaunchCtx&, const float* v, uint8_t* codes, int64_t n);
cudaError_t launch_test_e4m3_decode(const LaunchCtx&, const uint8_t* codes, float* out, int64_t n);
cudaError_t launch_test_e2m1_quotient(const LaunchCtx&, const float* x, const float* den,
                                      uint8_t* codes, int64_t n);
cudaError_t launch_test_e4m3_quotient(const LaunchCtx&, const float* v, const float* d,
                                      uint8_t* codes, int64_t n);
// GEMMs: tensor maps are encoded by the caller (host) and passed by value.
cudaError_t launch_gemm_nvfp4(const LaunchCtx&, const CUtensorMap& tmap_a,
                              const CUtensorMap& tmap_b, const CUtensorMap& tmap_sfa,
                              const CUtensorMap& tmap_sfb, const CUtensorMap& tmap_y,
                              const float* a_srow, const float* w_st, const __nv_bfloat16* bias,
                              int64_t M, int64_t N, int64_t K, int withhold_kb = -1,
                              int64_t wait_limit_ns = 0, float* row_amax = nullptr);
cudaError_t launch_gemm_bf16(const LaunchCtx&, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                             const __nv_bfloat16* bias, int64_t M, int64_t N, int64_t K);
cudaError_t launch_test_wait_timeout(const LaunchCtx&, int64_t timeout_ns);

// ----------------------------------------------------------------- device side

#if defined(__CUDACC__)

// NVFP4 / E4M3 constants of the two-level scale convention.
constexpr float kE2M1Max = 6.0f;
constexpr float kE4M3Max = 448.0f;
constexpr float kAmaxDiv = 2688.0f;  // 6 * 448

// E2M1 codes of 8 fp32 values, round to nearest even, saturating, sign kept.
// Element i lands in bits 4i..4i+3 of the result (element 0 in the low nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float q0, float q1, float q2, float q3, float q4,
                                               float q5, float q6, float q7) {
    uint32_t out;
    // cvt ...e2m1x2.f32 d, a, b puts a in the high nibble and b in the low one.
    asm("{\n\t"
        ".reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t"
        "}"
        : "=r"(out)
        : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
    return out;
}

// E4M3 code (round to nearest even, saturating at 448) of v >= 0.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
    unsigned short out;
    // cvt ...e4m3x2.f32 d, a, b puts a in the high byte and b in the low one.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
    return (uint32_t)out & 0xFFu;
}

// Value of a non-negative E4M3 code, by the hardware conversion E4M3 -> f16 (every
// E4M3 value is an f16 value) and f16 -> f32 (exact).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    const unsigned short c = (unsigned short)(code & 0xFFu);
    // cvt ...f16x2.e4m3x2 d, a: the low byte of a lands in the low half of d.
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// True when the fp32 value with bit pattern u lies within 16 ulps of a number with
// at most (23 - kLowBits + 1) significant bits, i.e. when its low kLowBits mantissa
// bits are within 16 of 0 modulo 2^kLowBits.  Every E2M1 rounding boundary (0.25,
// 0.75, 1.25, 1.75, 2.5, 3.5, 5) has 3 significant bits (kLowBits = 20); every E4M3
// boundary (midpoints of adjacent codes) has at most 5 (kLowBits = 18).
//
// Written as one shift-add and one compare: shifting out the top 32 - kLowBits bits
// leaves ((u + 16) mod 2^kLowBits) * 2^(32 - kLowBits).
template <int kLowBits>
__device__ __forceinline__ uint32_t near_key(uint32_t u) {
    return (u << (32 - kLowBits)) + (16u << (32 - kLowBits));
}
template <int kLowBits>
__device__ __forceinline__ bool near_boundary(uint32_t u) {
    return near_key<kLowBits>(u) < (32u << (32 - kLowBits));
}

// Approximate reciprocal, at most 1 ulp from 1/d for normal d whose reciprocal is
// normal (the hardware's documented bound for rcp.approx.f32).
__device__ __forceinline__ float recip_approx(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// A reciprocal usable by the fast paths: den in the normal range, so that 1/den is
// a normal number too (den <= 448 * FLT_MAX / 2688 keeps 1/den >= 2^-126).
__device__ __forceinline__ bool fast_recip_ok(float den) {
    return den >= 1.17549435e-38f && den <= 8.5e37f;
}

struct F8 {
    float v[8];
};

// Slow path of e2m1_quotient8: the codes of the elements flagged in `redo` (a nonzero
// nibble each) from true IEEE divisions, the others kept from `codes`.  bf16 inputs
// make it common for one element of a block to sit on a rounding boundary (the
// quotient is then close to a ratio of small integers), so it recomputes only those.
static __device__ __noinline__ uint32_t e2m1_exact8(F8 x, float den, uint32_t codes, uint32_t redo) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t sh = 4u * (uint32_t)i;
        if ((redo >> sh) & 0xFu) {
            const uint32_t c = cvt_e2m1x8(__fdiv_rn(x.v[i], den), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
            codes = (codes & ~(0xFu << sh)) | (c << sh);
        }
    }
    return codes;
}

static __device__ __noinline__ float exact_quotient(float v, float d) { return __fdiv_rn(v, d); }

// Bracketing reciprocals of a block's divisor den > 0 for e2m1_quotient8:
// lo = RD(r (1 - 2^-20)), hi = RU(r (1 + 2^-20)) with r = rcp.approx(den), which is
// within 1 ulp (< 2^-23 relative) of 1/den when den and 1/den are normal (`fast`).
struct Recip {
    float lo, hi;
    bool fast;
};
__device__ __forceinline__ Recip make_recip(float den) {
    Recip rc;
    rc.fast = fast_recip_ok(den);
    const float r = rc.fast ? recip_approx(den) : 0.0f;
    rc.lo = __fmul_rd(r, 1.0f - 0x1p-20f);
    rc.hi = __fmul_ru(r, 1.0f + 0x1p-20f);
    return rc;
}

// RNE_E2M1_sat(fl(x / den)) for 8 values sharing den > 0.
//
// Fast path: the quotient is bracketed.  lo = fl(x * rc.lo) and hi = fl(x * rc.hi)
// satisfy |lo| < |fl(x / den)| < |hi| with the same sign wherever a rounding decision
// is made (rc.lo <= (1/den)(1 - 7 2^-23) and rc.hi >= (1/den)(1 + 7 2^-23); each
// product and the quotient round by at most 2^-24 relatively; every E2M1 boundary is
// a normal number, and below the smallest one all three give code 0 or 0x8).  E2M1
// rounding is monotone in the magnitude, so if lo and hi give the same 8 codes so
// does fl(x / den).  Otherwise the codes that differ (a quotient within about 2^-20 of
// a rounding boundary, or an exact tie), and all 8 whenever den or 1/den is not a
// normal number, come from true IEEE divisions.  Zero stays zero with its sign in
// both products.
__device__ __forceinline__ uint32_t e2m1_quotient8(const float (&x)[8], float den, const Recip& rc) {
    float lo[8], hi[8];
    const float2 rl = make_float2(rc.lo, rc.lo), rh = make_float2(rc.hi, rc.hi);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 xv = make_float2(x[i], x[i + 1]);
        const float2 a = __fmul2_rn(xv, rl), b = __fmul2_rn(xv, rh);
        lo[i] = a.x;
        lo[i + 1] = a.y;
        hi[i] = b.x;
        hi[i + 1] = b.y;
    }
    const uint32_t c_lo = cvt_e2m1x8(lo[0], lo[1], lo[2], lo[3], lo[4], lo[5], lo[6], lo[7]);
    const uint32_t c_hi = cvt_e2m1x8(hi[0], hi[1], hi[2], hi[3], hi[4], hi[5], hi[6], hi[7]);
    if (!rc.fast || c_lo != c_hi) {
        F8 xv;
#pragma unroll
        for (int i = 0; i < 8; ++i) xv.v[i] = x[i];
        return e2m1_exact8(xv, den, c_hi, rc.fast ? c_lo ^ c_hi : 0xFFFFFFFFu);
    }
    return c_hi;
}

// RNE_E4M3_sat(fl(v / d)) for v >= 0, d > 0, with inv_d within 1 ulp of 1/d: same
// argument as above with the E4M3 boundaries (<= 5 significant bits).
__device__ __forceinline__ uint32_t e4m3_quotient(float v, float d, float inv_d, bool fast_ok) {
    float q = __fmul_rn(v, inv_d);
    if (!fast_ok || near_boundary<18>(__float_as_uint(q))) q = exact_quotient(v, d);
    return cvt_e4m3(q);
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Barrier `id` (1..15) among `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// kCluster: acquire at cluster scope, for barriers that threads of the peer CTA
// arrive on (their release.cluster arrivals then order their prior writes, including
// tensor-memory stores fenced before the arrival, before the waiter's later work).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    if (kCluster)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may sleep in the instruction until the phase
// completes or about kSuspendNs have passed (the hint bounds the sleep; completion
// wakes it), instead of spinning and taking issue slots from the warps that work.
constexpr uint32_t kSuspendNs = 20000;
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t done;
    if (kCluster)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
    return done != 0;
}

// A flag that another thread may raise at any time, read so that the whole warp agrees
// (set if any lane saw it set).  Per-lane reads of such a flag must never steer a warp's
// lanes down different paths ahead of a warp-collective operation (__all_sync, a
// shuffle, tcgen05.ld/st): the lanes would then wait at different collectives.
__device__ __forceinline__ bool warp_flag(const volatile int* f) { return __any_sync(0xFFFFFFFFu, *f != 0); }
__device__ __forceinline__ bool warp_flag(const volatile unsigned int* f) {
    return __any_sync(0xFFFFFFFFu, *f != 0u);
}

// Waits for the phase of `bar` with the given parity to complete, for at most
// limit_ns of device time.  On expiry it records NVFP4_ERR_TIMEOUT in *status,
// raises the CTA's abort flag (so the CTA's other waits give up at once) and
// returns false.  It also returns false as soon as another thread of the CTA
// has raised the abort flag (checked at least every kSuspendNs).  An iteration cap
// backs up the clock.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait<kCluster>(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait_sleep<kCluster>(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) break;
    }
    atomicCAS(status, 0, (int)NVFP4_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// --- TMA (bulk tensor / bulk copies into shared memory, completion on an mbarrier)

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// L2 eviction policies for TMA loads: evict_last keeps a tile in L2 for a second read
// soon after (a later pass over the same data), evict_first lets a last read go.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_load_2d with an L2 cache policy (from l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(const CUtensorMap* map, uint64_t* bar, void* dst,
                                                 int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Loads with acquire semantics at GPU scope (a flag or counter written by other CTAs).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// --- CTA pairs (two CTAs of a cluster sharing one 2-CTA MMA)

// The shared::cluster address of the object at CTA-local address `local` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(local), "r"(rank));
    return out;
}

// Arrive once on an mbarrier given by its shared::cluster address (possibly in a peer CTA).
//
// Default semantics (release at CTA scope).  The data these arrivals publish is
// tensor memory whose tcgen05 loads or stores the arriving thread has already waited
// for (tcgen05.wait, then tcgen05.fence::before_thread_sync), so no cluster-scope
// release of ordinary memory is needed; a .release.cluster arrive measured ~1,250
// cycles per arrive in the GEMM (it waits for the SM's outstanding memory traffic),
// against ~100 for this form.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Tile load into this CTA's shared memory whose completion is counted on an mbarrier
// of either CTA of the pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar_cluster,
                                                 void* dst, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(const CUtensorMap* map, uint32_t bar_cluster,
                                                 void* dst, int32_t c0, int32_t c1, int32_t c2,
                                                 int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Tensor-memory allocation for a CTA pair: one warp of EACH CTA of the pair executes
// these collectively; the same columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// 2-CTA MMAs, issued by one thread of the even CTA of the pair: A rows 0..127 come
// from the even CTA's shared memory and rows 128..255 from the odd CTA's (same
// offsets), B's first N/2 rows from the even CTA and the rest from the odd one;
// each CTA's tensor memory receives its own 128 rows of D.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As mma_bf16_pair with the A operand in tensor memory: each CTA's 128 rows of A in
// its own lanes 0..127 at column a_tmem, two bf16 per 32-bit column (K-major).
__device__ __forceinline__ void mma_bf16_pair_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_nvfp4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrive once, in every CTA of `cta_mask`, when the pair's tcgen05 operations issued
// so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// --- TMA stores (shared -> global), tracked per thread in bulk groups

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most kPending bulk groups of this thread still read shared memory.
template <int kPending>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}

template <int kPending>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(kPending) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster (hardware barrier; used once, after the
// mbarriers are initialized and before any CTA touches a peer's shared memory).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// bulk_load with an L2 cache policy (from l2_policy_*).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream (launched with the
// programmatic-serialization attribute) start, and wait until the previous one has
// completed with its memory visible.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --- tcgen05 (5th-generation tensor cores, accumulators in tensor memory)

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread (thread i
// reads lane base+i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 32 registers per thread -> 32 lanes x 32 consecutive 32-bit columns (thread i
// writes lane base+i); and the 16-column form.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Tile load into this CTA's shared memory, completion on this CTA's own mbarrier.
__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Warp-group register rebalancing.  The four warp groups of a 512-thread CTA are
// launched with 128 registers per thread; the counts requested below must add up
// to at most 4 x 128 per lane, or an increase would wait forever.
template <uint32_t kRegs>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bits 46..47, layout
// (swizzle) mode at bits 61..63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7u) << 61;
    return d;
}
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSw128 = 2;

#endif  // __CUDACC__

}  // namespace nvfp4rl
