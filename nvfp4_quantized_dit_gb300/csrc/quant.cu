// NVFP4 quantizers.
//
//  * act_quant: per-row ("per token") NVFP4 of BF16 activations for the
//    NVFP4-quantized solver of Sol-RL's Stage 1 (Sol-RL project page,
//    "Two-Stage Pipeline").  One pass over X: a row is held in registers while
//    its amax is reduced, then quantized from registers.
//  * requant: LoRA merge W' = W + (alpha/r) B A (rank 32 in the AI Trends
//    summary, paragraph on training stability) followed by per-tensor NVFP4,
//    run after every policy update (Sol-RL project page, "Two-Stage Pipeline",
//    Stage 2).  Pass 1 merges and reduces amax|W'| into one fp32; pass 2 merges
//    again and quantizes; a one-thread kernel turns amax into s_t.
//
// Arithmetic follows the library's NVFP4 convention exactly (every scale step an
// IEEE fp32 operation); the quotient helpers in common.cuh make the per-element
// divisions cheap without changing any result.
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
    x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
    x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float absmax8(const float (&x)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    return m;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Byte offset of the 4-byte scale word holding K-blocks kb..kb+3 (kb % 4 == 0) of
// `row` in the 128x4 blocked scale layout.
__device__ __forceinline__ int64_t sf_word_offset(int64_t row, int64_t kb, int64_t K) {
    return ((row >> 7) * (K >> 6) + (kb >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// Quantizes 8 consecutive elements x of a 16-element block whose other half is
// held by the partner lane (lane ^ 1).  s is the second-level scale, d = 6*s and
// inv_d within 1 ulp of 1/d (when d_fast).  Returns the 8 packed codes; *sfc gets the
// block's E4M3 scale code.  Every lane of the warp must call it (shuffle).
__device__ __forceinline__ uint32_t quant_half_block(const float (&x)[8], float s, float d,
                                                     float inv_d, bool d_fast, uint32_t* sfc) {
    const float pm = absmax8(x);
    const float bamax = fmaxf(pm, __shfl_xor_sync(kFull, pm, 1));
    uint32_t code = 0;
    if (d > 0.0f) code = e4m3_quotient(bamax, d, inv_d, d_fast);
    *sfc = code;
    const float den = __fmul_rn(e4m3_value(code), s);
    if (!(den > 0.0f)) return 0u;
    const bool fast = fast_recip_ok(den);
    return e2m1_quotient8(x, den, fast ? recip_approx(den) : 0.0f, fast);
}

// Gathers the scale codes of 4 consecutive blocks held by lanes l, l+2, l+4, l+6
// (l % 8 == 0) into one little-endian word (valid in lane l).
__device__ __forceinline__ uint32_t gather_sf_word(uint32_t sfc) {
    const uint32_t s2 = __shfl_down_sync(kFull, sfc, 2);
    const uint32_t s4 = __shfl_down_sync(kFull, sfc, 4);
    const uint32_t s6 = __shfl_down_sync(kFull, sfc, 6);
    return sfc | (s2 << 8) | (s4 << 16) | (s6 << 24);
}

// ------------------------------------------------------------------ act_quant

// Persistent, several 8-warp CTAs per SM.  Warps form groups of G (32 G threads per
// row); each group owns a ring of kAqRing row buffers in shared memory that one lane
// fills with bulk copies (kAqRing rows ahead; a shallow ring keeps more CTAs per SM,
// which measured faster than a deeper one), so HBM streams while the group
// quantizes earlier rows from shared memory.  One lane per 16-element block:
//   pass 1: block maxima on packed bf16 pairs (kept in registers), row amax (warp
//           shuffles, then shared memory across the group's warps);
//   pass 2: the block's E4M3 scale, its 16 E2M1 codes (8 bytes), and one scale
//           word per 4 blocks.
// Rows M..rows_pad-1 are scale padding: their scale words are written as 0.
constexpr int kAqWarps = 8;
constexpr int kAqRing = 2;
constexpr int kAqMaxBpt = 8;  // 16-element blocks per thread (K <= 4096 * G)

__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w) {
    // Max of magnitudes, lane-wise on two bf16 values: clearing the sign bits makes the
    // bit patterns order like the magnitudes, so an unsigned 16-bit max is exact.
    return __vmaxu2(m, w & 0x7FFF7FFFu);
}

template <int G>
__global__ void __launch_bounds__(kAqWarps * 32)
    act_quant_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t K, int64_t rows_pad,
                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                     float* __restrict__ s_row, int* status) {
    constexpr int kGroups = kAqWarps / G;
    constexpr int kThreadsPerRow = 32 * G;
    extern __shared__ __align__(128) uint8_t aq_smem[];
    __shared__ uint64_t full[kGroups][kAqRing];
    __shared__ float red[kAqWarps];
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int group = warp / G;
    const int t = threadIdx.x % kThreadsPerRow;  // thread within the row group
    const int nblk = (int)(K >> 4);
    const uint32_t row_bytes = (uint32_t)(K * 2);
    uint8_t* ring = aq_smem + (size_t)group * kAqRing * row_bytes;
    const int64_t first = (int64_t)blockIdx.x * kGroups + group;
    const int64_t step = (int64_t)gridDim.x * kGroups;

    if (threadIdx.x == 0) abort_flag = 0;
    if (t == 0)
        for (int s = 0; s < kAqRing; ++s) mbar_init(&full[group][s], 1);
    fence_barrier_init();
    __syncthreads();

    // Prologue: the first kAqRing rows of this group.
    if (t == 0) {
        for (int s = 0; s < kAqRing; ++s) {
            const int64_t m = first + s * step;
            if (m < M) {
                mbar_arrive_expect_tx(&full[group][s], row_bytes);
                bulk_load(ring + s * row_bytes, X + m * K, row_bytes, &full[group][s]);
            }
        }
    }

    int slot = 0;
    uint32_t phase = 0;
    for (int64_t m = first; m < rows_pad; m += step) {
        const bool valid = m < M;
        const uint4* srow = reinterpret_cast<const uint4*>(ring + slot * row_bytes);
        if (valid) {
            bool ok = mbar_wait(&full[group][slot], phase, status, &abort_flag, 4000000000ull);
            ok = __all_sync(kFull, ok);
            if (!ok) break;
        }
        // Pass 1: block maxima and the row amax.
        float bmax[kAqMaxBpt];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kAqMaxBpt; ++i) {
            const int b = t + i * kThreadsPerRow;
            float bm = 0.0f;
            if (valid && b < nblk) {
                const uint4 u0 = srow[2 * b], u1 = srow[2 * b + 1];
                uint32_t mm = bf16x2_absmax(0u, u0.x);
                mm = bf16x2_absmax(mm, u0.y);
                mm = bf16x2_absmax(mm, u0.z);
                mm = bf16x2_absmax(mm, u0.w);
                mm = bf16x2_absmax(mm, u1.x);
                mm = bf16x2_absmax(mm, u1.y);
                mm = bf16x2_absmax(mm, u1.z);
                mm = bf16x2_absmax(mm, u1.w);
                bm = fmaxf(bf16_lo(mm), bf16_hi(mm));
            }
            bmax[i] = bm;
            amax = fmaxf(amax, bm);
        }
        amax = warp_max(amax);
        if (G > 1) {
            if (lane == 0) red[warp] = amax;
            named_barrier_sync(1 + group, kThreadsPerRow);
#pragma unroll
            for (int w = 0; w < G; ++w) amax = fmaxf(amax, red[group * G + w]);
        }
        const float s = __fdiv_rn(amax, kAmaxDiv);
        if (valid && t == 0) s_row[m] = s;
        const float d = __fmul_rn(6.0f, s);
        const bool d_fast = fast_recip_ok(d);
        const float inv_d = d_fast ? recip_approx(d) : 0.0f;

        // Pass 2: one block per lane.
        uint2* crow = reinterpret_cast<uint2*>(codes + (valid ? m : 0) * (K >> 1));
#pragma unroll
        for (int i = 0; i < kAqMaxBpt; ++i) {
            if (i * kThreadsPerRow >= nblk) break;  // uniform across the warp
            const int b = t + i * kThreadsPerRow;
            const bool have = b < nblk;
            uint32_t sfc = 0;
            if (d > 0.0f) sfc = e4m3_quotient(bmax[i], d, inv_d, d_fast);
            const float den = __fmul_rn(e4m3_value(sfc), s);
            uint2 packed = make_uint2(0u, 0u);
            if (valid && have && den > 0.0f) {
                const bool fast = fast_recip_ok(den);
                const float r = fast ? recip_approx(den) : 0.0f;
                float x[8];
                unpack8(srow[2 * b], x);
                packed.x = e2m1_quotient8(x, den, r, fast);
                unpack8(srow[2 * b + 1], x);
                packed.y = e2m1_quotient8(x, den, r, fast);
            }
            // Scale codes of blocks b..b+3 (lanes l..l+3, l % 4 == 0) -> one word.
            const uint32_t s1 = __shfl_down_sync(kFull, sfc, 1);
            const uint32_t s2 = __shfl_down_sync(kFull, sfc, 2);
            const uint32_t s3 = __shfl_down_sync(kFull, sfc, 3);
            if (have) {
                if (valid) crow[b] = packed;
                if ((b & 3) == 0)
                    *reinterpret_cast<uint32_t*>(sf + sf_word_offset(m, b, K)) =
                        sfc | (s1 << 8) | (s2 << 16) | (s3 << 24);
            }
        }

        // Every thread of the group is done with this slot: refill it kAqRing rows ahead.
        if (G > 1) named_barrier_sync(1 + group, kThreadsPerRow);
        else __syncwarp();
        if (t == 0) {
            const int64_t next = m + kAqRing * step;
            if (next < M) {
                mbar_arrive_expect_tx(&full[group][slot], row_bytes);
                bulk_load(ring + slot * row_bytes, X + next * K, row_bytes, &full[group][slot]);
            }
        }
        if (valid) {
            if (++slot == kAqRing) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
    // After an abort, give copies already issued time to land before the CTA exits.
    if (abort_flag && t == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
}

template <int G>
cudaError_t run_act_quant(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                          int64_t rows_pad, uint8_t* codes, uint8_t* sf, float* s_row) {
    const size_t smem = (size_t)(kAqWarps / G) * kAqRing * (size_t)K * 2;
    cudaError_t e = cudaFuncSetAttribute(act_quant_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, act_quant_kernel<G>, kAqWarps * 32,
                                                      smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (rows_pad + (kAqWarps / G) - 1) / (kAqWarps / G);
    if (grid > (int64_t)ctx.num_sms * per_sm) grid = (int64_t)ctx.num_sms * per_sm;
    act_quant_kernel<G><<<(unsigned)grid, kAqWarps * 32, smem, ctx.stream>>>(X, M, K, rows_pad, codes,
                                                                          sf, s_row, ctx.status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ requant

// CTA tile: 64 rows x 128 columns of W; thread tile 4 rows x 8 columns.  Lane
// l of warp w owns column group cg = l % 16 and row group rg = 2w + l / 16.
constexpr int kRqRows = 64;
constexpr int kRqCols = 128;

struct RqArgs {
    const void* W;
    const float* A;
    const float* B;
    int r;
    float c;
    int64_t N, K, rows_pad;
    uint8_t* codes;
    uint8_t* sf;
    float* s_t;
};

// Merged values w'[4][8] of this thread's tile, per the library's merge order:
// acc = +0; acc = fma(B[n,j], A[j,k], acc) for j = 0..r-1; w' = fma(c, acc, W).
template <int kWType>
__device__ __forceinline__ void merge_tile(const RqArgs& a, const float* As, const float* Bs,
                                           int64_t n0, int64_t k0, bool col_ok,
                                           float (&w)[4][8]) {
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    const int cg = threadIdx.x & 15;
    const int rg = threadIdx.x >> 4;
    if (a.r > 0) {
#pragma unroll 4
        for (int j = 0; j < a.r; ++j) {
            const float4 a0 = *reinterpret_cast<const float4*>(As + j * kRqCols + cg * 8);
            const float4 a1 = *reinterpret_cast<const float4*>(As + j * kRqCols + cg * 8 + 4);
            const float4 b = *reinterpret_cast<const float4*>(Bs + j * kRqRows + rg * 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[i][q] = __fmaf_rn(bv[i], av[q], acc[i][q]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = n0 + rg * 4 + i;
        float wv[8];
        if (n < a.N && col_ok) {
            if (kWType == NVFP4_W_BF16) {
                const uint4 raw = ld_stream_v4(static_cast<const __nv_bfloat16*>(a.W) + n * a.K +
                                               k0 + cg * 8);
                unpack8(raw, wv);
            } else {
                const float* p = static_cast<const float*>(a.W) + n * a.K + k0 + cg * 8;
                const uint4 r0 = ld_stream_v4(p);
                const uint4 r1 = ld_stream_v4(p + 4);
                wv[0] = __uint_as_float(r0.x); wv[1] = __uint_as_float(r0.y);
                wv[2] = __uint_as_float(r0.z); wv[3] = __uint_as_float(r0.w);
                wv[4] = __uint_as_float(r1.x); wv[5] = __uint_as_float(r1.y);
                wv[6] = __uint_as_float(r1.z); wv[7] = __uint_as_float(r1.w);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) wv[q] = 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) w[i][q] = (a.r > 0) ? __fmaf_rn(a.c, acc[i][q], wv[q]) : wv[q];
    }
}

// Stages A[:, k0:k0+128] as As[j][col] and B[n0:n0+64, :]^T as Bs[j][row].
__device__ __forceinline__ void stage_lora(const RqArgs& a, float* As, float* Bs, int64_t n0,
                                           int64_t k0) {
    const int tid = threadIdx.x;
    for (int e = tid; e < a.r * (kRqCols / 4); e += 256) {
        const int j = e / (kRqCols / 4), c4 = e % (kRqCols / 4);
        const int64_t k = k0 + c4 * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < a.K) v = *reinterpret_cast<const float4*>(a.A + (int64_t)j * a.K + k);
        *reinterpret_cast<float4*>(As + j * kRqCols + c4 * 4) = v;
    }
    for (int e = tid; e < a.r * kRqRows; e += 256) {
        const int row = e % kRqRows, j = e / kRqRows;
        const int64_t n = n0 + row;
        Bs[j * kRqRows + row] = (n < a.N) ? a.B[n * a.r + j] : 0.0f;
    }
}

template <int kWType>
__global__ void __launch_bounds__(256) requant_amax_kernel(RqArgs a) {
    extern __shared__ float smem[];
    float* As = smem;
    float* Bs = smem + a.r * kRqCols;
    __shared__ float red[8];
    const int64_t n0 = (int64_t)blockIdx.x * kRqRows;
    const int64_t k0 = (int64_t)blockIdx.y * kRqCols;
    if (a.r > 0) {
        stage_lora(a, As, Bs, n0, k0);
        __syncthreads();
    }
    const bool col_ok = k0 + (threadIdx.x & 15) * 8 < a.K;
    float w[4][8];
    merge_tile<kWType>(a, As, Bs, n0, k0, col_ok, w);
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(w[i][q]));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) b = fmaxf(b, red[i]);
        // |w'| >= 0, so the fp32 bit patterns order like the values.
        atomicMax(reinterpret_cast<unsigned int*>(a.s_t), __float_as_uint(b));
    }
}

template <int kWType>
__global__ void __launch_bounds__(256) requant_quant_kernel(RqArgs a) {
    extern __shared__ float smem[];
    float* As = smem;
    float* Bs = smem + a.r * kRqCols;
    const int64_t n0 = (int64_t)blockIdx.x * kRqRows;
    const int64_t k0 = (int64_t)blockIdx.y * kRqCols;
    const float amax = *reinterpret_cast<volatile const float*>(a.s_t);
    if (a.r > 0) {
        stage_lora(a, As, Bs, n0, k0);
        __syncthreads();
    }
    const int cg = threadIdx.x & 15;
    const int rg = threadIdx.x >> 4;
    const bool col_ok = k0 + cg * 8 < a.K;
    float w[4][8];
    merge_tile<kWType>(a, As, Bs, n0, k0, col_ok, w);

    const float s = __fdiv_rn(amax, kAmaxDiv);
    const float d = __fmul_rn(6.0f, s);
    const bool d_fast = fast_recip_ok(d);
    const float inv_d = d_fast ? recip_approx(d) : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = n0 + rg * 4 + i;
        uint32_t sfc;
        const uint32_t packed = quant_half_block(w[i], s, d, inv_d, d_fast, &sfc);
        const uint32_t word = gather_sf_word(sfc);
        if (col_ok) {
            if (n < a.N)
                *reinterpret_cast<uint32_t*>(a.codes + n * (a.K >> 1) + ((k0 + cg * 8) >> 1)) =
                    packed;
            if (n < a.rows_pad && (cg & 7) == 0)
                *reinterpret_cast<uint32_t*>(a.sf + sf_word_offset(n, (k0 + cg * 8) >> 4, a.K)) =
                    word;
        }
    }
}

__global__ void requant_finalize_kernel(float* s_t) {
    if (threadIdx.x == 0 && blockIdx.x == 0) *s_t = __fdiv_rn(*s_t, kAmaxDiv);
}

template <int kWType>
cudaError_t run_requant(const LaunchCtx& ctx, const RqArgs& a) {
    const dim3 grid((unsigned)((a.rows_pad + kRqRows - 1) / kRqRows),
                    (unsigned)((a.K + kRqCols - 1) / kRqCols));
    const size_t smem = (size_t)a.r * (kRqCols + kRqRows) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(requant_amax_kernel<kWType>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(requant_quant_kernel<kWType>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.s_t, 0, sizeof(float), ctx.stream);
    if (e != cudaSuccess) return e;
    requant_amax_kernel<kWType><<<grid, 256, smem, ctx.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    requant_quant_kernel<kWType><<<grid, 256, smem, ctx.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    requant_finalize_kernel<<<1, 32, 0, ctx.stream>>>(a.s_t);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ test hooks

__global__ void test_e2m1_kernel(const float* q, uint8_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(cvt_e2m1x8(q[i], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu);
}

__global__ void test_e4m3_kernel(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)cvt_e4m3(v[i]);
}

__global__ void test_e2m1_quotient_kernel(const float* x, const float* den, uint8_t* out,
                                          int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float dn = den[i];
        const bool fast = fast_recip_ok(dn);
        const float r = fast ? recip_approx(dn) : 0.0f;
        const float xs[8] = {x[i], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        out[i] = (uint8_t)(e2m1_quotient8(xs, dn, r, fast) & 0xFu);
    }
}

__global__ void test_e4m3_quotient_kernel(const float* v, const float* d, uint8_t* out,
                                          int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float dd = d[i];
        const bool fast = fast_recip_ok(dd);
        out[i] = (uint8_t)e4m3_quotient(v[i], dd, fast ? recip_approx(dd) : 0.0f, fast);
    }
}

unsigned grid_for(int64_t n, const LaunchCtx& ctx) {
    int64_t g = (n + 255) / 256;
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_act_quant(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                             uint8_t* codes, uint8_t* sf, float* s_row) {
    const int64_t rows_pad = (M + 127) / 128 * 128;
    // G warps per row: at most 4 blocks of 16 elements per thread up to K = 16384 (a
    // smaller ring footprint per CTA, so more CTAs per SM), 8 beyond.
    if (K <= 2048) return run_act_quant<1>(ctx, X, M, K, rows_pad, codes, sf, s_row);
    if (K <= 4096) return run_act_quant<2>(ctx, X, M, K, rows_pad, codes, sf, s_row);
    if (K <= 8192) return run_act_quant<4>(ctx, X, M, K, rows_pad, codes, sf, s_row);
    return run_act_quant<8>(ctx, X, M, K, rows_pad, codes, sf, s_row);
}

cudaError_t launch_requant(const LaunchCtx& ctx, const void* W, int w_dtype, const float* A,
                           const float* B, int r, float c, int64_t N, int64_t K, uint8_t* codes,
                           uint8_t* sf, float* s_t) {
    RqArgs a;
    a.W = W;
    a.A = A;
    a.B = B;
    a.r = r;
    a.c = c;
    a.N = N;
    a.K = K;
    a.rows_pad = (N + 127) / 128 * 128;
    a.codes = codes;
    a.sf = sf;
    a.s_t = s_t;
    return w_dtype == NVFP4_W_BF16 ? run_requant<NVFP4_W_BF16>(ctx, a)
                                   : run_requant<NVFP4_W_FP32>(ctx, a);
}

cudaError_t launch_test_e2m1(const LaunchCtx& ctx, const float* q, uint8_t* codes, int64_t n) {
    test_e2m1_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(q, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_test_e4m3(const LaunchCtx& ctx, const float* v, uint8_t* codes, int64_t n) {
    test_e4m3_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(v, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_test_e2m1_quotient(const LaunchCtx& ctx, const float* x, const float* den,
                                      uint8_t* codes, int64_t n) {
    test_e2m1_quotient_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(x, den, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_test_e4m3_quotient(const LaunchCtx& ctx, const float* v, const float* d,
                                      uint8_t* codes, int64_t n) {
    test_e4m3_quotient_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(v, d, codes, n);
    return cudaGetLastError();
}

}  // namespace nvfp4rl
