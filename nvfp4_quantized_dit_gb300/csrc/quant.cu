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
    return e2m1_quotient8(x, den, make_recip(den));
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
// row, G as small as 8 blocks per thread allows); each group owns kAqRing row buffers
// in shared memory that one lane fills with bulk copies.  A single buffer per group
// measured fastest: shared memory then holds the most groups per SM, and HBM streams
// while the other groups quantize their rows.  One lane per 16-element block:
//   pass 1: block maxima on packed bf16 pairs (kept in registers), row amax (warp
//           shuffles, then shared memory across the group's warps);
//   pass 2: the block's E4M3 scale, its 16 E2M1 codes (8 bytes), and one scale
//           word per 4 blocks.
// Rows M..rows_pad-1 are scale padding: their scale words are written as 0.
constexpr int kAqWarps = 8;
constexpr int kAqRing = 1;
constexpr int kAqMaxBpt = 8;  // 16-element blocks per thread (K <= 4096 * G)

__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w) {
    // Max of magnitudes, lane-wise on two bf16 values: clearing the sign bits makes the
    // bit patterns order like the magnitudes, so an unsigned 16-bit max is exact.
    return __vmaxu2(m, w & 0x7FFF7FFFu);
}

// Lane-wise magnitudes of two bf16 values.
__device__ __forceinline__ __nv_bfloat162 bf16x2_abs(uint32_t w) {
    return __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// Largest magnitude in each half of 16 bf16 values (8 words), as a bf16 pair; exact
// for finite inputs.
__device__ __forceinline__ uint32_t bf16x16_absmax(const uint4& u0, const uint4& u1) {
    const __nv_bfloat162 m01 = __hmax2(bf16x2_abs(u0.x), bf16x2_abs(u0.y));
    const __nv_bfloat162 m23 = __hmax2(bf16x2_abs(u0.z), bf16x2_abs(u0.w));
    const __nv_bfloat162 m45 = __hmax2(bf16x2_abs(u1.x), bf16x2_abs(u1.y));
    const __nv_bfloat162 m67 = __hmax2(bf16x2_abs(u1.z), bf16x2_abs(u1.w));
    const __nv_bfloat162 m = __hmax2(__hmax2(m01, m23), __hmax2(m45, m67));
    return *reinterpret_cast<const uint32_t*>(&m);
}

// kMode: how s is found.  kAqReduce: s = amax(|X[m,:]|) / 2688 from the row itself
// (pass 1 below), written to s_row[m].  kAqGivenRow: the row's amax is read from
// amax_in[m] (e.g. reduced by the epilogue of the GEMM that produced X), s written to
// s_row[m].  kAqGivenTensor: one amax for the whole tensor, amax_in[0]; nothing is
// written to s_row.
// kBpt > 0: every thread has exactly kBpt blocks (K == 512 G kBpt), so the block
// loops have fixed trip counts (no per-block bounds or exit tests, chains of
// consecutive blocks interleaved); 0: any K, blocks counted at run time.
enum { kAqReduce = 0, kAqGivenRow = 1, kAqGivenTensor = 2 };
template <int G, int kMode, int kBpt>
__global__ void __launch_bounds__(kAqWarps * 32)
    act_quant_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t K, int64_t rows_pad,
                     const float* __restrict__ amax_in, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
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

    const float s_all = kMode == kAqGivenTensor ? __fdiv_rn(__ldg(amax_in), kAmaxDiv) : 0.0f;
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
        constexpr int kB = kBpt > 0 ? kBpt : kAqMaxBpt;
        float bmax[kB];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            const int b = t + i * kThreadsPerRow;
            float bm = 0.0f;
            if (valid && (kBpt > 0 || b < nblk)) {
                const uint32_t mm = bf16x16_absmax(srow[2 * b], srow[2 * b + 1]);
                bm = fmaxf(bf16_lo(mm), bf16_hi(mm));
            }
            bmax[i] = bm;
            amax = fmaxf(amax, bm);
        }
        float s = s_all;
        if (kMode == kAqReduce) {
            amax = warp_max(amax);
            if (G > 1) {
                if (lane == 0) red[warp] = amax;
                named_barrier_sync(1 + group, kThreadsPerRow);
#pragma unroll
                for (int w = 0; w < G; ++w) amax = fmaxf(amax, red[group * G + w]);
            }
            s = __fdiv_rn(amax, kAmaxDiv);
        } else if (kMode == kAqGivenRow) {
            s = valid ? __fdiv_rn(__ldg(amax_in + m), kAmaxDiv) : 0.0f;
        }
        if (kMode != kAqGivenTensor && valid && t == 0) s_row[m] = s;
        const float d = __fmul_rn(6.0f, s);
        const bool d_fast = fast_recip_ok(d);
        const float inv_d = d_fast ? recip_approx(d) : 0.0f;

        // Pass 2: one block per lane.
        uint2* crow = reinterpret_cast<uint2*>(codes + (valid ? m : 0) * (K >> 1));
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            if (kBpt == 0 && i * kThreadsPerRow >= nblk) break;  // uniform across the warp
            const int b = t + i * kThreadsPerRow;
            const bool have = kBpt > 0 || b < nblk;
            uint32_t sfc = 0;
            if (d > 0.0f) sfc = e4m3_quotient(bmax[i], d, inv_d, d_fast);
            const float den = __fmul_rn(e4m3_value(sfc), s);
            uint2 packed = make_uint2(0u, 0u);
            if (valid && have && den > 0.0f) {
                const Recip rc = make_recip(den);
                float x[8];
                unpack8(srow[2 * b], x);
                packed.x = e2m1_quotient8(x, den, rc);
                unpack8(srow[2 * b + 1], x);
                packed.y = e2m1_quotient8(x, den, rc);
            }
            // One scale byte per lane: lanes l..l+3 (l % 4 == 0) fill one 4-byte word.
            if (have) {
                if (valid) crow[b] = packed;
                sf[sf_word_offset(m, b, K) + (b & 3)] = (uint8_t)sfc;
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

template <int G, int kMode, int kBpt = 0>
cudaError_t run_act_quant(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                          int64_t rows_pad, const float* amax_in, uint8_t* codes, uint8_t* sf, float* s_row) {
    const size_t smem = (size_t)(kAqWarps / G) * kAqRing * (size_t)K * 2;
    static OccupancyCache occupancy;
    int per_sm = 0;
    const cudaError_t e =
        blocks_per_sm(occupancy, ctx, act_quant_kernel<G, kMode, kBpt>, kAqWarps * 32, smem, &per_sm);
    if (e != cudaSuccess) return e;
    int64_t grid = (rows_pad + (kAqWarps / G) - 1) / (kAqWarps / G);
    if (grid > (int64_t)ctx.num_sms * per_sm) grid = (int64_t)ctx.num_sms * per_sm;
    act_quant_kernel<G, kMode, kBpt><<<(unsigned)grid, kAqWarps * 32, smem, ctx.stream>>>(
        X, M, K, rows_pad, amax_in, codes, sf, s_row, ctx.status);
    return cudaGetLastError();
}

// Per-tensor activation scale, pass 1: amax|X| over the whole tensor into *amax (fp32
// bits, atomicMax: every value is >= 0, so the bit patterns order like the values;
// zeroed before the launch).  Streaming loads, 4 in flight per thread.
constexpr int kAmaxThreads = 256;
__global__ void __launch_bounds__(kAmaxThreads) act_amax_kernel(const uint4* __restrict__ X, int64_t n_vec,
                                                                float* __restrict__ amax) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    __nv_bfloat162 m = __float2bfloat162_rn(0.0f);
    for (; i + 3 * stride < n_vec; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_stream_v4(X + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            m = __hmax2(m, __hmax2(__hmax2(bf16x2_abs(v[u].x), bf16x2_abs(v[u].y)),
                                   __hmax2(bf16x2_abs(v[u].z), bf16x2_abs(v[u].w))));
    }
    for (; i < n_vec; i += stride) {
        const uint4 v = ld_stream_v4(X + i);
        m = __hmax2(m, __hmax2(__hmax2(bf16x2_abs(v.x), bf16x2_abs(v.y)),
                               __hmax2(bf16x2_abs(v.z), bf16x2_abs(v.w))));
    }
    const uint32_t mm = *reinterpret_cast<const uint32_t*>(&m);
    const float f = warp_max(fmaxf(bf16_lo(mm), bf16_hi(mm)));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(f));
}

// Per-tensor activation scale, last step: *s_t = amax / 2688 (fp32).
__global__ void act_scale_kernel(float* s_t) { *s_t = __fdiv_rn(*s_t, kAmaxDiv); }

// ------------------------------------------------------------------ requant
//
// Both kernels walk the same tiles: kRqRows x kRqCols pieces of W in strip-major
// order (a strip is kRqCols columns), each CTA a contiguous run of tiles, so a CTA
// stages the r x kRqCols strip of A in shared memory about once.  Warp w owns rows
// 16 (w / 2) .. +15 and columns 64 (w % 2) .. +63 of a tile; lane l owns the 4
// consecutive rows 4 (l / 8) .. +3 of that block and the 8 columns 8 (l % 8) .. +7,
// so the 16-element scale block of a row lives in lanes l, l ^ 1 and one scale word
// (4 blocks) in 8 consecutive lanes.
//
// Shared memory holds the operands of the packed fp32 fma (fma.rn.f32x2, an IEEE fma
// in each half) in the pairs it consumes, so that no register moves are needed:
//   As2  A strip, each value twice: piece t of lane group g (4 floats) holds columns
//        8 g + 2 t and 8 g + 2 t + 1 of its 64, as {a, a, a', a'}; the 8 pieces a load
//        instruction touches (one per g) are contiguous (no bank conflicts).
//   Bs   per warp, double-buffered one tile ahead: its 16 rows of B as copied
//        (row-major, row stride rs = r rounded up to 4, plus 4);
//   Bt   per warp (pass 2): the same rows transposed, Bt[j][row] with a stride of
//        20 floats per j, so one 16-byte load gives a lane its 4 rows at step j.
constexpr int kRqRows = 64;
constexpr int kRqCols = 128;
constexpr int kRqThreads = 256;
constexpr int kRqWarps = kRqThreads / 32;
constexpr int kRqMaxR = 64;
constexpr int kRqA2 = 2 * kRqCols;  // floats per row of As2

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
    float* dump;  // test hook: merged values instead of codes
    int64_t row_tiles, tiles;    // pass 1: kRqRows-row tiles
    int64_t row_tiles2, tiles2;  // pass 2: kQRows-row tiles
    int rs;     // row stride of Bs (floats)
    int inv_r;  // ceil(2^16 / r): x / r == (x * inv_r) >> 16 for 0 <= x < 16 r
    int b_vec;  // B 16-byte aligned and r % 4 == 0: 16-byte copies
};

constexpr int kRqBtStride = 20;

__host__ __device__ constexpr int rq_bstride(int r) { return ((r + 3) & ~3) + 4; }

__host__ __device__ constexpr int rq_inv_r(int r) { return r > 0 ? (65536 + r - 1) / r : 0; }

// The multiply-shift quotient is exact for every index a B copy uses.
constexpr bool rq_inv_r_exact() {
    for (int r = 1; r <= kRqMaxR; ++r)
        for (int x = 0; x < 16 * r; ++x)
            if (((x * rq_inv_r(r)) >> 16) != x / r) return false;
    return true;
}
static_assert(rq_inv_r_exact(), "x * ceil(2^16 / r) >> 16 must equal x / r for x < 16 r");

// Per warp: Bs double buffer, then Bt (rows of j rounded up to 8).
__host__ __device__ constexpr int rq_warp_floats(int r) {
    return 2 * 16 * rq_bstride(r) + ((r + 7) & ~7) * kRqBtStride;
}

__host__ __device__ inline size_t rq_smem_bytes(int r) {
    return ((size_t)r * kRqA2 + (size_t)kRqWarps * rq_warp_floats(r)) * sizeof(float);
}

struct RqLane {
    int warp, lane, wr, wc, cg, rg;
    __device__ __forceinline__ RqLane() {
        warp = threadIdx.x >> 5;
        lane = threadIdx.x & 31;
        wr = warp >> 1;
        wc = warp & 1;
        cg = lane & 7;
        rg = lane >> 3;
    }
    // Tile-local row of this lane's row i, and the warp-slice row of B it reads.
    __device__ __forceinline__ int row(int i) const { return wr * 16 + rg * 4 + i; }
    __device__ __forceinline__ int brow(int i) const { return rg * 4 + i; }
    __device__ __forceinline__ int col() const { return wc * 64 + cg * 8; }
};

// Float index within an As2 row of column q (0..7) of lane group g in col-warp wc.
__device__ __forceinline__ int rq_a2_index(int wc, int g, int q) {
    return wc * 128 + ((q >> 1) * 8 + g) * 4 + 2 * (q & 1);
}

// Position in the strip-major tile order (tiles of `rows` rows, row_tiles per
// strip), advanced one tile at a time.
struct RqCursor {
    int64_t strip, rt, row_tiles;
    int rows;
    __device__ __forceinline__ void init(int64_t row_tiles_, int rows_, int64_t t) {
        row_tiles = row_tiles_;
        rows = rows_;
        strip = t / row_tiles;
        rt = t - strip * row_tiles;
    }
    __device__ __forceinline__ void next() {
        if (++rt == row_tiles) {
            rt = 0;
            ++strip;
        }
    }
    __device__ __forceinline__ int64_t n0() const { return rt * rows; }
    __device__ __forceinline__ int64_t k0() const { return strip * kRqCols; }
};

// A[:, k0:k0+kRqCols] -> As2 (zero past K).  Called by the whole CTA.
__device__ __forceinline__ void rq_stage_a(const RqArgs& a, float* As2, int64_t k0) {
    // Thread e: row j, columns 8 g + 2 t, +1 of col-warp wc (one 4-float piece).
    for (int e = threadIdx.x; e < a.r * (kRqCols / 2); e += kRqThreads) {
        const int j = e / (kRqCols / 2), pc = e % (kRqCols / 2);
        const int wc = pc >> 5, g = (pc >> 2) & 7, t = pc & 3;
        const int64_t k = k0 + wc * 64 + g * 8 + 2 * t;
        float2 v = make_float2(0.f, 0.f);
        if (k < a.K) v = *reinterpret_cast<const float2*>(a.A + (int64_t)j * a.K + k);
        *reinterpret_cast<float4*>(As2 + j * kRqA2 + wc * 128 + (t * 8 + g) * 4) =
            make_float4(v.x, v.x, v.y, v.y);
    }
}

// Asynchronous copies of B[row0 : row0+16, :] (the warp's rows; rows past N are
// zero-filled) into Bs with row stride rs: 16-byte pieces when B allows, else 4-byte
// ones.  One commit group.
__device__ __forceinline__ void rq_copy_b(const RqArgs& a, int lane, int64_t row0, float* Bs) {
    if (a.b_vec) {
        for (int c = lane; c < 4 * a.r; c += 32) {
            const int x = 4 * c;
            const int rl = (x * a.inv_r) >> 16, j = x - rl * a.r;
            const bool valid = row0 + rl < a.N;
            const float* src = a.B + (valid ? (row0 + rl) * a.r + j : 0);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                             smem_u32(Bs + rl * a.rs + j)),
                         "l"(src), "r"(valid ? 16 : 0)
                         : "memory");
        }
    } else {
        for (int x = lane; x < 16 * a.r; x += 32) {
            const int rl = (x * a.inv_r) >> 16, j = x - rl * a.r;
            const bool valid = row0 + rl < a.N;
            const float* src = a.B + (valid ? (row0 + rl) * a.r + j : 0);
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                             smem_u32(Bs + rl * a.rs + j)),
                         "l"(src), "r"(valid ? 4 : 0)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void rq_commit_empty() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most one of this lane's copy groups is pending, then makes the
// warp's copies visible to the whole warp.
__device__ __forceinline__ void rq_wait_b() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncwarp();
}

// W rows of this lane for one tile, as raw 16-byte words (bf16: one per row; fp32: two).
template <int kWType>
struct RqW {
    static constexpr int kWords = kWType == NVFP4_W_BF16 ? 1 : 2;
    uint4 v[4][kWords];

    template <bool kEdge>
    __device__ __forceinline__ void load(const RqArgs& a, const RqLane& L, int64_t n0, int64_t k0) {
        const int64_t k = k0 + L.col();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t n = n0 + L.row(i);
            const bool ok = !kEdge || (n < a.N && k < a.K);
#pragma unroll
            for (int w = 0; w < kWords; ++w) {
                if (ok) {
                    if (kWType == NVFP4_W_BF16)
                        v[i][w] = ld_stream_v4(static_cast<const __nv_bfloat16*>(a.W) + n * a.K + k);
                    else
                        v[i][w] = ld_stream_v4(static_cast<const float*>(a.W) + n * a.K + k + 4 * w);
                } else {
                    v[i][w] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    }

    __device__ __forceinline__ void row(int i, float (&x)[8]) const {
        if (kWType == NVFP4_W_BF16) {
            unpack8(v[i][0], x);
        } else {
            x[0] = __uint_as_float(v[i][0].x); x[1] = __uint_as_float(v[i][0].y);
            x[2] = __uint_as_float(v[i][0].z); x[3] = __uint_as_float(v[i][0].w);
            x[4] = __uint_as_float(v[i][kWords - 1].x); x[5] = __uint_as_float(v[i][kWords - 1].y);
            x[6] = __uint_as_float(v[i][kWords - 1].z); x[7] = __uint_as_float(v[i][kWords - 1].w);
        }
    }

    // Bit 8 i + q set where row i is in `rows` and |W[i][q]| >= t.
    __device__ __forceinline__ unsigned mask_ge(unsigned rows, float t) const {
        unsigned msk = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float x[8];
            row(i, x);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                msk |= (((rows >> i) & 1u) && fabsf(x[q]) >= t) ? 1u << (i * 8 + q) : 0u;
        }
        return msk;
    }

    // Element e = 8 i + q (selects from registers; no local-memory indexing).
    __device__ __forceinline__ float at(int e) const {
        const int i = e >> 3, q = e & 7;
        uint4 lo = v[0][0], hi = v[0][kWords - 1];
#pragma unroll
        for (int k = 1; k < 4; ++k)
            if (i == k) {
                lo = v[k][0];
                hi = v[k][kWords - 1];
            }
        if (kWType == NVFP4_W_BF16) {
            const uint32_t w = (q >> 1) == 0 ? lo.x : (q >> 1) == 1 ? lo.y : (q >> 1) == 2 ? lo.z : lo.w;
            return (q & 1) ? bf16_hi(w) : bf16_lo(w);
        } else {
            const uint4 h = q < 4 ? lo : hi;
            const int qq = q & 3;
            return __uint_as_float(qq == 0 ? h.x : qq == 1 ? h.y : qq == 2 ? h.z : h.w);
        }
    }

    // max |W| over the rows whose bit is set in `rows` (-1 when none).
    __device__ __forceinline__ float absmax(unsigned rows) const {
        if (kWType == NVFP4_W_BF16) {
            uint32_t m = 0;
            bool any = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((rows >> i) & 1u) {
                    any = true;
                    m = bf16x2_absmax(m, v[i][0].x);
                    m = bf16x2_absmax(m, v[i][0].y);
                    m = bf16x2_absmax(m, v[i][0].z);
                    m = bf16x2_absmax(m, v[i][0].w);
                }
            }
            const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
            return any ? __uint_as_float((hi > lo ? hi : lo) << 16) : -1.0f;
        } else {
            float m = -1.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((rows >> i) & 1u) {
                    float x[8];
                    row(i, x);
#pragma unroll
                    for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(x[q]));
                }
            }
            return m;
        }
    }
};

// The merged value of one element, in the library's order: acc = +0;
// acc = fma(B[n,j], A[j,k], acc) for j = 0..r-1; w' = fma(c, acc, W) (w' = W when r = 0).
// brow walks a row of Bs, acol a column of As2 (stride kRqA2).
__device__ __forceinline__ float rq_merge_one(const RqArgs& a, const float* brow, const float* acol,
                                              float w) {
    if (a.r == 0) return w;
    float acc = 0.0f;
#pragma unroll 4
    for (int j = 0; j < a.r; ++j) acc = __fmaf_rn(brow[j], acol[j * kRqA2], acc);
    return __fmaf_rn(a.c, acc, w);
}

// ---- pass 1: exact amax|W'| without merging every element.
//
// For every element, |W'| <= (|W| + D) (1 + 2^-23) + 2^-140 with
// D >= |c| (||B[n,:]||_2 ||A[:,k]||_2 (1 + 2^-17) + 2^-142): Cauchy-Schwarz bounds the
// products' absolute sum, (1 + 2^-24)^r <= 1 + 2^-17 covers the r roundings of the
// fma chain for r <= 64, and the absolute terms cover subnormal results.  A warp keeps
// L, the largest |W'| it has evaluated exactly so far; an element can only raise it
// if |W| >= tau(L, D), a round-down of (L - 2^-140) / (1 + 2^-23) - D, so only those
// elements are merged (exactly, with the same fma chain as pass 2).  The norms are
// upper bounds (sums of squares inflated for their own rounding, square roots
// rounded up), D per warp and tile uses the largest row norm of its 16 rows and the
// largest column norm of its 64 columns, every bound step rounds up (fp32 directed
// rounding).  L is seeded from the exact value at the warp's largest |W| of the tile,
// so typically a few elements per thousand are merged.
__device__ __forceinline__ float rq_norm_ub(float sumsq) {
    return __fsqrt_ru(__fmaf_ru(sumsq, 1.0f + 0x1p-17f, 0x1p-143f));
}

__device__ __forceinline__ float rq_tau(float L, float D) {
    if (!(L > 0x1p-139f)) return -1.0f;
    // (1 - 2^-22) <= 1 / (1 + 2^-23), and every step rounds down.
    return __fsub_rd(__fmul_rd(__fsub_rd(L, 0x1p-140f), 1.0f - 0x1p-22f), D);
}

template <int kWType>
__global__ void __launch_bounds__(kRqThreads, 2) requant_amax_kernel(RqArgs a) {
    extern __shared__ __align__(16) float rq_smem[];
    float* As2 = rq_smem;
    const RqLane L;
    float* Bs0 = rq_smem + a.r * kRqA2 + L.warp * rq_warp_floats(a.r);

    const int64_t t_begin = (int64_t)blockIdx.x * a.tiles / gridDim.x;
    const int64_t t_end = (int64_t)(blockIdx.x + 1) * a.tiles / gridDim.x;
    const float ac = fabsf(a.c);
    int64_t staged = -1;
    float amax_col = 0.0f;  // largest column norm of this warp's 64 columns (upper bound)
    float Lw = 0.0f;        // warp-uniform: largest exact |W'| seen
    RqW<kWType> wcur, wnext;
    RqCursor cur;
    cur.init(a.row_tiles, kRqRows, t_begin);
    if (t_begin < t_end) {
        wcur.template load<true>(a, L, cur.n0(), cur.k0());
        if (a.r > 0) rq_copy_b(a, L.lane, cur.n0() + L.wr * 16, Bs0);
    }
    int buf = 0;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t n0 = cur.n0(), k0 = cur.k0();
        if (cur.strip != staged) {
            __syncthreads();
            rq_stage_a(a, As2, k0);
            __syncthreads();
            staged = cur.strip;
            // Column norms: lane l covers columns 2l, 2l+1 of the warp's 64.
            float m = 0.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int cl = 2 * L.lane + h;
                const float* acol = As2 + rq_a2_index(L.wc, cl >> 3, cl & 7);
                float s2 = 0.0f;
#pragma unroll 4
                for (int j = 0; j < a.r; ++j) s2 = __fmaf_rn(acol[j * kRqA2], acol[j * kRqA2], s2);
                m = fmaxf(m, rq_norm_ub(s2));
            }
            amax_col = warp_max(m);
        }
        __syncwarp();
        cur.next();
        if (t + 1 < t_end) {
            wnext.template load<true>(a, L, cur.n0(), cur.k0());
            if (a.r > 0) rq_copy_b(a, L.lane, cur.n0() + L.wr * 16, Bs0 + (buf ^ 1) * 16 * a.rs);
            else rq_commit_empty();
        } else {
            rq_commit_empty();
        }
        rq_wait_b();
        const float* Bs = Bs0 + buf * 16 * a.rs;
        buf ^= 1;

        const bool col_ok = k0 + L.col() < a.K;
        unsigned rows_ok = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) rows_ok |= (col_ok && n0 + L.row(i) < a.N) ? 1u << i : 0u;
        const float m = wcur.absmax(rows_ok);
        const float wm = warp_max(m);

        float D = 0.0f;
        if (a.r > 0) {
            // Row norms: lanes 2m, 2m+1 share row m of the warp's 16 (halves of j).
            float s2 = 0.0f;
            const float* brow = Bs + (L.lane >> 1) * a.rs;
#pragma unroll 4
            for (int j = L.lane & 1; j < a.r; j += 2) s2 = __fmaf_rn(brow[j], brow[j], s2);
            s2 += __shfl_xor_sync(kFull, s2, 1);  // two sums >= 0: one more rounding
            const float bnorm = warp_max(rq_norm_ub(__fmul_ru(s2, 1.0f + 0x1p-22f)));
            D = __fadd_ru(__fmul_ru(__fmul_ru(__fmul_ru(ac, bnorm), amax_col), 1.0f + 0x1p-16f),
                          __fmul_ru(ac, 0x1p-140f));
        }
        // Only a tile whose largest |W| is within reach of L can raise it.
        if (wm >= 0.0f && wm >= rq_tau(Lw, D)) {
            // Seed: the exact value at the warp's largest |W| (lowest lane holding it).
            const unsigned holders = __ballot_sync(kFull, m == wm);
            int seed = -1;
            float v = 0.0f;
            if (L.lane == __ffs(holders) - 1) {
                seed = __ffs(wcur.mask_ge(rows_ok, m)) - 1;
                v = fabsf(rq_merge_one(a, Bs + L.brow(seed >> 3) * a.rs,
                                       As2 + rq_a2_index(L.wc, L.cg, seed & 7), wcur.at(seed)));
            }
            Lw = fmaxf(Lw, warp_max(v));
            // Then every element that could still exceed L, one merge call site.
            const float tau = rq_tau(Lw, D);
            float lm = 0.0f;
            unsigned cand = m >= tau ? wcur.mask_ge(rows_ok, tau) : 0u;
            if (seed >= 0) cand &= ~(1u << seed);
            while (cand) {
                const int e = __ffs(cand) - 1;
                cand &= cand - 1;
                lm = fmaxf(lm, fabsf(rq_merge_one(a, Bs + L.brow(e >> 3) * a.rs,
                                                  As2 + rq_a2_index(L.wc, L.cg, e & 7), wcur.at(e))));
            }
            Lw = fmaxf(Lw, warp_max(lm));
        }
        wcur = wnext;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // |W'| >= 0, so the fp32 bit patterns order like the values.
    if (L.lane == 0 && Lw > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(a.s_t), __float_as_uint(Lw));
}

// ---- pass 2: merge every element once and quantize it.
//
// The merge is bound by how fast shared memory hands operands to the FMA pipe (a
// lane receives 4 bytes per shared-memory wavefront), so each lane keeps an 8 x 8
// block of accumulators: 16 operands per step j for 64 fmas.  Tiles are
// kQRows x kRqCols; warp w owns rows 32 (w / 2) .. +31 and columns 64 (w % 2) .. +63,
// lane l the rows 8 (l / 8) .. +7 and columns 8 (l % 8) .. +7 of that block.
// Shared memory:
//   As   the A strip, As[j][col] (staged by the whole CTA when the strip changes);
//   Bt   per pair of warps sharing rows, double-buffered one tile ahead: their 32
//        rows of B transposed, element (j, row) at 32 j + (row ^ (j % 32)).  Each
//        copy instruction moves one row (lane = j, a coalesced 128-byte read) into
//        32 distinct banks; a 16-byte load at 32 j + (4 m ^ (j & 28)) returns rows
//        4 m .. 4 m + 3 in the order e ^ (j & 3);
//   Ws   per warp: its 32 x 64 block of W, copied when the tile starts and read by
//        the epilogue, so its latency hides behind the merge.
constexpr int kQRows = 128;

template <int kWType>
struct Rq2Geom {
    static constexpr int kWBytes = kWType == NVFP4_W_BF16 ? 2 : 4;
    static constexpr int kWsFloats = 32 * 64 * kWBytes / 4;  // per warp
};

template <int kWType>
__host__ __device__ inline size_t rq2_smem_bytes(int r) {
    return ((size_t)r * kRqCols + 4 * 2 * (size_t)r * 32 + (size_t)kRqWarps * Rq2Geom<kWType>::kWsFloats) *
           sizeof(float);
}

struct RqScale {
    float s, d, inv_d;
    bool d_fast;
};

// Copies this warp's half (16 rows) of the pair's 32 rows of B, starting at pair row
// 16 h, transposed into Bt.  Lane j copies B[row][j] (and B[row][j + 32] for r > 32).
__device__ __forceinline__ void rq2_copy_b(const RqArgs& a, int lane, int64_t pair_row0, int h,
                                           float* Bt) {
    for (int rr = 16 * h; rr < 16 * h + 16; ++rr) {
        const int64_t n = pair_row0 + rr;
        const bool valid = n < a.N;
        for (int j = lane; j < a.r; j += 32) {
            const float* src = a.B + (valid ? n * a.r + j : 0);
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                             smem_u32(Bt + j * 32 + (rr ^ (j & 31)))),
                         "l"(src), "r"(valid ? 4 : 0)
                         : "memory");
        }
    }
}

// Copies the warp's 32 x 64 block of W (rows n0w.., columns k0w..; zero outside W)
// into Ws, row-major with 64 * kWBytes bytes per row.
template <int kWType>
__device__ __forceinline__ void rq2_copy_w(const RqArgs& a, int lane, int64_t n0w, int64_t k0w,
                                           float* Ws) {
    constexpr int kChunksPerRow = 64 * Rq2Geom<kWType>::kWBytes / 16;
    for (int c = lane; c < 32 * kChunksPerRow; c += 32) {
        const int row = c / kChunksPerRow, pc = c % kChunksPerRow;
        const int64_t n = n0w + row;
        const int64_t k = k0w + pc * (16 / Rq2Geom<kWType>::kWBytes);
        const bool valid = n < a.N && k < a.K;
        const char* src = static_cast<const char*>(a.W) +
                          (valid ? (n * a.K + k) * Rq2Geom<kWType>::kWBytes : 0);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         smem_u32(reinterpret_cast<char*>(Ws) + c * 16)),
                     "l"(src), "r"(valid ? 16 : 0)
                     : "memory");
    }
}

template <int kWType>
__device__ __forceinline__ void rq2_w_row(const float* Ws, int row, int cg, float (&x)[8]) {
    if (kWType == NVFP4_W_BF16) {
        const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(Ws) + row * 128 + cg * 16);
        unpack8(v, x);
    } else {
        const float4 v0 = *reinterpret_cast<const float4*>(Ws + row * 64 + cg * 8);
        const float4 v1 = *reinterpret_cast<const float4*>(Ws + row * 64 + cg * 8 + 4);
        x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
        x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
    }
}

// One merged row (8 columns) -> codes (at cp) and its scale word (at sp, written by
// lane group 0 of the word), or the merged values (kDump, at dp).
template <bool kEdge, bool kDump>
__device__ __forceinline__ void rq2_emit_row(const RqScale& sc, int cg, bool row_ok, bool col_ok,
                                             uint8_t* cp, uint8_t* sp, float* dp, float (&x)[8]) {
    if (kDump) {
        if (col_ok && row_ok) {
            *reinterpret_cast<float4*>(dp) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(dp + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
        return;
    }
    uint32_t sfc;
    const uint32_t packed = quant_half_block(x, sc.s, sc.d, sc.inv_d, sc.d_fast, &sfc);
    const uint32_t word = gather_sf_word(sfc);
    if (!kEdge || col_ok) {
        if (!kEdge || row_ok) *reinterpret_cast<uint32_t*>(cp) = packed;
        if (cg == 0) *reinterpret_cast<uint32_t*>(sp) = word;
    }
}

template <int kWType, bool kDump>
__global__ void __launch_bounds__(kRqThreads, 2) requant_quant_kernel(RqArgs a) {
    extern __shared__ __align__(16) float rq_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr = warp >> 1, wc = warp & 1, rg = lane >> 3, cg = lane & 7;
    float* As = rq_smem;
    float* Bt0 = As + a.r * kRqCols + wr * 2 * a.r * 32;
    float* Ws = As + a.r * kRqCols + 4 * 2 * a.r * 32 + warp * Rq2Geom<kWType>::kWsFloats;

    const int64_t t_begin = (int64_t)blockIdx.x * a.tiles2 / gridDim.x;
    const int64_t t_end = (int64_t)(blockIdx.x + 1) * a.tiles2 / gridDim.x;
    RqScale sc;
    // The dump variant (test hook) has no s_t: it writes merged values only.
    const float amax = kDump ? 0.0f : *reinterpret_cast<volatile const float*>(a.s_t);
    sc.s = __fdiv_rn(amax, kAmaxDiv);
    sc.d = __fmul_rn(6.0f, sc.s);
    sc.d_fast = fast_recip_ok(sc.d);
    sc.inv_d = sc.d_fast ? recip_approx(sc.d) : 0.0f;
    const float2 cc = make_float2(a.c, a.c);
    const int pair_bar = 1 + wr;  // named barrier of the two warps sharing rows

    int64_t staged = -1;
    RqCursor cur;
    cur.init(a.row_tiles2, kQRows, t_begin);
    if (t_begin < t_end && a.r > 0) rq2_copy_b(a, lane, cur.n0() + wr * 32, wc, Bt0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    int buf = 0;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t n0 = cur.n0(), k0 = cur.k0();
        const bool edge = n0 + kQRows > a.N || k0 + kRqCols > a.K;  // CTA-uniform
        if (cur.strip != staged) {
            __syncthreads();
            for (int e = threadIdx.x; e < a.r * (kRqCols / 4); e += kRqThreads) {
                const int j = e / (kRqCols / 4), c4 = e % (kRqCols / 4);
                const int64_t k = k0 + c4 * 4;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k < a.K) v = *reinterpret_cast<const float4*>(a.A + (int64_t)j * a.K + k);
                *reinterpret_cast<float4*>(As + j * kRqCols + c4 * 4) = v;
            }
            __syncthreads();
            staged = cur.strip;
        }
        // This tile's W block, then the next tile's B rows (both asynchronous).
        __syncwarp();
        rq2_copy_w<kWType>(a, lane, n0 + wr * 32, k0 + wc * 64, Ws);
        asm volatile("cp.async.commit_group;" ::: "memory");
        cur.next();
        // The pair's other buffer was last read in the previous tile's merge.
        named_barrier_sync(pair_bar, 64);
        if (t + 1 < t_end && a.r > 0)
            rq2_copy_b(a, lane, cur.n0() + wr * 32, wc, Bt0 + (buf ^ 1) * a.r * 32);
        asm volatile("cp.async.commit_group;" ::: "memory");
        // B of this tile (committed one tile ago) has landed, in both warps of the pair.
        asm volatile("cp.async.wait_group 2;" ::: "memory");
        named_barrier_sync(pair_bar, 64);
        const float* Bt = Bt0 + buf * a.r * 32;
        buf ^= 1;

        // acc[i][p]: row i of this lane's 8, columns 2p, 2p+1.
        float2 acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[i][p] = make_float2(0.0f, 0.0f);
        const float* ap = As + wc * 64 + cg * 8;
        int j4 = 0;
#pragma unroll 1
        for (; j4 + 4 <= a.r; j4 += 4) {
            const int sw = j4 & 28;
            const float* b0p = Bt + j4 * 32 + ((rg * 8) ^ sw);
            const float* b1p = Bt + j4 * 32 + ((rg * 8 + 4) ^ sw);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 b0 = *reinterpret_cast<const float4*>(b0p + u * 32);
                const float4 b1 = *reinterpret_cast<const float4*>(b1p + u * 32);
                const float4 a0 = *reinterpret_cast<const float4*>(ap + (j4 + u) * kRqCols);
                const float4 a1 = *reinterpret_cast<const float4*>(ap + (j4 + u) * kRqCols + 4);
                const float bl[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float2 av[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w),
                                      make_float2(a1.x, a1.y), make_float2(a1.z, a1.w)};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // Row i sits at element (i % 4) ^ u of its 16-byte group.
                    const float bv = bl[(i & 4) | ((i & 3) ^ u)];
                    const float2 bb = make_float2(bv, bv);
#pragma unroll
                    for (int p = 0; p < 4; ++p) acc[i][p] = __ffma2_rn(bb, av[p], acc[i][p]);
                }
            }
        }
#pragma unroll 1
        for (int j = j4; j < a.r; ++j) {
            const float4 a0 = *reinterpret_cast<const float4*>(ap + j * kRqCols);
            const float4 a1 = *reinterpret_cast<const float4*>(ap + j * kRqCols + 4);
            const float2 av[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w),
                                  make_float2(a1.x, a1.y), make_float2(a1.z, a1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float bv = Bt[j * 32 + ((rg * 8 + i) ^ (j & 31))];
                const float2 bb = make_float2(bv, bv);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[i][p] = __ffma2_rn(bb, av[p], acc[i][p]);
            }
        }

        // This tile's W block has landed (the next tile's B may still be in flight).
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncwarp();
        // Row i of this lane: codes at cp + i K/2, its scale word at sp + 16 i (the 8
        // rows share one 32-row group of the scale layout).
        const int64_t k = k0 + wc * 64 + cg * 8;
        const int64_t nb = n0 + wr * 32 + rg * 8;
        const bool col_ok = k < a.K;
        uint8_t* cp = kDump ? nullptr : a.codes + nb * (a.K >> 1) + (k >> 1);
        uint8_t* sp = kDump ? nullptr : a.sf + sf_word_offset(nb, k >> 4, a.K);
        float* dp = kDump ? a.dump + nb * a.K + k : nullptr;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float x[8];
            rq2_w_row<kWType>(Ws, rg * 8 + i, cg, x);
            if (a.r > 0) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 y = __ffma2_rn(cc, acc[i][p], make_float2(x[2 * p], x[2 * p + 1]));
                    x[2 * p] = y.x;
                    x[2 * p + 1] = y.y;
                }
            }
            if (edge) {
                const bool row_ok = nb + i < a.N;
                if (!row_ok) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) x[q] = 0.0f;  // scale padding rows quantize zeros
                }
                rq2_emit_row<true, kDump>(sc, cg, row_ok, col_ok, cp, sp, dp, x);
            } else {
                rq2_emit_row<false, kDump>(sc, cg, true, true, cp, sp, dp, x);
            }
            if (!kDump) {
                cp += a.K >> 1;
                sp += 16;
            } else {
                dp += a.K;
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__global__ void requant_finalize_kernel(float* s_t) {
    if (threadIdx.x == 0 && blockIdx.x == 0) *s_t = __fdiv_rn(*s_t, kAmaxDiv);
}

template <typename Kern>
cudaError_t rq_grid(OccupancyCache& occupancy, const LaunchCtx& ctx, Kern kern, size_t smem,
                    int64_t tiles, unsigned* grid) {
    int per_sm = 0;
    const cudaError_t e = blocks_per_sm(occupancy, ctx, kern, kRqThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t g = (int64_t)ctx.num_sms * per_sm;
    *grid = (unsigned)(tiles < g ? tiles : g);
    return cudaSuccess;
}

RqArgs rq_args(const void* W, const float* A, const float* B, int r, float c, int64_t N, int64_t K,
               uint8_t* codes, uint8_t* sf, float* s_t, float* dump) {
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
    a.dump = dump;
    a.row_tiles = a.rows_pad / kRqRows;
    a.tiles = a.row_tiles * ((K + kRqCols - 1) / kRqCols);
    a.row_tiles2 = a.rows_pad / kQRows;
    a.tiles2 = a.row_tiles2 * ((K + kRqCols - 1) / kRqCols);
    a.rs = rq_bstride(r);
    a.inv_r = rq_inv_r(r);
    a.b_vec = r > 0 && r % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    return a;
}

template <int kWType>
cudaError_t run_requant(const LaunchCtx& ctx, const RqArgs& a) {
    const size_t smem1 = rq_smem_bytes(a.r), smem2 = rq2_smem_bytes<kWType>(a.r);
    unsigned g1 = 0, g2 = 0;
    static OccupancyCache occ_amax, occ_quant;
    cudaError_t e = rq_grid(occ_amax, ctx, requant_amax_kernel<kWType>, smem1, a.tiles, &g1);
    if (e != cudaSuccess) return e;
    e = rq_grid(occ_quant, ctx, requant_quant_kernel<kWType, false>, smem2, a.tiles2, &g2);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.s_t, 0, sizeof(float), ctx.stream);
    if (e != cudaSuccess) return e;
    requant_amax_kernel<kWType><<<g1, kRqThreads, smem1, ctx.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    requant_quant_kernel<kWType, false><<<g2, kRqThreads, smem2, ctx.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    requant_finalize_kernel<<<1, 32, 0, ctx.stream>>>(a.s_t);
    return cudaGetLastError();
}

template <int kWType>
cudaError_t run_merge_dump(const LaunchCtx& ctx, const RqArgs& a) {
    const size_t smem = rq2_smem_bytes<kWType>(a.r);
    unsigned g = 0;
    static OccupancyCache occupancy;
    cudaError_t e = rq_grid(occupancy, ctx, requant_quant_kernel<kWType, true>, smem, a.tiles2, &g);
    if (e != cudaSuccess) return e;
    requant_quant_kernel<kWType, true><<<g, kRqThreads, smem, ctx.stream>>>(a);
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

__global__ void test_e4m3_decode_kernel(const uint8_t* c, float* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = e4m3_value(c[i]);
}

__global__ void test_e2m1_quotient_kernel(const float* x, const float* den, uint8_t* out,
                                          int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float dn = den[i];
        const float xs[8] = {x[i], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        out[i] = (uint8_t)(e2m1_quotient8(xs, dn, make_recip(dn)) & 0xFu);
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

// G warps per row: the fewest that keep a thread at kAqMaxBpt blocks of 16 or less;
// for K a multiple of 512 up to 4096, one warp per row with a fixed block count.
template <int kMode>
cudaError_t dispatch_act_quant(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                               const float* amax_in, uint8_t* codes, uint8_t* sf, float* s_row) {
    const int64_t rows_pad = (M + 127) / 128 * 128;
    if (K <= 4096 && K % 512 == 0) {
        switch (K / 512) {
            case 1: return run_act_quant<1, kMode, 1>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 2: return run_act_quant<1, kMode, 2>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 3: return run_act_quant<1, kMode, 3>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 4: return run_act_quant<1, kMode, 4>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 5: return run_act_quant<1, kMode, 5>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 6: return run_act_quant<1, kMode, 6>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            case 7: return run_act_quant<1, kMode, 7>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
            default: return run_act_quant<1, kMode, 8>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
        }
    }
    if (K <= 4096) return run_act_quant<1, kMode>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
    if (K <= 8192) return run_act_quant<2, kMode>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
    if (K <= 16384) return run_act_quant<4, kMode>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
    return run_act_quant<8, kMode>(ctx, X, M, K, rows_pad, amax_in, codes, sf, s_row);
}

}  // namespace

cudaError_t launch_act_quant(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                             uint8_t* codes, uint8_t* sf, float* s_row) {
    return dispatch_act_quant<kAqReduce>(ctx, X, M, K, nullptr, codes, sf, s_row);
}

cudaError_t launch_act_quant_prescaled(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                                       const float* row_amax, uint8_t* codes, uint8_t* sf, float* s_row) {
    return dispatch_act_quant<kAqGivenRow>(ctx, X, M, K, row_amax, codes, sf, s_row);
}

cudaError_t launch_act_quant_tensor(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                                    uint8_t* codes, uint8_t* sf, float* s_t) {
    cudaError_t e = cudaMemsetAsync(s_t, 0, sizeof(float), ctx.stream);
    if (e != cudaSuccess) return e;
    const int64_t n_vec = M * K / 8;
    int64_t grid = (n_vec + kAmaxThreads - 1) / kAmaxThreads;
    if (grid > (int64_t)ctx.num_sms * 8) grid = (int64_t)ctx.num_sms * 8;
    act_amax_kernel<<<(unsigned)grid, kAmaxThreads, 0, ctx.stream>>>(reinterpret_cast<const uint4*>(X), n_vec,
                                                                     s_t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // Pass 2 with the tensor's amax (still in *s_t); then s_t = amax / 2688.
    e = dispatch_act_quant<kAqGivenTensor>(ctx, X, M, K, s_t, codes, sf, nullptr);
    if (e != cudaSuccess) return e;
    act_scale_kernel<<<1, 1, 0, ctx.stream>>>(s_t);
    return cudaGetLastError();
}

cudaError_t launch_requant(const LaunchCtx& ctx, const void* W, int w_dtype, const float* A,
                           const float* B, int r, float c, int64_t N, int64_t K, uint8_t* codes,
                           uint8_t* sf, float* s_t) {
    const RqArgs a = rq_args(W, A, B, r, c, N, K, codes, sf, s_t, nullptr);
    return w_dtype == NVFP4_W_BF16 ? run_requant<NVFP4_W_BF16>(ctx, a)
                                   : run_requant<NVFP4_W_FP32>(ctx, a);
}

cudaError_t launch_test_merge(const LaunchCtx& ctx, const void* W, int w_dtype, const float* A,
                              const float* B, int r, float c, int64_t N, int64_t K, float* out) {
    const RqArgs a = rq_args(W, A, B, r, c, N, K, nullptr, nullptr, nullptr, out);
    return w_dtype == NVFP4_W_BF16 ? run_merge_dump<NVFP4_W_BF16>(ctx, a)
                                   : run_merge_dump<NVFP4_W_FP32>(ctx, a);
}

cudaError_t launch_test_e2m1(const LaunchCtx& ctx, const float* q, uint8_t* codes, int64_t n) {
    test_e2m1_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(q, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_test_e4m3(const LaunchCtx& ctx, const float* v, uint8_t* codes, int64_t n) {
    test_e4m3_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(v, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_test_e4m3_decode(const LaunchCtx& ctx, const uint8_t* codes, float* out,
                                    int64_t n) {
    test_e4m3_decode_kernel<<<grid_for(n, ctx), 256, 0, ctx.stream>>>(codes, out, n);
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
