// LoRA merge on the tensor cores with certified-exact NVFP4 decisions.
//
// nvfp4_requant's result is defined by the fp32 fma chain of the merge
// (acc = +0; acc = fma(B[n,j], A[j,k], acc), j = 0..r-1; w' = fma(c, acc, W[n,k]))
// followed by the NVFP4 quantization of w' (Sol-RL project page, "Two-Stage
// Pipeline", Stage 2: the updated weights are quantized again; AI Trends summary:
// LoRA rank 32).  On CUDA cores the chain costs 32 fp32 FMAs per element and pass,
// more than the weights' memory traffic.  Here the rank-32 product P = B A is taken
// from the tensor cores instead, from two-part bf16 splits of both factors
// (b = b0 + b1 and a = a0 + a1 with b0 = bf16(b), b1 = bf16(b - b0); b - b0 is exact),
// as one bf16 GEMM with K' = 4 x 32 whose operands are [b0 b0 b1 b1] and [a0 a1 a0 a1]:
//     P~[n,k] = sum_j (b0 a0 + b0 a1 + b1 a0 + b1 a1)[n,j,k],     w~ = fma(c, P~, W).
//
// The bound.  For a thread's row n and 64 columns, with b = ||B[n,:]||_2 and
// a = max_k ||A[:,k]||_2 (upper bounds),
//     E = |c| (2^-14 b a + 2^-120 (b + a) + 2^-117)      (rounded up, at least 2^-149)
// covers |c| |P(chain) - P~|.  Relative part, by Cauchy-Schwarz relative to b a: the
// chain's own rounding (r 2^-24 = 2^-19), the dropped split remainder (b1 and a1 are
// bf16 roundings: 2 x 2^-9 x 2^-8 plus 2^-18, about 2^-16.4) and the tensor cores'
// accumulation (8 MMAs of 16 exact bf16 products in fp32, at most 17 x 2^-23 of the
// magnitudes each, 2^-15.9) sum to about 2^-15.1; the factor of two left covers the
// roundings of the final fma (2^-23 relative, taken up by the 2^-19 nudges below) and
// the second-order terms.  Absolute part, should the tensor cores flush subnormals:
// a flushed split part (below 2^-126) loses at most 2^-124 sum_j |a_j| <= 2^-121.5 a
// (or b), flushed products and partial sums at most 128 x 2^-126.  The chain's own
// subnormal roundings are far below 2^-117.  Every decision is taken on the interval
// [|w~| - E, |w~| + E] (with the final fma's own rounding covered by 2^-19 / 2^-21
// nudges of the reciprocals and factors):
//   * tensor amax (pass 1): a warp's maximum is among its elements whose upper bound
//     reaches the largest lower bound of the warp; those are recomputed with the exact
//     chain and the warp's maximum of them goes to the tensor amax;
//   * block scale (pass 2): the E4M3 codes of both ends of [bam - E, bam + E] must agree,
//     else the block's 16 values are recomputed exactly;
//   * element code (pass 2): the E2M1 codes of both ends must agree (an interval that
//     holds zero gives codes of both signs and never agrees), else that element alone
//     is recomputed.
// So codes, scales and s_t are bit-identical to the fp32 chain's.  The exact chain
// reads the fp32 factors from shared memory.
//
// Kernels.  A split kernel writes A' = [a0 a1 a0 a1] per column of A (bf16, 256 bytes
// per row) into the caller's workspace, with upper bounds of every row norm of B and,
// per 64 columns, of the largest column norm of A.  Then both passes run as persistent
// clusters of two CTAs; a pair tile is 256 weight rows (128 per CTA) x 128 columns,
// walked k-strip first, so the rows of B usually stay the same from one tile to the
// next.  Per CTA, 20 warps:
//   warp 0      TMA: W tiles (128 x 128 bf16; 4 slots) and the fp32 strip of A for the
//               exact chain (3 slots), each freed when the epilogue is done with the tile;
//   warp 1      tensor-memory allocation; lane 0 of the even CTA issues the 8 pair MMAs
//               (kind::f16, M = 256, N = 128, A from tensor memory) into a
//               double-buffered accumulator;
//   warp 2      TMA: this CTA's 64 rows of A' (the MMA's B operand; 3 slots),
//               completing on the even CTA's barrier, freed by the MMAs;
//   warp 3      idle;
//   warps 4-19  epilogue: four warps per tensor-memory lane quarter, 32 columns each (a
//               thread owns one weight row): accumulator + W -> w~ -> pass 1 amax or
//               pass 2 codes and scales, stored straight to global memory.
// The rows of B live in tensor memory next to the accumulators (lane = row), in two
// buffers for consecutive row blocks: [b0 b0 b1 b1] as bf16 pairs (the MMA's A
// operand) and the fp32 values (for the exact chain).  The epilogue warps write the
// next row block's buffer one tile ahead; only the rare uncertain elements read the
// fp32 rows and the strip of A.
// Every mbarrier wait is bounded (mbar_wait).
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int kTM = 128;        // weight rows per CTA
constexpr int kTK = 128;        // weight columns per pair tile (64 per CTA in the MMA's B)
constexpr int kPair = 2;
constexpr int kRank = 32;       // the rank this path serves (A [32, K], B [N, 32])
constexpr int kJp = 4 * kRank;  // K' of the merge GEMM
constexpr int kEpiWarp0 = 4, kEpiWarps = 16;  // warp groups: 0 control, 1-4 epilogue
constexpr int kCols = 32;       // columns per epilogue warp
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kWSlots = 4, kXSlots = 3, kOpSlots = 3;
constexpr uint32_t kOpBBytes = (kTK / kPair) * kJp * 2;  // 16 KB: A' rows, two 64-column atoms
constexpr uint32_t kWBox = kTM * 128;                    // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kWBytes = 2 * kWBox;                  // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kAfBytes = kRank * kTK * 4;           // 16 KB: fp32 strip of A
constexpr uint32_t kMiscBytes = 512;
constexpr uint32_t kSmemBytes =
    1024 + kOpSlots * kOpBBytes + kWSlots * kWBytes + kXSlots * kAfBytes + kMiscBytes;
// Tensor memory: two accumulators of 128 columns, then two row buffers of 96 columns:
// 64 columns of [b0 b0 b1 b1] (bf16 pairs) and 32 columns of fp32 B.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRowBuf0 = 2 * kTK, kRowBufCols = 96, kRowBufF32 = 64;
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kEvenCta = 0x1;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kModeAmax = 0, kModeQuant = 1;
constexpr int kSplitThreads = 256;
constexpr int kSplitRows = kSplitThreads / 4;  // rows of B per split block (4 threads a row)
constexpr int kSplitCols = kSplitThreads / 4;  // columns of A per split block (4 threads a column)
// Registers: launched at 96 per thread (20 warps, 5 per scheduler); the control warp
// group drops to 32 and the epilogue warp groups rise to 112 (4 x 32 + 16 x 112 <=
// 20 x 96).
constexpr uint32_t kRegsCtl = 56, kRegsEpi = 104;
static_assert(4 * kRegsCtl + kEpiWarps * kRegsEpi <= (uint32_t)(kThreads / 32) * 96, "register split");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kRowBuf0 + 2 * kRowBufCols <= kTmemCols, "tensor memory budget");

// kind::f16, bf16 A and B, fp32 accumulator, K-major, N = 128, M = 256 (pair).
constexpr uint32_t idesc_merge() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTK >> 3) << 17) |
           ((uint32_t)(kTM * kPair >> 4) << 24);
}

struct TcArgs {
    float c;
    int N, K, rows_pad;
    uint8_t* codes;
    uint8_t* sf;
    float* s_t;  // pass 1: amax accumulator (fp32 bits, atomicMax); pass 2: reads it
    const float* rnorm;  // [N padded to 256] upper bounds of ||B[n,:]||_2 (0 past N)
    const float* B;      // [N, 32] fp32
    const float* cnorm;  // [K/128][4]: per 128-column strip, the largest ||A[:,k]||_2
                         // of each 64-column half (upper bounds), then 2 unused
    unsigned int* counter;  // CTAs of the quantize pass that are done (zeroed by the split)
    int* status;
    int zero;    // 0 (a value the compiler cannot see; used for data dependencies)
    int nks;     // 128-column strips
    int tiles;   // 256-row blocks x nks, row block major
};

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Upper bound of the 2-norm from a sum of 32 squares accumulated with round-to-nearest
// fmas (relative error below 2^-19; the absolute term covers underflow).
__device__ __forceinline__ float norm_ub(float sumsq) {
    return __fsqrt_ru(__fmaf_ru(sumsq, 1.0f + 0x1p-17f, 0x1p-143f));
}

__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two-part bf16 split of 8 values: p0 = bf16(v), p1 = bf16(v - p0).
__device__ __forceinline__ void split8(const float* v, uint4& p0, uint4& p1) {
    float h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
        l[i] = v[i] - h[i];
    }
    p0 = make_uint4(bf16_pair(h[0], h[1]), bf16_pair(h[2], h[3]), bf16_pair(h[4], h[5]),
                    bf16_pair(h[6], h[7]));
    p1 = make_uint4(bf16_pair(l[0], l[1]), bf16_pair(l[2], l[3]), bf16_pair(l[4], l[5]),
                    bf16_pair(l[6], l[7]));
}

// Four threads per row of B or column of A (8 values each).  Blocks [0, nb_rows) take
// 64 rows of B: rnorm[n] (0 for the padding rows up to rows_pad256).  The other blocks
// take 64 columns of A: A'[k] = [a0 a1 a0 a1] and the block's largest column norm.
// Block 0 also clears the amax accumulator s_t and the quantize pass's CTA counter.
__global__ void __launch_bounds__(kSplitThreads)
    merge_split_kernel(const float* __restrict__ A, const float* __restrict__ B, int N, int K,
                       int rows_pad256, int nb_rows, uint8_t* __restrict__ Ap,
                       float* __restrict__ rnorm, float* __restrict__ cnorm,
                       float* __restrict__ s_t, unsigned int* __restrict__ counter) {
    __shared__ float red[kSplitThreads];
    __shared__ float red2[kSplitCols / 32];
    const int tid = (int)threadIdx.x;
    grid_dep_launch();  // the amax pass may start streaming W at once
    if (blockIdx.x == 0 && tid == 0) {
        *s_t = 0.0f;
        *counter = 0u;
    }
    float v[8];
    if ((int)blockIdx.x < nb_rows) {
        const int n = (int)blockIdx.x * kSplitRows + (tid >> 2), g = tid & 3;
        float s2 = 0.0f;
        if (n < N) {
            const float4* src = reinterpret_cast<const float4*>(B + (int64_t)n * kRank + 8 * g);
            const float4 x0 = src[0], x1 = src[1];
            s2 = __fmaf_rn(x0.x, x0.x, s2);
            s2 = __fmaf_rn(x0.y, x0.y, s2);
            s2 = __fmaf_rn(x0.z, x0.z, s2);
            s2 = __fmaf_rn(x0.w, x0.w, s2);
            s2 = __fmaf_rn(x1.x, x1.x, s2);
            s2 = __fmaf_rn(x1.y, x1.y, s2);
            s2 = __fmaf_rn(x1.z, x1.z, s2);
            s2 = __fmaf_rn(x1.w, x1.w, s2);
        }
        // The four partial sums of the row (lanes 4r .. 4r + 3 of the warp).
        s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, 1);
        s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, 2);
        if (g == 0 && n < rows_pad256) rnorm[n] = n < N ? norm_ub(s2) : 0.0f;
    } else {
        const int k0 = ((int)blockIdx.x - nb_rows) * kSplitCols;
        const int kk = tid & (kSplitCols - 1), g = tid / kSplitCols;
        const int k = k0 + kk;
        float s2 = 0.0f;
        if (k < K) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = A[(int64_t)(8 * g + j) * K + k];
#pragma unroll
            for (int j = 0; j < 8; ++j) s2 = __fmaf_rn(v[j], v[j], s2);
            uint4 p0, p1;
            split8(v, p0, p1);
            uint4* dst = reinterpret_cast<uint4*>(Ap + (int64_t)k * (kJp * 2));
            dst[g] = p0;
            dst[4 + g] = p1;
            dst[8 + g] = p0;
            dst[12 + g] = p1;
        }
        red[tid] = s2;
        __syncthreads();
        if (tid < kSplitCols) {
            const float t = (red[tid] + red[tid + kSplitCols]) + (red[tid + 2 * kSplitCols] + red[tid + 3 * kSplitCols]);
            const float nrm = warp_max_f(k < K ? norm_ub(t) : 0.0f);
            if ((tid & 31) == 0) red2[tid >> 5] = nrm;
        }
        __syncthreads();
        if (tid == 0 && k0 < K) cnorm[(k0 >> 7) * 4 + ((k0 >> 6) & 1)] = fmaxf(red2[0], red2[1]);
    }
}

// W[row, kt] of a W tile in shared memory (bf16, two 64-column boxes with the 128-byte
// swizzle: the 16-byte chunk u of a row sits at chunk u ^ (row % 8)).
__device__ __forceinline__ float w_at(const uint8_t* wt, int row, int kt) {
    const int u = (kt & 63) >> 3;
    const uint16_t h = *reinterpret_cast<const uint16_t*>(
        wt + (kt >> 6) * kWBox + row * 128 + ((u ^ (row & 7)) << 4) + (kt & 7) * 2);
    return __uint_as_float((uint32_t)h << 16);
}

// The library's merged value of one element (the fp32 fma chain, in order): b = the
// element's row of B (fp32 bits), column kt of the fp32 strip of A (32 x kTK), weight w.
__device__ __forceinline__ float exact_value(const uint32_t (&b)[kRank], const float* af, int kt,
                                             float c, float w) {
    float a[kRank];
#pragma unroll
    for (int j = 0; j < kRank; ++j) a[j] = af[j * kTK + kt];
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kRank; ++j) acc = __fmaf_rn(__uint_as_float(b[j]), a[j], acc);
    return __fmaf_rn(c, acc, w);
}

// Pass 2's rare path for one thread's 32 columns (called by the whole warp; `slow`
// says whether this thread has work): blocks whose scale is uncertain get their 16
// values from the exact chain (16 chains side by side), then the scale and codes by
// true divisions; elements whose interval ends disagree (diff) get their code from
// the exact chain.  tbrow is the tensor-memory address of the fp32 rows of B, af the
// fp32 strip of A, wt the W tile in shared memory and row this thread's row in it.
struct Codes32 {
    uint32_t cw[4];
    uint32_t sfc[2];
};
__device__ __forceinline__ Codes32 quant_fix(uint32_t tbrow, const float* af, int kt0, float c, float s,
                                          float d, Codes32 r, uint4 diff, float den0, float den1,
                                          bool cert0, bool cert1, bool slow, const uint8_t* wt, int row) {
    uint32_t bq[kRank];
    tmem_ld_32x32b_x32(tbrow, bq);
    tmem_ld_wait();
    if (!slow) return r;
#pragma unroll 1
    for (int bk = 0; bk < 2; ++bk) {
        if (bk == 0 ? cert0 : cert1) continue;
        const int kt = kt0 + 16 * bk;
        float x16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x16[e] = 0.0f;
#pragma unroll 2
        for (int j = 0; j < kRank; ++j) {
            const float bj = __uint_as_float(bq[j]);
            const float4* ar = reinterpret_cast<const float4*>(af + j * kTK + kt);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 v = ar[q4];
                x16[4 * q4] = __fmaf_rn(bj, v.x, x16[4 * q4]);
                x16[4 * q4 + 1] = __fmaf_rn(bj, v.y, x16[4 * q4 + 1]);
                x16[4 * q4 + 2] = __fmaf_rn(bj, v.z, x16[4 * q4 + 2]);
                x16[4 * q4 + 3] = __fmaf_rn(bj, v.w, x16[4 * q4 + 3]);
            }
        }
        float bam = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            x16[e] = __fmaf_rn(c, x16[e], w_at(wt, row, kt + e));
            bam = fmaxf(bam, fabsf(x16[e]));
        }
        uint32_t sc = 0;
        if (d > 0.0f) sc = cvt_e4m3(__fdiv_rn(bam, d));
        const float dn = __fmul_rn(e4m3_value(sc), s);
        uint32_t c0 = 0u, c1 = 0u;
        if (dn > 0.0f) {
#pragma unroll
            for (int e = 0; e < 16; ++e) x16[e] = __fdiv_rn(x16[e], dn);
            c0 = cvt_e2m1x8(x16[0], x16[1], x16[2], x16[3], x16[4], x16[5], x16[6], x16[7]);
            c1 = cvt_e2m1x8(x16[8], x16[9], x16[10], x16[11], x16[12], x16[13], x16[14], x16[15]);
        }
        if (bk == 0) {
            r.cw[0] = c0; r.cw[1] = c1; r.sfc[0] = sc;
        } else {
            r.cw[2] = c0; r.cw[3] = c1; r.sfc[1] = sc;
        }
    }
    // Elements whose two ends disagree (in blocks with a certain scale).
    const uint32_t dw[4] = {diff.x, diff.y, diff.z, diff.w};
    uint32_t um = 0u;
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int j = 0; j < 8; ++j) um |= (((dw[w] >> (4 * j)) & 0xFu) != 0u ? 1u : 0u) << (8 * w + j);
    if (!cert0) um &= 0xFFFF0000u;
    if (!cert1) um &= 0x0000FFFFu;
#pragma unroll 1
    while (um != 0u) {
        const int e = __ffs((int)um) - 1;
        um &= um - 1u;
        const float x = exact_value(bq, af, kt0 + e, c, w_at(wt, row, kt0 + e));
        const uint32_t code = cvt_e2m1x8(__fdiv_rn(x, e < 16 ? den0 : den1), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
        const uint32_t sh = 4u * (uint32_t)(e & 7), keep = ~(0xFu << sh);
        const int wi = e >> 3;
        if (wi == 0) r.cw[0] = (r.cw[0] & keep) | (code << sh);
        else if (wi == 1) r.cw[1] = (r.cw[1] & keep) | (code << sh);
        else if (wi == 2) r.cw[2] = (r.cw[2] & keep) | (code << sh);
        else r.cw[3] = (r.cw[3] & keep) | (code << sh);
    }
    return r;
}

// Writes the rows of row block nbw into row buffer nrb & 1 of tensor memory (this
// warp's 8 of the 32 columns of B for its 32 rows: the bf16 parts for the MMA, fp32
// for the exact chain), once the lane quarter's 4 warps are all past the tiles that
// used the buffer, and publishes them to the quarter (qbar) and to the MMA (rows_ready,
// on the even CTA).  Returns false if a wait gave up.
__device__ __forceinline__ bool write_rows(const TcArgs& args, uint32_t tmem_base, uint32_t tlane,
                                           uint64_t* qbar, uint32_t rows_ready_even, int nbw,
                                           uint32_t rank, int rloc, int chunk, int lane, int& nrb,
                                           int& nqb, volatile int* abort_flag) {
    if (lane == 0) mbar_arrive(qbar);
    bool ok = mbar_wait(qbar, (uint32_t)(nqb & 1), args.status, abort_flag, kWaitLimitNs);
    ++nqb;
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    tc_fence_after_sync();
    const int n = nbw * (kTM * kPair) + (int)rank * kTM + rloc;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (n < args.N) {
        const float4* src = reinterpret_cast<const float4*>(args.B + (int64_t)n * kRank + 8 * chunk);
        const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    }
    uint4 p0, p1;
    split8(v, p0, p1);
    const uint32_t base = tmem_base + tlane + kRowBuf0 + kRowBufCols * (uint32_t)(nrb & 1);
    // [b0 b0 b1 b1]: K' index 32 g + j (g = part, j = column of B) sits in column
    // (32 g + j) / 2 as the low (j even) or high half.
    const uint32_t r0[4] = {p0.x, p0.y, p0.z, p0.w}, r1[4] = {p1.x, p1.y, p1.z, p1.w};
    const uint32_t col = 4u * (uint32_t)chunk;
    tmem_st_32x32b_x4(base + col, r0);
    tmem_st_32x32b_x4(base + 16u + col, r0);
    tmem_st_32x32b_x4(base + 32u + col, r1);
    tmem_st_32x32b_x4(base + 48u + col, r1);
    uint32_t f[8];
#pragma unroll
    for (int z = 0; z < 8; ++z) f[z] = __float_as_uint(v[z]);
    tmem_st_32x32b_x8(base + kRowBufF32 + 8u * (uint32_t)chunk, f);
    tmem_st_wait();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
        mbar_arrive_cluster(rows_ready_even + 8u * (uint32_t)(nrb & 1));
        mbar_arrive(qbar);
    }
    ok = mbar_wait(qbar, (uint32_t)(nqb & 1), args.status, abort_flag, kWaitLimitNs);
    ++nqb;
    ++nrb;
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    tc_fence_after_sync();
    return true;
}

// Pass 1's candidate path (called by the whole warp): the largest |W'| over the
// elements of `mask` (this thread's columns kt0 + e), by the exact chain.
__device__ __forceinline__ float amax_exact(uint32_t tbrow, const float* af, int kt0, float c, uint32_t mask,
                                         const uint8_t* wt, int row) {
    uint32_t bq[kRank];
    tmem_ld_32x32b_x32(tbrow, bq);
    tmem_ld_wait();
    float em = 0.0f;
#pragma unroll 1
    while (mask != 0u) {
        const int e = __ffs((int)mask) - 1;
        mask &= mask - 1u;
        em = fmaxf(em, fabsf(exact_value(bq, af, kt0 + e, c, w_at(wt, row, kt0 + e))));
    }
    return em;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    merge_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_ap,
                    const __grid_constant__ CUtensorMap tmap_af, const TcArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* opB = smem;                          // [kOpSlots]: A' rows of this CTA's 64 columns
    uint8_t* wring = opB + kOpSlots * kOpBBytes;  // [kWSlots]: W tiles
    uint8_t* xring = wring + kWSlots * kWBytes;   // [kXSlots]: fp32 strips of A
    uint64_t* bars = reinterpret_cast<uint64_t*>(xring + kXSlots * kAfBytes);
    uint64_t* w_full = bars;                         // [kWSlots]
    uint64_t* w_empty = w_full + kWSlots;            // [kWSlots] the 16 epilogue warps
    uint64_t* op_full = w_empty + kWSlots;           // [kOpSlots] even CTA: both CTAs' A'
    uint64_t* op_empty = op_full + kOpSlots;         // [kOpSlots] the pair's MMAs are done
    uint64_t* x_full = op_empty + kOpSlots;          // [kXSlots]
    uint64_t* x_empty = x_full + kXSlots;            // [kXSlots] the 16 epilogue warps
    uint64_t* tmem_full = x_empty + kXSlots;         // [2]
    uint64_t* tmem_empty = tmem_full + 2;            // [2] even CTA
    uint64_t* rows_ready = tmem_empty + 2;           // [2] even CTA: a row buffer is written
    uint64_t* quarter_bar = rows_ready + 2;          // [4] the 4 warps of a lane quarter
    uint64_t* drain = quarter_bar + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x / kPair), npairs = (int)(gridDim.x / kPair);
    const int t_begin = (int)((int64_t)pair * args.tiles / npairs);
    const int t_end = (int)((int64_t)(pair + 1) * args.tiles / npairs);
    // Tile t of the pair's range: row block t / nks, strip t % nks (walked strip first).
    const int nks = args.nks;
    const int nb_begin = t_begin / nks, ks_begin = t_begin - nb_begin * nks;
    // The next pass may start as SMs free up: W does not depend on this one.  What
    // depends on the previous kernel (A', the norms, s_t) is read after grid_dep_wait.
    if (kMode == kModeAmax) grid_dep_launch();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWSlots; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kOpSlots; ++i) {
            mbar_init(&op_full[i], 1);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < kXSlots; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], kEpiWarps * kPair);
            mbar_init(&rows_ready[i], kEpiWarps * kPair);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&quarter_bar[i], kEpiWarps / 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_w);
        prefetch_tmap(&tmap_af);
    }
    if (warp == 2 && lane == 0) prefetch_tmap(&tmap_ap);
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < kEpiWarp0) {
        regs_decrease<kRegsCtl>();
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA: W and strips of A
            int nb = nb_begin, ks = ks_begin, i = 0;
            for (int t = t_begin; t < t_end; ++t, ++i) {
                const int ws = i % kWSlots, xs = i % kXSlots;
                const int row0 = nb * (kTM * kPair) + (int)rank * kTM;
                // W (the stream from HBM).
                if (!mbar_wait(&w_empty[ws], (uint32_t)((i / kWSlots) & 1) ^ 1u, args.status,
                               abort_flag, kWaitLimitNs))
                    break;
                uint8_t* wt = wring + ws * kWBytes;
                mbar_arrive_expect_tx(&w_full[ws], kWBytes);
                tma_load_2d(&tmap_w, &w_full[ws], wt, ks * kTK, row0);
                tma_load_2d(&tmap_w, &w_full[ws], wt + kWBox, ks * kTK + 64, row0);
                // The fp32 strip of A: the slot's previous strip has landed (its phase is
                // complete) and the epilogue is done with it.
                const uint32_t xph = (uint32_t)((i / kXSlots) & 1) ^ 1u;
                if (!mbar_wait(&x_full[xs], xph, args.status, abort_flag, kWaitLimitNs) ||
                    !mbar_wait(&x_empty[xs], xph, args.status, abort_flag, kWaitLimitNs))
                    break;
                mbar_arrive_expect_tx(&x_full[xs], kAfBytes);
                tma_load_2d(&tmap_af, &x_full[xs], xring + xs * kAfBytes, ks * kTK, 0);
                if (++ks == nks) {
                    ks = 0;
                    ++nb;
                }
            }
            if (!*abort_flag) {
                // Tail: the last strips of A land before exit.
                for (int j = (i >= kXSlots ? i - kXSlots : 0); j < i; ++j)
                    if (!mbar_wait(&x_full[j % kXSlots], (uint32_t)((j / kXSlots) & 1), args.status,
                                   abort_flag, kWaitLimitNs))
                        break;
            }
            if (*abort_flag) {
                // Let copies already issued land before the pair tears down.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------ TMA: A' (the MMA's B operand)
            grid_dep_wait();  // A' is written by the split kernel
            const uint32_t op_full_even = map_to_rank(smem_u32(op_full), 0);
            int ks = ks_begin, i = 0;
            for (int t = t_begin; t < t_end; ++t, ++i) {
                const int os = i % kOpSlots;
                if (!mbar_wait(&op_empty[os], (uint32_t)((i / kOpSlots) & 1) ^ 1u, args.status,
                               abort_flag, kWaitLimitNs))
                    break;
                if (leader) mbar_arrive_expect_tx(&op_full[os], kPair * kOpBBytes);
                const uint32_t bar = op_full_even + 8u * (uint32_t)os;
                const int arow = ks * kTK + (int)rank * (kTK / kPair);
                uint8_t* ob = opB + os * kOpBBytes;
                tma_load_2d_pair(&tmap_ap, bar, ob, 0, arow);
                tma_load_2d_pair(&tmap_ap, bar, ob + kOpBBytes / 2, 64, arow);
                if (++ks == nks) ks = 0;
            }
            if (!*abort_flag) {
                // Tail: the last MMAs' releases of the operand slots land before exit.
                for (int j = (i >= kOpSlots ? i - kOpSlots : 0); j < i; ++j)
                    if (!mbar_wait(&op_empty[j % kOpSlots], (uint32_t)((j / kOpSlots) & 1), args.status,
                                   abort_flag, kWaitLimitNs))
                        break;
            }
            if (*abort_flag) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const uint32_t idesc = idesc_merge();
            bool any = false;
            int nb = nb_begin, ks = ks_begin, rb = -1, nrb = 0;  // row block in use, buffers filled
            for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
                const int b = i & 1, os = i % kOpSlots;
                if (nb != rb) {
                    // A new row block: its [b0 b0 b1 b1] rows are written by the epilogue.
                    if (!mbar_wait<true>(&rows_ready[nrb & 1], (uint32_t)((nrb >> 1) & 1), args.status,
                                         abort_flag, kWaitLimitNs))
                        break;
                    rb = nb;
                    ++nrb;
                }
                if (!mbar_wait<true>(&op_full[os], (uint32_t)((i / kOpSlots) & 1), args.status,
                                     abort_flag, kWaitLimitNs) ||
                    !mbar_wait<true>(&tmem_empty[b], ((i >> 1) & 1) ^ 1u, args.status,
                                     abort_flag, kWaitLimitNs))
                    break;
                tc_fence_after_sync();
                const uint32_t a_col = tmem_base + kRowBuf0 + kRowBufCols * (uint32_t)((nrb - 1) & 1);
                const uint64_t bd = smem_desc(smem_u32(opB + os * kOpBBytes), 16, 1024, kLayoutSw128);
#pragma unroll
                for (int kk = 0; kk < kJp / 16; ++kk) {
                    // 16 bf16 per step: 8 tensor-memory columns of A; 32 bytes of B, 4 steps
                    // per 64-column atom.
                    const uint64_t bo = (uint64_t)((kk >> 2) * ((kOpBBytes / 2) >> 4) + (kk & 3) * 2);
                    mma_bf16_pair_ta(tmem_base + (uint32_t)(b * kTK), a_col + 8u * (uint32_t)kk, bd + bo,
                                     idesc, kk > 0 ? 1u : 0u);
                }
                any = true;
                mma_commit_pair_multicast(&op_empty[os], kBothCtas);
                mma_commit_pair_multicast(&tmem_full[b], kBothCtas);
                if (++ks == nks) {
                    ks = 0;
                    ++nb;
                }
            }
            if (*abort_flag && any) {
                mma_commit_pair_multicast(drain, kEvenCta);
                int dummy = 0;
                mbar_wait(drain, 0, args.status, &dummy, kDrainLimitNs);
            }
        }
    }
    } else {
        regs_increase<kRegsEpi>();
        // ------------------------------------------------ epilogue (warps 4-19, both CTAs)
        const int q = warp & 3;                             // tensor-memory lane quarter
        const int chunk = (warp - kEpiWarp0) >> 2;          // 0..3
        const int kt0 = chunk * kCols;                      // this warp's columns in the tile
        const int rloc = q * 32 + lane;                     // this thread's row in the CTA's 128
        const uint32_t tlane = (uint32_t)(q * 32) << 16;
        const uint32_t rows_ready_even = map_to_rank(smem_u32(rows_ready), 0);
        const uint32_t tmem_empty_even = map_to_rank(smem_u32(tmem_empty), 0);
        const float c = args.c, ac = fabsf(args.c);
        float s = 0.0f, d = 0.0f, idlo = 0.0f, idhi = 0.0f;
        bool d_fast = false;
        int nrb = 0, nqb = 0;  // row buffers written, quarter_bar phases
        // The first row block's rows (B is an input: no wait), then the previous kernel's
        // results (norms, s_t).
        bool alive = t_begin >= t_end ||
                     write_rows(args, tmem_base, tlane, quarter_bar + q, rows_ready_even, nb_begin, rank, rloc,
                                chunk, lane, nrb, nqb, abort_flag);
        grid_dep_wait();
        if (kMode == kModeQuant) {
            const float amax = *reinterpret_cast<volatile const float*>(args.s_t);
            s = __fdiv_rn(amax, kAmaxDiv);
            d = __fmul_rn(6.0f, s);
            d_fast = fast_recip_ok(d);
            const float rd = d_fast ? recip_approx(d) : 0.0f;
            idlo = __fmul_rd(rd, 1.0f - 0x1p-19f);
            idhi = __fmul_ru(rd, 1.0f + 0x1p-19f);
        }
        int nb = nb_begin, ks = ks_begin;
        // The norms for E (global, read one tile ahead) and, in pass 1, the running lower
        // bound of the tensor amax (any value s_t has held is one), read at the end of a
        // tile for use in the next.
        float rb_next = 0.0f, ra_next = 0.0f;
        if (t_begin < t_end) {
            const int k = ks * kTK + kt0;
            rb_next = __ldg(args.rnorm + nb * (kTM * kPair) + (int)rank * kTM + rloc);
            ra_next = k < args.K ? __ldg(args.cnorm + (k >> 7) * 4 + ((k >> 6) & 1)) : 0.0f;
        }
        float st_now = 0.0f, st_next = 0.0f;
        int cur_buf = 0;  // row buffer of the current tile's row block
        for (int t = t_begin, i = 0; alive && t < t_end; ++t, ++i) {
            const int b = i & 1, ws = i % kWSlots, xs = i % kXSlots;
            const uint32_t ph = (uint32_t)((i >> 1) & 1);
            const int n = nb * (kTM * kPair) + (int)rank * kTM + rloc;
            const int k0 = ks * kTK + kt0;        // this warp's first column in W
            const bool row_ok = n < args.N;
            const bool col_ok = k0 < args.K;      // K is a multiple of 64: all 32 columns or none
            const float rb = rb_next, ra = ra_next;
            int nb1 = nb, ks1 = ks + 1;
            if (ks1 == nks) {
                ks1 = 0;
                ++nb1;
            }
            if (t + 1 < t_end) {
                const int k = ks1 * kTK + kt0;
                rb_next = __ldg(args.rnorm + nb1 * (kTM * kPair) + (int)rank * kTM + rloc);
                ra_next = k < args.K ? __ldg(args.cnorm + (k >> 7) * 4 + ((k >> 6) & 1)) : 0.0f;
                // The next tile starts a new row block: write its rows one tile ahead.
                if (nb1 != nb && !write_rows(args, tmem_base, tlane, quarter_bar + q, rows_ready_even, nb1, rank,
                                             rloc, chunk, lane, nrb, nqb, abort_flag))
                    break;
            }
            const uint32_t tbrow = tmem_base + tlane + kRowBuf0 + kRowBufCols * (uint32_t)cur_buf + kRowBufF32;
            if (t + 1 < t_end && nb1 != nb) cur_buf ^= 1;  // from the next tile on
            // The accumulator's 32 columns (released at once) and this thread's 32 weights.
            bool ok = mbar_wait(&tmem_full[b], ph, args.status, abort_flag, kWaitLimitNs) &&
                      mbar_wait(&w_full[ws], (uint32_t)((i / kWSlots) & 1), args.status, abort_flag,
                                kWaitLimitNs);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after_sync();
            const uint8_t* wt = wring + ws * kWBytes;  // this tile's W, held until the tile's end
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tmem_base + tlane + (uint32_t)(b * kTK + kt0), acc);
            uint4 wr[4];
            {
                const uint8_t* wb = wt + (kt0 >> 6) * kWBox + rloc * 128;
                const int u0 = (kt0 & 63) >> 3;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    wr[u] = *reinterpret_cast<const uint4*>(wb + (((u0 + u) ^ (rloc & 7)) << 4));
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tmem_empty_even + 8u * (uint32_t)b);
            // w~ = fma(c, P~, W) for the 32 columns.
            float wv[kCols];
            {
                const float2 cc = make_float2(c, c);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t rw[4] = {wr[u].x, wr[u].y, wr[u].z, wr[u].w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int e = 8 * u + 2 * p;
                        const float2 y = __ffma2_rn(
                            cc, make_float2(__uint_as_float(acc[e]), __uint_as_float(acc[e + 1])),
                            make_float2(__uint_as_float(rw[p] << 16), __uint_as_float(rw[p] & 0xFFFF0000u)));
                        wv[e] = y.x;
                        wv[e + 1] = y.y;
                    }
                }
            }
            // E for this row and these columns, every step rounded up.
            float E;
            {
                const float rel = __fmul_ru(__fmul_ru(ac, 0x1p-14f), __fmul_ru(rb, ra));
                const float abs_ = __fmul_ru(ac, __fmaf_ru(0x1p-120f, __fadd_ru(rb, ra), 0x1p-117f));
                E = fmaxf(__fadd_ru(rel, abs_), 0x1p-149f);
            }
            const float* af = reinterpret_cast<const float*>(xring + xs * kAfBytes);
            const uint32_t xph = (uint32_t)((i / kXSlots) & 1);
            bool x_read = false;  // warp-uniform: the exact chain read the strip of A

            if (kMode == kModeAmax) {
                float m = 0.0f;
#pragma unroll
                for (int e = 0; e < kCols; ++e) m = fmaxf(m, fabsf(wv[e]));
                const bool in = row_ok && col_ok;
                // A lower bound of the tensor amax from this warp's elements.
                const float lo = warp_max_f(in ? __fsub_rd(__fmul_rd(m, 1.0f - 0x1p-21f), E) : 0.0f);
                st_now = fmaxf(st_now, st_next);
                const float thr = fmaxf(lo, st_now);
                // Only elements whose upper bound reaches thr can be the maximum.
                const bool cand = in && __fadd_ru(__fmul_ru(m, 1.0f + 0x1p-21f), E) >= thr;
                float em = 0.0f;
                if (__any_sync(0xFFFFFFFFu, cand)) {
                    uint32_t mask = 0u;
#pragma unroll
                    for (int e = 0; e < kCols; ++e)
                        mask |= (__fadd_ru(__fmul_ru(fabsf(wv[e]), 1.0f + 0x1p-21f), E) >= thr ? 1u : 0u) << e;
                    if (!cand) mask = 0u;
                    ok = mbar_wait(&x_full[xs], xph, args.status, abort_flag, kWaitLimitNs);
                    if (!__all_sync(0xFFFFFFFFu, ok)) break;
                    x_read = true;
                    em = warp_max_f(amax_exact(tbrow, af, kt0, c, mask, wt, rloc));
                }
                const float best = fmaxf(em, lo);
                // |W'| >= 0: the fp32 bit patterns order like the values.
                if (lane == 0 && best > st_now)
                    atomicMax(reinterpret_cast<unsigned int*>(args.s_t), __float_as_uint(best));
                st_next = *reinterpret_cast<volatile const float*>(args.s_t);
            } else {
                uint32_t cw[4], diff[4], sfc[2];
                float den[2];
                bool cert[2];
                float Eb = E;
#pragma unroll
                for (int bk = 0; bk < 2; ++bk) {
                    if (bk == 1) {
                        // Block 1 after block 0 (an empty asm that "reads" block 0's results
                        // and "writes" E): keeps the two blocks' temporaries from being
                        // live at once.
                        asm volatile("" : "+f"(Eb) : "r"(cw[0]), "r"(cw[1]), "r"(diff[0]), "r"(diff[1]));
                    }
                    const float E = Eb;
                    const float* x = wv + 16 * bk;
                    float bam = 0.0f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) bam = fmaxf(bam, fabsf(x[e]));
                    // Block scale: both ends of [bam - E, bam + E] must give the same code.
                    // Rows past N are scale padding (not part of W): scale 0, no codes.
                    const bool scaled = d > 0.0f && row_ok;
                    const uint32_t slo = cvt_e4m3(__fmul_rn(fmaxf(__fsub_rd(bam, E), 0.0f), idlo));
                    const uint32_t shi = cvt_e4m3(__fmul_rn(__fadd_ru(bam, E), idhi));
                    cert[bk] = !scaled || (d_fast && slo == shi);
                    sfc[bk] = scaled ? shi : 0u;
                    den[bk] = __fmul_rn(e4m3_value(sfc[bk]), s);
                    const bool live = den[bk] > 0.0f;
                    const bool fast = fast_recip_ok(den[bk]);
                    const float rr = fast ? recip_approx(den[bk]) : 0.0f;
                    const float2 rlo = make_float2(__fmul_rd(rr, 1.0f - 0x1p-19f), __fmul_rd(rr, 1.0f - 0x1p-19f));
                    const float2 rhi = make_float2(__fmul_ru(rr, 1.0f + 0x1p-19f), __fmul_ru(rr, 1.0f + 0x1p-19f));
                    // Element codes: both ends of [|w~| - E, |w~| + E], with w~'s sign, 8
                    // elements at a time.
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        float lo8[8], hi8[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 xv = make_float2(x[8 * g + e], x[8 * g + e + 1]);
                            const float2 sE = make_float2(copysignf(E, xv.x), copysignf(E, xv.y));
                            const float2 l = __fmul2_rn(__ffma2_rn(make_float2(-1.0f, -1.0f), sE, xv), rlo);
                            const float2 h = __fmul2_rn(__fadd2_rn(xv, sE), rhi);
                            lo8[e] = l.x;
                            lo8[e + 1] = l.y;
                            hi8[e] = h.x;
                            hi8[e + 1] = h.y;
                        }
                        const uint32_t lw = cvt_e2m1x8(lo8[0], lo8[1], lo8[2], lo8[3], lo8[4], lo8[5], lo8[6], lo8[7]);
                        const uint32_t hw = cvt_e2m1x8(hi8[0], hi8[1], hi8[2], hi8[3], hi8[4], hi8[5], hi8[6], hi8[7]);
                        cw[2 * bk + g] = live ? hw : 0u;
                        diff[2 * bk + g] = !live ? 0u : fast ? (lw ^ hw) : 0xFFFFFFFFu;
                    }
                }
                const bool slow = row_ok && col_ok &&
                                  (!cert[0] || !cert[1] || (diff[0] | diff[1] | diff[2] | diff[3]) != 0u);
                if (__any_sync(0xFFFFFFFFu, slow)) {
                    ok = mbar_wait(&x_full[xs], xph, args.status, abort_flag, kWaitLimitNs);
                    if (!__all_sync(0xFFFFFFFFu, ok)) break;
                    x_read = true;
                    Codes32 r;
                    r.cw[0] = cw[0]; r.cw[1] = cw[1]; r.cw[2] = cw[2]; r.cw[3] = cw[3];
                    r.sfc[0] = sfc[0]; r.sfc[1] = sfc[1];
                    r = quant_fix(tbrow, af, kt0, c, s, d, r, make_uint4(diff[0], diff[1], diff[2], diff[3]),
                                  den[0], den[1], cert[0], cert[1], slow, wt, rloc);
                    cw[0] = r.cw[0]; cw[1] = r.cw[1]; cw[2] = r.cw[2]; cw[3] = r.cw[3];
                    sfc[0] = r.sfc[0]; sfc[1] = r.sfc[1];
                }
                if (col_ok) {
                    if (row_ok)
                        *reinterpret_cast<uint4*>(args.codes + (int64_t)n * (args.K >> 1) + (k0 >> 1)) =
                            make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    if (n < args.rows_pad)
                        *reinterpret_cast<uint16_t*>(
                            args.sf + ((int64_t)(n >> 7) * (args.K >> 6) + (k0 >> 6)) * 512 +
                            (n & 31) * 16 + ((n >> 5) & 3) * 4 + ((k0 >> 5) & 1) * 2) =
                            (uint16_t)(sfc[0] | (sfc[1] << 8));
                }
            }
            // Done with this tile's W and strip of A: every shared-memory read of them has
            // returned (its value was used), and, where the exact chain read them, is
            // fenced against the TMA that will overwrite the slots.
            if (x_read) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&w_empty[ws]);
                mbar_arrive(&x_empty[xs]);
            }
            nb = nb1;
            ks = ks1;
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (kMode == kModeQuant && threadIdx.x == 0) {
        // The last CTA to finish (every CTA has read s_t by now) turns the tensor amax
        // into the per-tensor scale.
        __threadfence();
        if (atomicAdd(args.counter, 1u) == gridDim.x - 1) {
            volatile float* st = args.s_t;
            *st = __fdiv_rn(*st, kAmaxDiv);
        }
    }
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int kMode>
cudaError_t run_merge_tc(const LaunchCtx& ctx, const RequantTcMaps& m, const TcArgs& a) {
    static OccupancyCache occupancy;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // May start before the previous kernel on the stream ends (programmatic dependent
    // launch); the kernel waits (griddepcontrol.wait) before reading its results.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(ctx.num_sms / kPair * kPair), 1, 1);
    int max_clusters = 0;
    const cudaError_t e = clusters_per_device(occupancy, ctx, merge_tc_kernel<kMode>, cfg, &max_clusters);
    if (e != cudaSuccess) return e;
    const int clusters = a.tiles < max_clusters ? a.tiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(clusters * kPair), 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, merge_tc_kernel<kMode>, m.w, m.ap, m.af, a);
}

}  // namespace

size_t requant_tc_workspace_bytes(int w_dtype, int r, int64_t N, int64_t K) {
    const int64_t tiles = (N + kTM * kPair - 1) / (kTM * kPair) * ((K + kTK - 1) / kTK);
    if (w_dtype != NVFP4_W_BF16 || r != kRank || N <= 0 || K <= 0 || tiles >= (int64_t(1) << 30))
        return 0;
    return requant_tc_layout(nullptr, N, K).bytes;
}

cudaError_t launch_requant_tc(const LaunchCtx& ctx, const RequantTcMaps& maps, const float* A,
                              const float* B, void* workspace, float c, int64_t N, int64_t K,
                              uint8_t* codes, uint8_t* sf, float* s_t) {
    const RequantTcLayout ws = requant_tc_layout(workspace, N, K);
    TcArgs a;
    a.c = c;
    a.N = (int)N;
    a.K = (int)K;
    a.rows_pad = (int)((N + 127) / 128 * 128);
    a.codes = codes;
    a.sf = sf;
    a.s_t = s_t;
    a.rnorm = ws.rnorm;
    a.counter = ws.counter;
    a.B = B;
    a.cnorm = ws.cnorm;
    a.status = ctx.status;
    a.zero = 0;
    a.nks = (int)((K + kTK - 1) / kTK);
    a.tiles = (int)((N + kTM * kPair - 1) / (kTM * kPair)) * a.nks;
    const int rows_pad256 = (int)((N + 255) / 256 * 256);
    const int nb_rows = (rows_pad256 + kSplitRows - 1) / kSplitRows;
    const int nb_cols = (int)((K + kSplitCols - 1) / kSplitCols);
    merge_split_kernel<<<(unsigned)(nb_rows + nb_cols), kSplitThreads, 0, ctx.stream>>>(
        A, B, (int)N, (int)K, rows_pad256, nb_rows, ws.ap, ws.rnorm, ws.cnorm, s_t, ws.counter);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = run_merge_tc<kModeAmax>(ctx, maps, a)) != cudaSuccess) return e;
    return run_merge_tc<kModeQuant>(ctx, maps, a);
}

}  // namespace nvfp4rl
