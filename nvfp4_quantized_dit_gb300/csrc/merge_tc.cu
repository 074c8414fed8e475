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
// [w~ - E, w~ + E], widened for the final fma's own rounding:
//   * tensor amax (amax phase, no MMA): with Ecs = |c| ||B[n,:]|| max ||A[:,k]|| (Cauchy-
//     Schwarz, plus the roundings) every |w'| lies within Ecs of |W|; a warp's maximum is
//     among its elements whose |W| + Ecs reaches the largest |W| - Ecs of the warp (or the
//     running tensor amax); those few are merged exactly and the warp's maximum of them
//     goes to the tensor amax;
//   * block scale (quantize phase): the E4M3 codes of both ends of [bam - E, bam + E]
//     must agree, else the block's 16 values are recomputed exactly;
//   * element code (quantize phase): with r ~ 1/den, the two ends x r -+ dl of an
//     interval that holds w'/den (dl per block, from E, the block's largest magnitude
//     and the reciprocal's error) must give the same E2M1 code, else that element alone
//     is recomputed (an interval that holds zero gives codes of both signs and never
//     agrees).
// So codes, scales and s_t are bit-identical to the fp32 chain's.  The exact chain
// reads the fp32 factors and W from global memory (L2).
//
// Kernels.  A split kernel writes A' = [a0 a1 a0 a1] per column of A (bf16, 256 bytes
// per row) into the caller's workspace, with upper bounds of every row norm of B and,
// per 64 columns, of the largest column norm of A.  Then one persistent kernel on
// clusters of two CTAs (one per SM, every CTA resident) runs both phases: the amax phase
// streams W from HBM in contiguous chunks of up to 32 KB (each CTA its first five by
// index, the rest claimed from a counter), keeping it in L2; a grid-wide barrier (a
// counter in the workspace, bounded wait) gathers every CTA's contribution to the
// tensor amax; the quantize phase walks its pair's 256 x 128 tiles, reading W back
// from L2.  Only the epilogue waits at the barrier: the copies and MMAs of the first
// quantize-phase tiles run ahead.  A pair tile is 256 weight rows (128 per CTA) x 128
// columns, walked k-strip first, so the rows of B usually stay the same from one tile
// to the next.  Per CTA, 20 warps:
//   warp 0      copies of W into 5 slots of 32 KB, each freed when the epilogue is done
//               with it: amax-phase chunks (bulk copies, with the row norms of the rows
//               they touch), then quantize-phase tiles (128 x 128 bf16, tensor copies);
//   warp 1      tensor-memory allocation; lane 0 of the even CTA issues the 8 pair MMAs
//               (kind::f16, M = 256, N = 128, A from tensor memory) into a
//               double-buffered accumulator;
//   warp 2      TMA: this CTA's 64 rows of A' (the MMA's B operand; 3 slots),
//               completing on the even CTA's barrier, freed by the MMAs;
//   warp 3      idle;
//   warps 4-19  epilogue: four warps per tensor-memory lane quarter, 32 columns each (a
//               thread owns one weight row in the quantize phase, 32 consecutive weights
//               of a chunk in the amax phase): W (amax phase) or accumulator + W -> w~
//               (quantize phase) -> the amax bound or codes and scales, stored straight
//               to global memory.
// The rows of B live in tensor memory next to the accumulators (lane = row), in two
// buffers for consecutive row blocks, as [b0 b0 b1 b1] bf16 pairs (the MMA's A
// operand); the epilogue warps write the next row block's buffer one tile ahead.  The
// rare undecided elements of the quantize phase are queued (two tiles per thread, in
// shared memory) and merged exactly after the last tile, so that the exact chain's
// latency stays out of the pair's tile pipeline; their provisional codes are then
// overwritten.
// Every wait, the grid barrier's included, is bounded (mbar_wait).
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
constexpr int kWSlots = 5, kOpSlots = 3;
constexpr uint32_t kOpBBytes = (kTK / kPair) * kJp * 2;  // 16 KB: A' rows, two 64-column atoms
constexpr uint32_t kWBox = kTM * 128;                    // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kWBytes = 2 * kWBox;                  // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kMiscBytes = 512;
constexpr int kDefer = 512;  // deferred (thread, tile) entries per CTA, exact work after the tile loop
constexpr int kStatic = kWSlots;  // amax tiles a CTA takes by index (the rest from a counter)
constexpr uint32_t kDeferBytes = kDefer * 16;  // (tile, element mask, row | chunk | flags, task base)
constexpr int kTasks = 1024;  // exact values computed for the deferred entries (one per element)
constexpr uint32_t kTaskBytes = kTasks * (2 + 4);  // task (entry << 5 | column) and its exact value
// Per W slot, the tile's bounds (bulk copies beside the W tile).  Quantize phase: the
// 128 row norms of this CTA's rows of B and the 4 column-norm entries of the tile's
// 128-column strip (kSideQBytes).  Amax phase: the row norms of the rows the chunk
// touches (at most kChunkRows + 2, from a 16-byte aligned row on).
constexpr uint32_t kSideQBytes = kTM * 4 + 16;
constexpr int kChunkRows = 128;  // a chunk spans at most this many whole rows
constexpr uint32_t kSideBytes = (kChunkRows + 2 + 3 + 3) / 4 * 16;  // 544
static_assert(kSideBytes >= kSideQBytes && kSideBytes % 16 == 0, "side area");
constexpr uint32_t kSmemBytes =
    1024 + kOpSlots * kOpBBytes + kWSlots * kWBytes + kWSlots * kSideBytes + kDeferBytes + kTaskBytes + kMiscBytes;
// Tensor memory: two accumulators of 128 columns, then two row buffers of 64 columns of
// [b0 b0 b1 b1] (bf16 pairs).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRowBuf0 = 2 * kTK, kRowBufCols = 64;
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kEvenCta = 0x1;
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kSplitThreads = 256;
constexpr int kSplitRows = kSplitThreads / 4;  // rows of B per split block (4 threads a row)
constexpr int kSplitCols = kSplitThreads / 4;  // columns of A per split block (4 threads a column)
// Registers: launched at 96 per thread (20 warps, 5 per scheduler); the control warp
// group drops to 32 and the epilogue warp groups rise to 112 (4 x 32 + 16 x 112 <=
// 20 x 96).
constexpr uint32_t kRegsCtl = 56, kRegsEpi = 104;
static_assert(4 * kRegsCtl + kEpiWarps * kRegsEpi <= (uint32_t)(kThreads / 32) * 96, "register split");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kDefer <= 2048, "a task names its entry in 11 bits");
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
    float* s_t;  // amax phase: amax accumulator (fp32 bits, atomicMax); quantize phase: reads it
    const float* rnorm;  // [N padded to 256] upper bounds of ||B[n,:]||_2 (0 past N)
    const float* B;      // [N, 32] fp32
    const float* A;      // [32, K] fp32
    const uint16_t* W;   // [N, K] bf16 bits
    const float* cnorm;  // [K/128][4]: per 128-column strip, the largest ||A[:,k]||_2
                         // of each 64-column half (upper bounds), then 2 unused
    unsigned int* counter;  // CTAs that are done (zeroed by the split)
    unsigned int* arrive;   // CTAs past the amax phase: the grid barrier (zeroed by the split)
    unsigned int* next;     // the amax phase's next dynamically taken tile (zeroed by the split)
    int units;              // amax-phase chunks: ceil(N K / chunk) contiguous pieces of W
    int chunk;              // elements per amax chunk: min(16384, 128 K) (at most 32 KB)
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
// Block 0 also clears the amax accumulator s_t and the fused kernel's counters
// (counter[0]: CTAs done; counter[1]: CTAs past the amax phase; counter[2]: the amax
// phase's next dynamic tile; counter[3], counter[4]: elements merged by the exact chain
// in the quantize and the amax phase, a diagnostic).
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
        counter[0] = 0u;
        counter[1] = 0u;
        counter[2] = 0u;
        counter[3] = 0u;
        counter[4] = 0u;
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

// The quantize phase's exact path for one thread's 32 weights W[n, k0 .. k0 + 31],
// everything read from global memory (the row of B, the columns of A, the bf16 W):
// blocks whose scale is undecided (fix0, fix1) get their 16 values from the exact chain
// (16 chains side by side), then the scale and codes by true divisions; the elements
// marked in um (one bit per column, in blocks with a decided scale) get their code from
// the exact chain and a true division.  r holds the codes and scale codes decided so far.
struct Codes32 {
    uint32_t cw[4];
    uint32_t sfc[2];
};
__device__ __noinline__ Codes32 quant_fix(const float* brow, const float* A, int K, int k0, const uint16_t* wrow,
                                         float c, float s, float d, Codes32 r, uint32_t um, bool fix0, bool fix1) {
    uint32_t bq[kRank];
#pragma unroll
    for (int j = 0; j < kRank; j += 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(brow + j));
        bq[j] = v.x;
        bq[j + 1] = v.y;
        bq[j + 2] = v.z;
        bq[j + 3] = v.w;
    }
#pragma unroll 1
    for (int bk = 0; bk < 2; ++bk) {
        if (!(bk == 0 ? fix0 : fix1)) continue;
        const int kk = k0 + 16 * bk;
        float x16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x16[e] = 0.0f;
#pragma unroll 1
        for (int j0 = 0; j0 < kRank; j0 += 4) {
            // 4 rows of A's 16 columns in flight at once, then their FMAs in chain order.
            float4 v[4][4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    v[jj][q4] = __ldg(reinterpret_cast<const float4*>(A + (int64_t)(j0 + jj) * K + kk) + q4);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const float bj = __uint_as_float(bq[j0 + jj]);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    x16[4 * q4] = __fmaf_rn(bj, v[jj][q4].x, x16[4 * q4]);
                    x16[4 * q4 + 1] = __fmaf_rn(bj, v[jj][q4].y, x16[4 * q4 + 1]);
                    x16[4 * q4 + 2] = __fmaf_rn(bj, v[jj][q4].z, x16[4 * q4 + 2]);
                    x16[4 * q4 + 3] = __fmaf_rn(bj, v[jj][q4].w, x16[4 * q4 + 3]);
                }
            }
        }
        float bam = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            x16[e] = __fmaf_rn(c, x16[e], __uint_as_float((uint32_t)wrow[16 * bk + e] << 16));
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
    if (fix0) um &= 0xFFFF0000u;
    if (fix1) um &= 0x0000FFFFu;
    const float den0 = __fmul_rn(e4m3_value(r.sfc[0]), s), den1 = __fmul_rn(e4m3_value(r.sfc[1]), s);
#pragma unroll 1
    while (um != 0u) {
        const int e = __ffs((int)um) - 1;
        um &= um - 1u;
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < kRank; ++j)
            acc = __fmaf_rn(__uint_as_float(bq[j]), __ldg(A + (int64_t)j * K + k0 + e), acc);
        const float x = __fmaf_rn(c, acc, __uint_as_float((uint32_t)wrow[e] << 16));
        const float den = e < 16 ? den0 : den1;
        const uint32_t code =
            den > 0.0f ? cvt_e2m1x8(__fdiv_rn(x, den), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu : 0u;
        const uint32_t sh = 4u * (uint32_t)(e & 7), keep = ~(0xFu << sh);
        const int wi = e >> 3;
        if (wi == 0) r.cw[0] = (r.cw[0] & keep) | (code << sh);
        else if (wi == 1) r.cw[1] = (r.cw[1] & keep) | (code << sh);
        else if (wi == 2) r.cw[2] = (r.cw[2] & keep) | (code << sh);
        else r.cw[3] = (r.cw[3] & keep) | (code << sh);
    }
    return r;
}

// The byte address of the two scale bytes of row n, columns k0 .. k0 + 31 (k0 % 32 == 0)
// in the 128x4 blocked layout.
__device__ __forceinline__ int64_t sf_pair_offset(int n, int k0, int K) {
    return ((int64_t)(n >> 7) * (K >> 6) + (k0 >> 6)) * 512 + (n & 31) * 16 + ((n >> 5) & 3) * 4 +
           ((k0 >> 5) & 1) * 2;
}

// Loads this thread's 8 of the 32 values of B's row n (8 chunk .. 8 chunk + 7; zeros past N).
__device__ __forceinline__ void load_brow8(const TcArgs& args, int n, int chunk, float (&v)[8]) {
    if (n < args.N) {
        const float4* src = reinterpret_cast<const float4*>(args.B + (int64_t)n * kRank + 8 * chunk);
        const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    } else {
#pragma unroll
        for (int z = 0; z < 8; ++z) v[z] = 0.0f;
    }
}

// Writes a row block's rows of B into row buffer nrb & 1 of tensor memory (this warp's 8
// of the 32 columns, v, for its 32 rows, as the bf16 parts the MMA reads) and reports it
// to the MMA issuer (rows_ready, on the even CTA).  The buffer's previous row block was
// used only by MMAs of tiles this warp has already waited for, so no other wait is needed.
__device__ __forceinline__ void write_rows(uint32_t tmem_base, uint32_t tlane, uint32_t rows_ready_even, int chunk,
                                           int lane, int& nrb, const float (&v)[8]) {
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
    tmem_st_wait();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(rows_ready_even + 8u * (uint32_t)(nrb & 1));
    ++nrb;
}

// The library's merged value W'[n, k] (the fp32 fma chain, in order), everything from
// global memory: one round of loads (the row of B, the column of A, W).  Out of line:
// its 64 loaded values stay out of the callers' register budget.
__device__ __noinline__ float exact_element(const TcArgs& args, int n, int k, float c) {
    float bv[kRank], av[kRank];
#pragma unroll
    for (int j = 0; j < kRank; j += 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(args.B + (int64_t)n * kRank + j));
        bv[j] = v.x;
        bv[j + 1] = v.y;
        bv[j + 2] = v.z;
        bv[j + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < kRank; ++j) av[j] = __ldg(args.A + (int64_t)j * args.K + k);
    const float w = __uint_as_float((uint32_t)__ldg(args.W + (int64_t)n * args.K + k) << 16);
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kRank; ++j) acc = __fmaf_rn(bv[j], av[j], acc);
    return __fmaf_rn(c, acc, w);
}

// The pair's quantize-phase tiles: the range [t_begin, t_end), walked backwards
// (tile(T + j) for j = 0 .. T - 1).  Tile t is row block t / nks (256 rows, the pair's),
// 128-column strip t % nks.
struct TileSeq {
    int t_begin, t_end, T;
    __device__ __forceinline__ int tile(int i) const { return i < T ? t_begin + i : t_end - 1 - (i - T); }
};

// This thread's 32 weights W[n, k0 .. k0 + 31] (read from global memory, all four 16-byte
// loads in flight at once): the largest |W'| of those whose bound |W| + Ecs reaches thr.
__device__ __forceinline__ float amax_recheck(const TcArgs& args, int n, int k0, float Ecs, float c, float thr,
                                              unsigned int* xcnt) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const uint4*>(args.W + (int64_t)n * args.K + k0) + u);
    float em = 0.0f;
#pragma unroll 1
    for (int e = 0; e < 32; ++e) {
        const uint4 q = e < 8 ? v[0] : e < 16 ? v[1] : e < 24 ? v[2] : v[3];
        const int h = (e & 7) >> 1;
        const uint32_t wd = h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w;
        const float a = __uint_as_float(((e & 1) ? wd : wd << 16) & 0x7FFF0000u);
        if (__fadd_ru(__fmul_ru(a, 1.0f + 0x1p-23f), Ecs) < thr) continue;
        atomicAdd(xcnt, 1u);
        em = fmaxf(em, fabsf(exact_element(args, n, k0 + e, c)));
    }
    return em;
}

// The end of the amax phase for one epilogue thread: the largest |W'| among the
// elements that can still be the tensor amax, i.e. whose bound reaches s_t now: this
// thread's 32 weights of the CTA's seed tile (its first, whose candidates were not
// queued; bound U0, slack E0, skipped when U0 < 0), and the queued candidates (entries
// et, et + 512, ...; what did not fit in the queue was merged in place).
__device__ __noinline__ float amax_candidates(const TcArgs& args, const uint4* defq, const unsigned int* defn,
                                              int n0, int k00, float U0, float E0, float c, int et,
                                              unsigned int* xcnt) {
    const float st_seen = *reinterpret_cast<volatile const float*>(args.s_t);
    float em = 0.0f;
    if (U0 >= st_seen) em = amax_recheck(args, n0, k00, E0, c, st_seen, xcnt);
    const unsigned int nc = min(*reinterpret_cast<volatile const unsigned int*>(defn), (unsigned int)kDefer);
    for (unsigned int z = (unsigned int)et; z < nc; z += kEpiWarps * 32) {
        const uint4 dq = defq[z];
        if (__uint_as_float(dq.z) >= st_seen) {
            atomicAdd(xcnt, 1u);
            em = fmaxf(em, fabsf(exact_element(args, (int)dq.x, (int)dq.y, c)));
        }
    }
    return em;
}

__global__ void __launch_bounds__(kThreads, 1)
    merge_fused_kernel(const __grid_constant__ CUtensorMap tmap_w,
                       const __grid_constant__ CUtensorMap tmap_ap, const TcArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* opB = smem;                          // [kOpSlots]: A' rows of this CTA's 64 columns
    uint8_t* wring = opB + kOpSlots * kOpBBytes;  // [kWSlots]: W tiles
    uint8_t* side = wring + kWSlots * kWBytes;                           // [kWSlots]: tile bounds
    uint4* defq = reinterpret_cast<uint4*>(side + kWSlots * kSideBytes);  // [kDefer] the CTA's deferred work
    float* task_val = reinterpret_cast<float*>(defq + kDefer);           // [kTasks]
    uint16_t* task_id = reinterpret_cast<uint16_t*>(task_val + kTasks);  // [kTasks]
    uint64_t* bars = reinterpret_cast<uint64_t*>(task_id + kTasks);
    uint64_t* w_full = bars;                         // [kWSlots]
    uint64_t* w_empty = w_full + kWSlots;            // [kWSlots] the 16 epilogue warps
    uint64_t* op_full = w_empty + kWSlots;           // [kOpSlots] even CTA: both CTAs' A'
    uint64_t* op_empty = op_full + kOpSlots;         // [kOpSlots] the pair's MMAs are done
    uint64_t* tmem_full = op_empty + kOpSlots;       // [2]
    uint64_t* tmem_empty = tmem_full + 2;            // [2] even CTA
    uint64_t* rows_ready = tmem_empty + 2;           // [2] even CTA: a row buffer is written
    uint64_t* drain = rows_ready + 2;
    uint64_t* epi_done = drain + 1;                  // the 16 epilogue warps finished the amax phase
    uint64_t* amax_ready = epi_done + 1;             // the tensor amax is in amax_smem
    uint64_t* loop_done = amax_ready + 1;            // the 16 epilogue warps left the tile loop
    uint64_t* tasks_ready = loop_done + 1;           // ... listed the deferred elements
    uint64_t* vals_ready = tasks_ready + 1;          // ... computed their exact values
    uint64_t* cand_done = vals_ready + 1;            // ... queued their amax candidates
    uint64_t* ra_ready = cand_done + 1;              // ... contributed to ra_all
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ra_ready + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile float* amax_smem = reinterpret_cast<volatile float*>(tmem_slot + 2);
    unsigned int* defn = tmem_slot + 3;              // entries pushed to defq
    unsigned int* ntask = tmem_slot + 4;             // elements claimed in task_id (may pass kTasks)
    unsigned int* p0_overflow = tmem_slot + 5;       // the amax phase's queue overflowed
    unsigned int* p1_overflow = tmem_slot + 6;       // the quantize phase's queue overflowed
    volatile int* slot_unit = reinterpret_cast<volatile int*>(tmem_slot + 7);  // [kWSlots] amax chunk per slot
    unsigned int* xcount = tmem_slot + 7 + kWSlots;  // [2] exact merges: quantize (whole blocks), amax
    // The end of the listed tasks: the entries that fit occupy task_id[0, nfill) (the
    // first entry that does not fit, and every later one, claims past kTasks).
    unsigned int* nfill = tmem_slot + 9 + kWSlots;
    volatile int* slot_n0 = reinterpret_cast<volatile int*>(tmem_slot + 10 + kWSlots);  // [kWSlots] chunk's row
    volatile int* slot_r0 = slot_n0 + kWSlots;  // [kWSlots] and column of its first element
    float* ra_all = reinterpret_cast<float*>(tmem_slot + 10 + 3 * kWSlots);  // max_k ||A[:,k]|| bound

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x / kPair), npairs = (int)(gridDim.x / kPair);
    TileSeq seq;
    seq.t_begin = (int)((int64_t)pair * args.tiles / npairs);
    seq.t_end = (int)((int64_t)(pair + 1) * args.tiles / npairs);
    seq.T = seq.t_end - seq.t_begin;
    const int nks = args.nks;
    // The W ring's iterations: first the amax phase's tiles (128 rows x 128 columns: this
    // CTA's kStatic tiles blockIdx.x + m gridDim.x, then tiles taken from a counter; a
    // sentinel slot, unit -1, ends the phase), then the quantize phase's T tiles of the
    // pair.  Producer and epilogue count the amax iterations (F) the same way.

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWSlots; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kOpSlots; ++i) {
            mbar_init(&op_full[i], 1);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tmem_full[i], 1);
            mbar_init(&tmem_empty[i], kEpiWarps * kPair);
            mbar_init(&rows_ready[i], kEpiWarps * kPair);
        }
        mbar_init(drain, 1);
        mbar_init(epi_done, kEpiWarps);
        mbar_init(amax_ready, 1);
        mbar_init(loop_done, kEpiWarps);
        mbar_init(tasks_ready, kEpiWarps);
        mbar_init(vals_ready, kEpiWarps);
        mbar_init(cand_done, kEpiWarps);
        mbar_init(ra_ready, kEpiWarps);
        *abort_flag = 0;
        *amax_smem = 0.0f;
        *defn = 0u;
        *ntask = 0u;
        *p0_overflow = 0u;
        *p1_overflow = 0u;
        xcount[0] = 0u;
        xcount[1] = 0u;
        *nfill = 0u;
        *ra_all = 0.0f;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmap_w);
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
            // ------------------------------------------------ TMA: W
            // Amax phase: contiguous chunks of W (args.chunk elements, one bulk copy each),
            // kept in L2 (evict_last) for the quantize phase, whose 128 x 128 tiles (tensor
            // copies) let them go (evict_first).  Each W slot also receives bounds written by
            // the split kernel: for a chunk, the row norms of the rows it touches; the first
            // kStatic chunks are requested at once, their bounds once the split kernel is
            // done.
            const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
            const int G = (int)gridDim.x;
            const int64_t NK = (int64_t)args.N * args.K;
            const int rows_pad256 = (args.N + 255) / 256 * 256;
            int i = 0, nstatic = 0;
            bool ended = false;
            uint32_t side_bytes[kStatic];
            // Requests chunk u into slot ws; returns the bytes of its row-norm slice.
            auto issue_w = [&](int ws, int u) -> uint32_t {
                const int64_t e0 = (int64_t)u * args.chunk;
                const uint32_t bytes = (uint32_t)min((int64_t)args.chunk, NK - e0) * 2u;
                const int n0 = (int)(e0 / args.K);
                const int n_last = (int)((e0 + bytes / 2 - 1) / args.K);
                const int n0a = n0 & ~3;
                const uint32_t sb = (uint32_t)min((n_last - n0a + 4) & ~3, rows_pad256 - n0a) * 4u;
                slot_unit[ws] = u;
                slot_n0[ws] = n0;
                slot_r0[ws] = (int)(e0 - (int64_t)n0 * args.K);
                mbar_arrive_expect_tx(&w_full[ws], bytes + sb);
                bulk_load_hint(wring + ws * kWBytes, args.W + e0, bytes, &w_full[ws], keep);
                return sb;
            };
            auto issue_side_rows = [&](int ws, uint32_t sb) {
                bulk_load(side + ws * kSideBytes, args.rnorm + (slot_n0[ws] & ~3), sb, &w_full[ws]);
            };
            auto issue_side = [&](int ws, int row0, int ks) {
                uint8_t* sd = side + ws * kSideBytes;
                bulk_load(sd, args.rnorm + row0, kTM * 4, &w_full[ws]);
                bulk_load(sd + kTM * 4, args.cnorm + ks * 4, 16, &w_full[ws]);
            };
            for (; i < kStatic && !ended; ++i) {
                if (!mbar_wait(&w_empty[i], 1u, args.status, abort_flag, kWaitLimitNs)) break;
                const int u = (int)blockIdx.x + i * G;
                if (u >= args.units) {
                    slot_unit[i] = -1;
                    mbar_arrive(&w_full[i]);
                    ended = true;
                } else {
                    side_bytes[i] = issue_w(i, u);
                    ++nstatic;
                }
            }
            grid_dep_wait();  // the norms and the chunk counter are written by the split kernel
            for (int z = 0; z < nstatic; ++z) issue_side_rows(z, side_bytes[z]);
            // Each unit is claimed before its slot is free (the claim's round trip overlaps
            // the wait).
            int u_next = ended ? args.units : kStatic * G + (int)atomicAdd(args.next, 1u);
            for (; !ended && !*abort_flag; ++i) {
                const int ws = i % kWSlots;
                const int u = u_next;
                if (u < args.units) u_next = kStatic * G + (int)atomicAdd(args.next, 1u);
                if (!mbar_wait(&w_empty[ws], (uint32_t)((i / kWSlots) & 1) ^ 1u, args.status, abort_flag,
                               kWaitLimitNs))
                    break;
                if (u >= args.units) {
                    slot_unit[ws] = -1;
                    mbar_arrive(&w_full[ws]);
                    ended = true;
                } else {
                    issue_side_rows(ws, issue_w(ws, u));
                }
            }
            // i = the amax iterations, the sentinel's included; the quantize phase's
            // tiles follow in the ring.
            for (int j = 0; ended && j < seq.T && !*abort_flag; ++j, ++i) {
                const int ws = i % kWSlots;
                if (!mbar_wait(&w_empty[ws], (uint32_t)((i / kWSlots) & 1) ^ 1u, args.status, abort_flag,
                               kWaitLimitNs))
                    break;
                const int t = seq.tile(seq.T + j);
                const int nb = t / nks, ks = t - nb * nks;
                const int row0 = nb * (kTM * kPair) + (int)rank * kTM;
                // A quantize-phase tile of W (from L2), and its bounds.
                mbar_arrive_expect_tx(&w_full[ws], kWBytes + kSideQBytes);
                tma_load_2d_hint(&tmap_w, &w_full[ws], wring + ws * kWBytes, ks * kTK, row0, drop);
                tma_load_2d_hint(&tmap_w, &w_full[ws], wring + ws * kWBytes + kWBox, ks * kTK + 64, row0, drop);
                issue_side(ws, row0, ks);
            }
            if (!*abort_flag) {
                // Tail: the last tiles of W land before exit.
                for (int j = (i >= kWSlots ? i - kWSlots : 0); j < i; ++j)
                    if (!mbar_wait(&w_full[j % kWSlots], (uint32_t)((j / kWSlots) & 1), args.status,
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
            // The quantize phase's tiles only (the amax phase takes no MMA).
            grid_dep_wait();  // A' is written by the split kernel
            const uint32_t op_full_even = map_to_rank(smem_u32(op_full), 0);
            int i = 0;
            for (; i < seq.T; ++i) {
                const int t = seq.tile(seq.T + i);
                const int ks = t - (t / nks) * nks;
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
            int rb = -1, nrb = 0;  // row block in use, row buffers filled
            for (int i = 0; i < seq.T; ++i) {  // the quantize phase's tiles
                const int t = seq.tile(seq.T + i);
                const int nb = t / nks;
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
        const int et = (int)threadIdx.x - kEpiWarp0 * 32;   // 0..511
        const uint32_t tlane = (uint32_t)(q * 32) << 16;
        const uint32_t rows_ready_even = map_to_rank(smem_u32(rows_ready), 0);
        const uint32_t tmem_empty_even = map_to_rank(smem_u32(tmem_empty), 0);
        const float c = args.c, ac = fabsf(args.c);
        float s = 0.0f, d = 0.0f, idlo = 0.0f, idhi = 0.0f;
        bool d_fast = false;
        int nrb = 0;           // row buffers written
        grid_dep_wait();       // the split kernel's results (norms, s_t, the counters)
        // In the amax phase, the running lower bound of the tensor amax (any value s_t has
        // held is one), read before each tile's wait for its data (the load's round trip
        // overlaps the wait).
        float st_now = 0.0f;
        int cur_buf = 0;  // row buffer of the current tile's row block (quantize phase)
        bool alive = true;
        // ---- amax phase: one chunk of W per slot until the sentinel (unit -1).  Thread
        // et takes the chunk's elements 32 et .. 32 et + 31 (row n, columns k0 ..; K is a
        // multiple of 64, so they never straddle a row).  With rb >= ||B[n,:]|| (the
        // slot's row norms) and ra >= max_k ||A[:,k]|| every |w'| lies within
        //   Ecs = |c| rb ra (1 + 2^-17) + 2^-126
        // of |W| (Cauchy-Schwarz; the slack covers the chain's rounding, the final fma's
        // beyond 2^-23 |W|, and subnormal roundings).
        {
            // ra: the largest column-norm entry (the split kernel wrote one per 64 columns).
            float m = 0.0f;
            for (int i = et; i < args.K / 64; i += kEpiWarps * 32) m = fmaxf(m, args.cnorm[(i >> 1) * 4 + (i & 1)]);
            m = warp_max_f(m);
            if (lane == 0) {
                atomicMax(reinterpret_cast<unsigned int*>(ra_all), __float_as_uint(m));
                mbar_arrive(ra_ready);
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(ra_ready, 0, args.status, abort_flag, kWaitLimitNs))) alive = false;
        }
        const float ra = *reinterpret_cast<volatile float*>(ra_all);
        int F = 0;                            // amax iterations, the sentinel's included
        float seed_U = -1.0f, seed_E = 0.0f;  // the first tile's largest bound and Ecs
        int seed_n = 0, seed_k0 = 0;
        auto amax_tile = [&](int i, bool slow_mode) -> int {  // 0: phase over, 1: done, 2: redo
            const int ws = i % kWSlots;
            const uint8_t* wt = wring + ws * kWBytes;  // this tile's W, held until its end
            const float st_pre = *reinterpret_cast<volatile const float*>(args.s_t);
            bool ok = mbar_wait(&w_full[ws], (uint32_t)((i / kWSlots) & 1), args.status, abort_flag, kWaitLimitNs);
            if (!__all_sync(0xFFFFFFFFu, ok)) return 0;
            const int u = slot_unit[ws];
            if (u < 0) {  // the sentinel: the phase ends here
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);
                F = i + 1;
                return 0;
            }
            const int n0 = slot_n0[ws];
            const int off = slot_r0[ws] + 32 * et;  // < K + chunk
            const int q = off / args.K;
            const int n = n0 + q;
            const int k0 = off - q * args.K;
            const bool in = 32 * et < args.chunk && (int64_t)u * args.chunk + 32 * et < (int64_t)args.N * args.K;
            const float rb = in ? reinterpret_cast<const float*>(side + ws * kSideBytes)[n - (n0 & ~3)] : 0.0f;
            const float Ecs = __fadd_ru(__fmul_ru(__fmul_ru(ac, __fmul_ru(rb, ra)), 1.0f + 0x1p-17f), 0x1p-126f);
            uint4 wr[4];
            {
                const uint4* wb = reinterpret_cast<const uint4*>(wt) + 4 * et;
#pragma unroll
                for (int z = 0; z < 4; ++z) wr[z] = wb[z];
            }
            uint32_t mx = 0u;  // bf16 magnitudes order like their bit patterns
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                mx = __vmaxu2(mx, wr[z].x & 0x7FFF7FFFu);
                mx = __vmaxu2(mx, wr[z].y & 0x7FFF7FFFu);
                mx = __vmaxu2(mx, wr[z].z & 0x7FFF7FFFu);
                mx = __vmaxu2(mx, wr[z].w & 0x7FFF7FFFu);
            }
            const float mW = in ? __uint_as_float(max(mx & 0xFFFFu, mx >> 16) << 16) : 0.0f;
            // A lower bound of the tensor amax from this warp's weights.
            const float lo = warp_max_f(fmaxf(__fsub_rd(__fmul_rd(mW, 1.0f - 0x1p-23f), Ecs), 0.0f));
            st_now = fmaxf(st_now, st_pre);
            const float thr = fmaxf(lo, st_now);
            const float U_t = __fadd_ru(__fmul_ru(mW, 1.0f + 0x1p-23f), Ecs);
            // Only weights with |W| + Ecs at the threshold can be the maximum: queued for
            // the end of the phase (when the threshold is higher still), or, in slow mode,
            // merged here.  The CTA's first tile only publishes its bound (the threshold is
            // low then); it is checked again at the end.
            if (i == 0 && in) {
                seed_U = U_t;
                seed_E = Ecs;
                seed_n = n;
                seed_k0 = k0;
            }
            const bool cand = in && i > 0 && U_t >= thr;
            bool full = false;
            if (__any_sync(0xFFFFFFFFu, cand) && cand) {
                float em = 0.0f;
#pragma unroll 1
                for (int z = 0; z < 4; ++z) {
                    const uint32_t rw[4] = {wr[z].x, wr[z].y, wr[z].z, wr[z].w};
#pragma unroll 1
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t wd = (e >> 1) == 0 ? rw[0] : (e >> 1) == 1 ? rw[1] : (e >> 1) == 2 ? rw[2] : rw[3];
                        const float a = __uint_as_float(((e & 1) ? wd : wd << 16) & 0x7FFF0000u);
                        const float U = __fadd_ru(__fmul_ru(a, 1.0f + 0x1p-23f), Ecs);
                        if (U < thr) continue;
                        const int k = k0 + 8 * z + e;
                        if (slow_mode) {
                            atomicAdd(&xcount[1], 1u);
                            em = fmaxf(em, fabsf(exact_element(args, n, k, c)));
                        } else {
                            const unsigned int slot = atomicAdd(defn, 1u);
                            if (slot < (unsigned int)kDefer)
                                defq[slot] = make_uint4((uint32_t)n, (uint32_t)k, __float_as_uint(U), 0u);
                            else
                                full = true;
                        }
                    }
                }
                if (em > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(args.s_t), __float_as_uint(em));
            }
            if (__any_sync(0xFFFFFFFFu, full)) {
                // The queue is full: this tile is done again, and the rest of the phase, in
                // slow mode (the slot is not released yet).
                if (lane == 0) *p0_overflow = 1u;
                return 2;
            }
            // |W'| >= 0: the fp32 bit patterns order like the values.
            if (lane == 0 && lo > st_now) atomicMax(reinterpret_cast<unsigned int*>(args.s_t), __float_as_uint(lo));
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[ws]);
            return 1;
        };
        int resume = -1;
        // Loop conditions are voted on by the warp (warp_flag): amax_tile is collective.
        for (int i = 0; alive && !warp_flag(abort_flag); ++i) {
            const int r = amax_tile(i, false);
            if (r == 0) break;
            if (r == 2 || warp_flag(reinterpret_cast<volatile unsigned int*>(p0_overflow))) {
                resume = r == 2 ? i : i + 1;
                break;
            }
        }
        if (resume >= 0) {
            // Slow mode (the queue filled, in this warp or another): from the tile that
            // overflowed (or the next one), candidates are merged in place.
            __syncwarp();
            for (int i = resume; !warp_flag(abort_flag); ++i)
                if (amax_tile(i, true) == 0) break;
        }
        if (warp_flag(abort_flag)) alive = false;
        if (alive) {
            // ---- between the phases.  First the queued amax candidates (elements
            // whose bound reached the running threshold when their chunk was read):
            // those whose bound still reaches the current tensor amax bound are merged
            // exactly (one round of loads each) and their maximum goes to s_t.
            __syncwarp();
            if (lane == 0) mbar_arrive(cand_done);
            if (!mbar_wait(cand_done, 0, args.status, abort_flag, kWaitLimitNs)) alive = false;
            {
                const float em = warp_max_f(amax_candidates(args, defq, defn, seed_n, seed_k0, seed_U, seed_E, c, et,
                                                                        &xcount[1]));
                if (lane == 0 && em > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(args.s_t), __float_as_uint(em));
            }
            // Then every CTA's contributions are in s_t: each warp's atomics are fenced,
            // the warp reports to epi_done, one thread joins the grid-wide count
            // (bounded wait) and reads the amax.
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_done);
            if (warp == kEpiWarp0 && lane == 0) {
                bool ok = mbar_wait(epi_done, 0, args.status, abort_flag, kWaitLimitNs);
                float amax = 0.0f;
                if (ok) {
                    *defn = 0u;  // the queue now collects the quantize phase's deferred work
                    __threadfence();
                    atomicAdd(args.arrive, 1u);
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(args.arrive) < gridDim.x) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            atomicCAS(args.status, 0, (int)NVFP4_ERR_TIMEOUT);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (ok) amax = __uint_as_float(ld_acquire_gpu(reinterpret_cast<const unsigned int*>(args.s_t)));
                }
                *amax_smem = amax;
                mbar_arrive(amax_ready);
            }
            const bool ok = mbar_wait(amax_ready, 0, args.status, abort_flag, kWaitLimitNs);
            if (!__all_sync(0xFFFFFFFFu, ok) || warp_flag(abort_flag)) alive = false;
            const float amax = *amax_smem;
            s = __fdiv_rn(amax, kAmaxDiv);
            d = __fmul_rn(6.0f, s);
            d_fast = fast_recip_ok(d);
            const float rd = d_fast ? recip_approx(d) : 0.0f;
            idlo = __fmul_rd(rd, 1.0f - 0x1p-19f);
            idhi = __fmul_ru(rd, 1.0f + 0x1p-19f);
            // The first quantize-phase tile's rows of B (buffer 0), for the MMAs.
            if (alive) {
                float bfirst[8];
                load_brow8(args, (seq.tile(seq.T) / nks) * (kTM * kPair) + (int)rank * kTM + rloc, chunk, bfirst);
                write_rows(tmem_base, tlane, rows_ready_even, chunk, lane, nrb, bfirst);
            }
        }
        // ---- quantize phase: tile j of the pair (walked backwards)
        for (int j = 0; alive && j < seq.T && !warp_flag(abort_flag); ++j) {
            const int i = F + j;
            const int ws = i % kWSlots;
            const uint8_t* wt = wring + ws * kWBytes;  // this tile's W, held until its end
            const int t = seq.tile(seq.T + j);
            const int nb = t / nks, ks = t - nb * nks;
            const int n = nb * (kTM * kPair) + (int)rank * kTM + rloc;
            const int k0 = ks * kTK + kt0;        // this warp's first column in W
            const bool row_ok = n < args.N;
            const bool col_ok = k0 < args.K;      // K is a multiple of 64: all 32 columns or none
            int nb1 = nb;
            if (j + 1 < seq.T) {
                nb1 = seq.tile(seq.T + j + 1) / nks;
                // The next tile starts a new row block: write its rows one tile ahead.
                if (nb1 != nb) {
                    float b1[8];
                    load_brow8(args, nb1 * (kTM * kPair) + (int)rank * kTM + rloc, chunk, b1);
                    write_rows(tmem_base, tlane, rows_ready_even, chunk, lane, nrb, b1);
                }
            }
            uint4 wr[4];  // this thread's 32 weights (bf16)
            {
                const int b = j & 1;
                const uint32_t ph = (uint32_t)((j >> 1) & 1);
                if (nb1 != nb) cur_buf ^= 1;  // from the next tile on
                // The accumulator's 32 columns (released at once) and this thread's 32 weights.
                bool ok = mbar_wait(&tmem_full[b], ph, args.status, abort_flag, kWaitLimitNs) &&
                          mbar_wait(&w_full[ws], (uint32_t)((i / kWSlots) & 1), args.status, abort_flag,
                                    kWaitLimitNs);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after_sync();
                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + tlane + (uint32_t)(b * kTK + kt0), acc);
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
                const float rb = reinterpret_cast<const float*>(side + ws * kSideBytes)[rloc];
                const float ra = reinterpret_cast<const float*>(side + ws * kSideBytes + kTM * 4)[(k0 >> 6) & 1];
                float E;
                {
                    const float rel = __fmul_ru(__fmul_ru(ac, 0x1p-14f), __fmul_ru(rb, ra));
                    const float abs_ = __fmul_ru(ac, __fmaf_ru(0x1p-120f, __fadd_ru(rb, ra), 0x1p-117f));
                    E = fmaxf(__fadd_ru(rel, abs_), 0x1p-149f);
                }
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
                    const float Ek = Eb;
                    const float* x = wv + 16 * bk;
                    float bam = 0.0f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) bam = fmaxf(bam, fabsf(x[e]));
                    // Block scale: both ends of [bam - E, bam + E] must give the same code.
                    // Rows past N are scale padding (not part of W): scale 0, no codes.
                    const bool scaled = d > 0.0f && row_ok;
                    const float X = __fadd_ru(bam, Ek);  // >= |w'| and |w~| of every element
                    const uint32_t slo = cvt_e4m3(__fmul_rn(fmaxf(__fsub_rd(bam, Ek), 0.0f), idlo));
                    const uint32_t shi = cvt_e4m3(__fmul_rn(X, idhi));
                    cert[bk] = !scaled || (d_fast && slo == shi);
                    sfc[bk] = scaled ? shi : 0u;
                    den[bk] = __fmul_rn(e4m3_value(sfc[bk]), s);
                    const bool live = den[bk] > 0.0f;
                    const bool fast = fast_recip_ok(den[bk]);
                    const float r = fast ? recip_approx(den[bk]) : 0.0f;
                    // Element codes from one product per element: with r within 2^-23 of
                    // 1/den (relative), w'/den lies within
                    //   dl >= E r (1 + 2^-19) + X r 2^-20
                    // of x r, and so do the rounded ends fl(x r -+ dl) (the slack covers the
                    // reciprocal's error on |x| <= X, w~'s and w''s own roundings, and the
                    // rounding of the ends).  fl(w'/den) is then between the two ends, and
                    // where both ends give the same E2M1 code (sign included) so does it.
                    const float dl = __fadd_ru(__fmul_ru(__fmul_ru(Ek, r), 1.0f + 0x1p-19f),
                                               __fmul_ru(__fmul_ru(X, r), 0x1p-20f));
                    const float2 r2 = make_float2(r, r), dp = make_float2(dl, dl), dn = make_float2(-dl, -dl);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        float lo8[8], hi8[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 xv = make_float2(x[8 * g + e], x[8 * g + e + 1]);
                            const float2 l = __ffma2_rn(xv, r2, dn);
                            const float2 h = __ffma2_rn(xv, r2, dp);
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
                if (slow) {
                    // Undecided elements (and blocks): their exact values come from the
                    // chain, out of this loop, after the last tile: queued for the whole
                    // CTA in shared memory (kDefer entries; beyond that, the blocks are
                    // marked and recomputed whole).  The codes stored below are then
                    // provisional for them.
                    uint32_t um = 0u;
#pragma unroll
                    for (int w = 0; w < 4; ++w)
#pragma unroll
                        for (int z = 0; z < 8; ++z)
                            um |= (((diff[w] >> (4 * z)) & 0xFu) != 0u ? 1u : 0u) << (8 * w + z);
                    const unsigned int slot = atomicAdd(defn, 1u);
                    if (slot < (unsigned int)kDefer) {
                        defq[slot] = make_uint4((uint32_t)j, um,
                                                (uint32_t)rloc | ((uint32_t)chunk << 8) | (cert[0] ? 0u : 1u << 16) |
                                                    (cert[1] ? 0u : 1u << 17),
                                                0u);
                    } else {
                        // Queue full: bit 7 of a block's scale byte (never set in an E4M3 scale)
                        // marks the block for a full exact recomputation after the loop.
                        if (!cert[0] || (um & 0x0000FFFFu) != 0u) sfc[0] |= 0x80u;
                        if (!cert[1] || (um & 0xFFFF0000u) != 0u) sfc[1] |= 0x80u;
                        *p1_overflow = 1u;
                    }
                }
                if (col_ok) {
                    if (row_ok)
                        *reinterpret_cast<uint4*>(args.codes + (int64_t)n * (args.K >> 1) + (k0 >> 1)) =
                            make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    if (n < args.rows_pad)
                        *reinterpret_cast<uint16_t*>(args.sf + sf_pair_offset(n, k0, args.K)) =
                            (uint16_t)(sfc[0] | (sfc[1] << 8));
                }
            }
            // Done with this tile's W: every shared-memory read of it has returned (its
            // value was used) before the slot is handed back to the TMA.
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[ws]);
        }
        // The deferred elements, once all 16 warps have left the tile loop, in three steps
        // spread over the CTA's 512 epilogue threads (one bounded CTA barrier between
        // steps):
        //   1. each queued entry (one thread's 32 weights of one tile) lists its elements
        //      with an undecided code, or all 16 of a block with an undecided scale;
        //   2. every listed element's exact value: the fp32 chain from global memory (the
        //      row of B, the column of A, W), one round of loads per element;
        //   3. each entry's codes (and, for blocks whose scale was undecided, the scale
        //      byte) from those values by true divisions, written over the provisional
        //      ones.  An entry whose elements did not fit the task list (kTasks) does its
        //      own exact work in step 3.
        __syncwarp();
        if (lane == 0) mbar_arrive(loop_done);
        bool go = mbar_wait(loop_done, 0, args.status, abort_flag, kWaitLimitNs);
        const unsigned int nq = min(*reinterpret_cast<volatile unsigned int*>(defn), (unsigned int)kDefer);
        if (go) {
            for (unsigned int z = (unsigned int)et; z < nq; z += kEpiWarps * 32) {
                const uint4 dq = defq[z];
                uint32_t em = dq.y;
                if ((dq.z >> 16) & 1u) em |= 0x0000FFFFu;
                if ((dq.z >> 17) & 1u) em |= 0xFFFF0000u;
                const unsigned int cnt = (unsigned int)__popc(em);
                const unsigned int base = atomicAdd(ntask, cnt);
                if (base + cnt <= (unsigned int)kTasks) {
                    atomicMax(nfill, base + cnt);
                    unsigned int u = base;
                    for (uint32_t m = em; m != 0u; m &= m - 1u) task_id[u++] = (uint16_t)((z << 5) | (uint32_t)(__ffs((int)m) - 1));
                    defq[z].w = base;
                } else {
                    defq[z].w = 0xFFFFFFFFu;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(tasks_ready);
        go = go && mbar_wait(tasks_ready, 0, args.status, abort_flag, kWaitLimitNs);
        if (go) {
            const unsigned int nt = *reinterpret_cast<volatile unsigned int*>(nfill);
            for (unsigned int u = (unsigned int)et; u < nt; u += kEpiWarps * 32) {
                const uint32_t id = task_id[u];
                if ((id >> 5) >= nq) continue;  // never: every listed task names a queued entry
                const uint4 dq = defq[id >> 5];
                const int t = seq.tile(seq.T + (int)dq.x);
                const int nb = t / nks;
                const int n = nb * (kTM * kPair) + (int)rank * kTM + (int)(dq.z & 0xFFu);
                const int k = (t - nb * nks) * kTK + (int)((dq.z >> 8) & 3u) * kCols + (int)(id & 31u);
                task_val[u] = exact_element(args, n, k, c);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(vals_ready);
        go = go && mbar_wait(vals_ready, 0, args.status, abort_flag, kWaitLimitNs);
        if (go) {
            for (unsigned int z = (unsigned int)et; z < nq && !*abort_flag; z += kEpiWarps * 32) {
                const uint4 dq = defq[z];
                const int t = seq.tile(seq.T + (int)dq.x);
                const int nb = t / nks;
                const int n = nb * (kTM * kPair) + (int)rank * kTM + (int)(dq.z & 0xFFu);
                const int k0 = (t - nb * nks) * kTK + (int)((dq.z >> 8) & 3u) * kCols;
                const bool fix0 = (dq.z >> 16) & 1u, fix1 = (dq.z >> 17) & 1u;
                uint4* cp = reinterpret_cast<uint4*>(args.codes + (int64_t)n * (args.K >> 1) + (k0 >> 1));
                uint16_t* sp = reinterpret_cast<uint16_t*>(args.sf + sf_pair_offset(n, k0, args.K));
                const uint4 cv = *cp;
                const uint32_t sv = *sp;
                Codes32 r;
                r.cw[0] = cv.x; r.cw[1] = cv.y; r.cw[2] = cv.z; r.cw[3] = cv.w;
                r.sfc[0] = sv & 0xFFu;
                r.sfc[1] = sv >> 8;
                if (dq.w == 0xFFFFFFFFu) {
                    r = quant_fix(args.B + (int64_t)n * kRank, args.A, args.K, k0, args.W + (int64_t)n * args.K + k0,
                                  c, s, d, r, dq.y, fix0, fix1);
                } else {
                    uint32_t em = dq.y;
                    if (fix0) em |= 0x0000FFFFu;
                    if (fix1) em |= 0xFFFF0000u;
                    const float* xv = task_val + dq.w;  // exact values, in column order of em's bits
#pragma unroll 1
                    for (int bk = 0; bk < 2; ++bk) {
                        if (!(bk == 0 ? fix0 : fix1)) continue;
                        // The block's 16 exact values: the first 16 (block 0) or the last 16
                        // of its listed elements.
                        const float* x16 = xv + (bk == 0 ? 0 : __popc(em & 0x0000FFFFu));
                        float bam = 0.0f;
#pragma unroll
                        for (int e = 0; e < 16; ++e) bam = fmaxf(bam, fabsf(x16[e]));
                        uint32_t sc = 0;
                        if (d > 0.0f) sc = cvt_e4m3(__fdiv_rn(bam, d));
                        const float dn = __fmul_rn(e4m3_value(sc), s);
                        float q[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) q[e] = dn > 0.0f ? __fdiv_rn(x16[e], dn) : 0.0f;
                        const uint32_t c0 = dn > 0.0f ? cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]) : 0u;
                        const uint32_t c1 = dn > 0.0f ? cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]) : 0u;
                        r.cw[2 * bk] = c0;
                        r.cw[2 * bk + 1] = c1;
                        r.sfc[bk] = sc;
                    }
                    // Elements of blocks whose scale was decided.
                    const float den0 = __fmul_rn(e4m3_value(r.sfc[0]), s), den1 = __fmul_rn(e4m3_value(r.sfc[1]), s);
                    int u = 0;
#pragma unroll 1
                    for (uint32_t m = em; m != 0u; m &= m - 1u, ++u) {
                        const int e = __ffs((int)m) - 1;
                        if ((e < 16 && fix0) || (e >= 16 && fix1)) continue;
                        const float den = e < 16 ? den0 : den1;
                        const uint32_t code =
                            den > 0.0f ? cvt_e2m1x8(__fdiv_rn(xv[u], den), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu : 0u;
                        const uint32_t sh = 4u * (uint32_t)(e & 7), keep = ~(0xFu << sh);
                        const int wi = e >> 3;
                        if (wi == 0) r.cw[0] = (r.cw[0] & keep) | (code << sh);
                        else if (wi == 1) r.cw[1] = (r.cw[1] & keep) | (code << sh);
                        else if (wi == 2) r.cw[2] = (r.cw[2] & keep) | (code << sh);
                        else r.cw[3] = (r.cw[3] & keep) | (code << sh);
                    }
                }
                *cp = make_uint4(r.cw[0], r.cw[1], r.cw[2], r.cw[3]);
                *sp = (uint16_t)(r.sfc[0] | (r.sfc[1] << 8));
            }
            // 4. If the queue overflowed: this thread's blocks marked in bit 7 of their scale
            // byte, each recomputed whole by the exact chain.
            if (*reinterpret_cast<volatile unsigned int*>(p1_overflow) != 0u) {
                for (int j = 0; j < seq.T && !*abort_flag; ++j) {
                    const int t = seq.tile(seq.T + j);
                    const int nb = t / nks;
                    const int n = nb * (kTM * kPair) + (int)rank * kTM + rloc;
                    const int k0 = (t - nb * nks) * kTK + kt0;
                    if (n >= args.N || k0 >= args.K) continue;
                    uint16_t* sp = reinterpret_cast<uint16_t*>(args.sf + sf_pair_offset(n, k0, args.K));
                    const uint32_t sv = *sp;
                    if ((sv & 0x8080u) == 0u) continue;
                    atomicAdd(&xcount[0], ((sv & 0x80u) ? 16u : 0u) + ((sv & 0x8000u) ? 16u : 0u));
                    uint4* cp = reinterpret_cast<uint4*>(args.codes + (int64_t)n * (args.K >> 1) + (k0 >> 1));
                    const uint4 cv = *cp;
                    Codes32 r;
                    r.cw[0] = cv.x; r.cw[1] = cv.y; r.cw[2] = cv.z; r.cw[3] = cv.w;
                    r.sfc[0] = sv & 0x7Fu;
                    r.sfc[1] = (sv >> 8) & 0x7Fu;
                    r = quant_fix(args.B + (int64_t)n * kRank, args.A, args.K, k0, args.W + (int64_t)n * args.K + k0, c,
                                  s, d, r, 0u, (sv & 0x80u) != 0u, (sv & 0x8000u) != 0u);
                    *cp = make_uint4(r.cw[0], r.cw[1], r.cw[2], r.cw[3]);
                    *sp = (uint16_t)(r.sfc[0] | (r.sfc[1] << 8));
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        // The last CTA to finish (every CTA has read the amax by now) turns it into the
        // per-tensor scale.
        __threadfence();
        // The exact chain's share (elements listed for it, blocks recomputed whole).
        const unsigned int xq = *reinterpret_cast<volatile unsigned int*>(ntask) + xcount[0];
        if (xq != 0u) atomicAdd(args.counter + 3, xq);
        if (xcount[1] != 0u) atomicAdd(args.counter + 4, xcount[1]);
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

cudaError_t run_merge_fused(const LaunchCtx& ctx, const RequantTcMaps& m, const TcArgs& a) {
    static OccupancyCache occupancy;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // May start before the split kernel ends (programmatic dependent launch); the kernel
    // waits (griddepcontrol.wait) before reading its results.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(ctx.num_sms / kPair * kPair), 1, 1);
    // The grid barrier between the phases needs every CTA resident at once: the grid is
    // at most the number of clusters the device holds together (one CTA per SM).
    int max_clusters = 0;
    const cudaError_t e = clusters_per_device(occupancy, ctx, merge_fused_kernel, cfg, &max_clusters);
    if (e != cudaSuccess) return e;
    const int clusters = a.tiles < max_clusters ? a.tiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(clusters * kPair), 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, merge_fused_kernel, m.w, m.ap, a);
}

}  // namespace

size_t requant_tc_workspace_bytes(int w_dtype, int r, int64_t N, int64_t K) {
    const int64_t tiles = (N + kTM * kPair - 1) / (kTM * kPair) * ((K + kTK - 1) / kTK);
    if (w_dtype != NVFP4_W_BF16 || r != kRank || N <= 0 || K <= 0 || tiles >= (int64_t(1) << 30))
        return 0;
    return requant_tc_layout(nullptr, N, K).bytes;
}

cudaError_t launch_requant_tc(const LaunchCtx& ctx, const RequantTcMaps& maps, const void* W,
                              const float* A, const float* B, void* workspace, float c, int64_t N,
                              int64_t K, uint8_t* codes, uint8_t* sf, float* s_t) {
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
    a.arrive = ws.counter + 1;
    a.next = ws.counter + 2;
    a.B = B;
    a.A = A;
    a.W = static_cast<const uint16_t*>(W);
    a.cnorm = ws.cnorm;
    a.status = ctx.status;
    a.zero = 0;
    a.nks = (int)((K + kTK - 1) / kTK);
    a.tiles = (int)((N + kTM * kPair - 1) / (kTM * kPair)) * a.nks;
    a.chunk = (int)(K >= 128 ? (int64_t)kWBytes / 2 : K * kChunkRows);
    a.units = (int)((N * K + a.chunk - 1) / a.chunk);
    const int rows_pad256 = (int)((N + 255) / 256 * 256);
    const int nb_rows = (rows_pad256 + kSplitRows - 1) / kSplitRows;
    const int nb_cols = (int)((K + kSplitCols - 1) / kSplitCols);
    merge_split_kernel<<<(unsigned)(nb_rows + nb_cols), kSplitThreads, 0, ctx.stream>>>(
        A, B, (int)N, (int)K, rows_pad256, nb_rows, ws.ap, ws.rnorm, ws.cnorm, s_t, ws.counter);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return run_merge_fused(ctx, maps, a);
}

}  // namespace nvfp4rl
