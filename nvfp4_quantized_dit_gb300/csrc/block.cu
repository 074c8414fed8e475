// The streaming kernels of the synthetic DiT block (a FLUX-shaped stand-in for the
// linears of the NVFP4-quantized solver, Sol-RL project page, "Two-Stage Pipeline",
// Stage 1): the per-head transpose of v for the fused attention (attn.cu), a row
// softmax (the attention's softmax step as an entry point of its own), the GELU and
// the residual add.  Every one is a streaming pass over bf16 data (HBM- or L2-bound);
// each rounds its result to bf16 once, to nearest-even.
//
//   heads_vt      qkv [B*S, 3D] -> V^T [B*H, dh, S]
//   softmax_rows  P = bf16(softmax(scale * L)) per row, in place allowed
//   gelu          y = bf16(x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))), fp32 (through
//                 the logistic form of the same function)
//   add           y = bf16(a + b), the sum in fp32
#include "block.cuh"

namespace nvfp4rl {
namespace {

constexpr int kBlkThreads = 256;

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t to_bf(float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&b);
}

// V transposed per head, through a 64 x 64 shared-memory tile: block (tile of S, tile of
// dh, head z) reads 64 tokens x 64 channels (16-byte loads, 8 threads per token row) and
// writes 64 channels x 64 tokens (16-byte stores, 8 threads per channel row).  S and dh
// are multiples of 64.
constexpr int kTr = 64;
constexpr int kTrPad = kTr + 8;  // row stride 144 bytes: the 8 rows a store gathers sit in distinct banks
__global__ void __launch_bounds__(kBlkThreads)
    heads_split_vt_kernel(const uint16_t* __restrict__ qkv, int64_t S, int64_t D, int64_t H,
                          uint16_t* __restrict__ Vt) {
    __shared__ __align__(16) uint16_t tile[kTr][kTrPad];
    const int64_t dh = D / H;
    const int64_t z = blockIdx.z, b = z / H, h = z - b * H;
    const int64_t s0 = (int64_t)blockIdx.x * kTr, c0 = (int64_t)blockIdx.y * kTr;
    for (int i = threadIdx.x; i < kTr * (kTr / 8); i += kBlkThreads) {
        const int rs = i >> 3, piece = i & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(qkv + (b * S + s0 + rs) * 3 * D + 2 * D + h * dh + c0 + piece * 8);
        *reinterpret_cast<uint4*>(&tile[rs][piece * 8]) = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTr * (kTr / 8); i += kBlkThreads) {
        const int rc = i >> 3, tg = i & 7;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = (uint32_t)tile[tg * 8 + 2 * q][rc] | ((uint32_t)tile[tg * 8 + 2 * q + 1][rc] << 16);
        *reinterpret_cast<uint4*>(Vt + (z * dh + c0 + rc) * S + s0 + tg * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One warp per row; the row (cols % 8 == 0) is read three times (maximum, sum of
// exponentials, output), the last two from L1/L2.  exp(scale (l - m)) in fp32.
__global__ void __launch_bounds__(kBlkThreads)
    softmax_rows_kernel(const uint16_t* L, int64_t rows, int64_t cols, float scale, uint16_t* P) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kBlkThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kBlkThreads) >> 5;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const uint4* row = reinterpret_cast<const uint4*>(L + r * cols);
        const int64_t n8 = cols / 8;
        float m = -INFINITY;
        for (int64_t i = lane; i < n8; i += 32) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(bf((uint16_t)w[q]), bf((uint16_t)(w[q] >> 16))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        float sum = 0.0f;
        for (int64_t i = lane; i < n8; i += 32) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                sum += expf(scale * (bf((uint16_t)w[q]) - m)) + expf(scale * (bf((uint16_t)(w[q] >> 16)) - m));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        const float inv = 1.0f / sum;
        uint4* out = reinterpret_cast<uint4*>(P + r * cols);
        for (int64_t i = lane; i < n8; i += 32) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t y[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float e0 = expf(scale * (bf((uint16_t)w[q]) - m)) * inv;
                const float e1 = expf(scale * (bf((uint16_t)(w[q] >> 16)) - m)) * inv;
                y[q] = (uint32_t)to_bf(e0) | ((uint32_t)to_bf(e1) << 16);
            }
            out[i] = make_uint4(y[0], y[1], y[2], y[3]);
        }
    }
}

// 8 values per thread and step (n % 8 == 0).
__global__ void __launch_bounds__(kBlkThreads)
    gelu_kernel(const uint16_t* x, int64_t n, uint16_t* y) {
    for (int64_t i = (int64_t)blockIdx.x * kBlkThreads + threadIdx.x; i < n / 8;
         i += (int64_t)gridDim.x * kBlkThreads) {
        const uint4 v = reinterpret_cast<const uint4*>(x)[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 g = gelu_f32x2(make_float2(bf((uint16_t)w[q]), bf((uint16_t)(w[q] >> 16))));
            o[q] = (uint32_t)to_bf(g.x) | ((uint32_t)to_bf(g.y) << 16);
        }
        reinterpret_cast<uint4*>(y)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void __launch_bounds__(kBlkThreads)
    add_kernel(const uint16_t* a, const uint16_t* b, int64_t n, uint16_t* y) {
    for (int64_t i = (int64_t)blockIdx.x * kBlkThreads + threadIdx.x; i < n / 8;
         i += (int64_t)gridDim.x * kBlkThreads) {
        const uint4 u = reinterpret_cast<const uint4*>(a)[i];
        const uint4 v = reinterpret_cast<const uint4*>(b)[i];
        const uint32_t wu[4] = {u.x, u.y, u.z, u.w}, wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = bf((uint16_t)wu[q]) + bf((uint16_t)wv[q]);
            const float hi = bf((uint16_t)(wu[q] >> 16)) + bf((uint16_t)(wv[q] >> 16));
            o[q] = (uint32_t)to_bf(lo) | ((uint32_t)to_bf(hi) << 16);
        }
        reinterpret_cast<uint4*>(y)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

unsigned stream_grid(int64_t work, const LaunchCtx& ctx) {
    int64_t g = (work + kBlkThreads - 1) / kBlkThreads;
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_heads_vt(const LaunchCtx& ctx, const uint16_t* qkv, int64_t B, int64_t S, int64_t D, int64_t H,
                            uint16_t* Vt) {
    const int64_t dh = D / H;
    const dim3 grid((unsigned)((S + kTr - 1) / kTr), (unsigned)((dh + kTr - 1) / kTr), (unsigned)(B * H));
    heads_split_vt_kernel<<<grid, kBlkThreads, 0, ctx.stream>>>(qkv, S, D, H, Vt);
    return cudaGetLastError();
}

cudaError_t launch_softmax_rows(const LaunchCtx& ctx, const uint16_t* L, int64_t rows, int64_t cols, float scale,
                                uint16_t* P) {
    softmax_rows_kernel<<<stream_grid(rows * 32, ctx), kBlkThreads, 0, ctx.stream>>>(L, rows, cols, scale, P);
    return cudaGetLastError();
}

cudaError_t launch_gelu(const LaunchCtx& ctx, const uint16_t* x, int64_t n, uint16_t* y) {
    gelu_kernel<<<stream_grid(n / 8, ctx), kBlkThreads, 0, ctx.stream>>>(x, n, y);
    return cudaGetLastError();
}

cudaError_t launch_add(const LaunchCtx& ctx, const uint16_t* a, const uint16_t* b, int64_t n, uint16_t* y) {
    add_kernel<<<stream_grid(n / 8, ctx), kBlkThreads, 0, ctx.stream>>>(a, b, n, y);
    return cudaGetLastError();
}

}  // namespace nvfp4rl
