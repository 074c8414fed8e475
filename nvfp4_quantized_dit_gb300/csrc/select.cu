// Contrastive seed selection and the DiffusionNFT reward transform.
//
// Selection: keep the seeds of the K/2 largest and the K/2 smallest of N proxy
// rewards per prompt (Sol-RL project page, "Two-Stage Pipeline", Stage 1: filter
// the N = 96 candidates to the top/bottom seeds, K = 24 kept; AI Trends summary,
// paragraph on the pipeline: top K/2 and bottom K/2).
// Transform: r = 1/2 + 1/2 clip((x - mean) / Z, -1, 1) ("DiffusionNFT",
// VeRL-Omni documentation, "Algorithm"), Z the population standard deviation
// over all selected rewards of the batch (the page's default, global) or over
// the prompt's group.
//
// Two kernels.  select_rank_kernel: one CTA per prompt, its N rewards staged in
// shared memory; each thread ranks its rewards against all N:
//   rank_top(i) = #{j : v_j > v_i or (v_j == v_i and j < i)}
//   rank_bot(i) = #{j : v_j < v_i or (v_j == v_i and j < i)}
// and seed i goes to slot rank_top(i) (if < K/2) and K/2 + rank_bot(i) (if < K/2).
// select_transform_kernel (only with r_out): one CTA per prompt (at most one per SM,
// each CTA then taking several), started early by programmatic dependent launch and
// waiting for the ranks, reads the selected raw rewards through idx; means and
// standard deviations in fp64 (two passes), then per element (x - mean) * (1 / Z) in
// fp64, clipped and rounded to fp32.  fp64 is slow on this part: the CTAs spread it
// over the SMs (each computes the global statistics itself rather than waiting for
// one that does), and each group takes one division, not one per element.
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxN = 1024;
constexpr int kRankThreads = 256;   // upper bound of the ranking CTA
constexpr int kXformThreads = 256;
constexpr int kKeep = 4;            // selected rewards per thread kept between the two passes

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// a / b from b's reciprocal inv_b = RN(1/b): q = RN(a inv_b), the exact remainder
// a - q b (one fma), and one correction step q + (a - q b) inv_b (Markstein).  An exact
// quotient comes out exact (equal rewards give a mean equal to them and Z = 0).
__device__ __forceinline__ double div_by(double a, double b, double inv_b) {
    const double q = a * inv_b;
    return fma(fma(-q, b, a), inv_b, q);
}

__global__ void __launch_bounds__(kRankThreads) select_rank_kernel(const float* __restrict__ rewards, int N,
                                                                   int K, int32_t* __restrict__ idx) {
    __shared__ float v[kMaxN];
    grid_dep_launch();  // the transform may start its launch; it waits for this grid's results
    const int64_t p = blockIdx.x;
    const int half = K >> 1;
    const float* row = rewards + p * N;
    for (int j = threadIdx.x; j < N; j += blockDim.x) v[j] = row[j];
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const float vi = v[i];
        int gt = 0, lt = 0, eq = 0;  // over all j; ties before i counted separately
        for (int j = 0; j < N; ++j) {
            const float vj = v[j];
            gt += vj > vi;
            lt += vj < vi;
            eq += (vj == vi) & (j < i);
        }
        const int rt = gt + eq, rb = lt + eq;
        if (rt < half) idx[p * K + rt] = i;
        if (rb < half) idx[p * K + half + rb] = i;
    }
}

// Sum over the CTA (every thread gets the result).
__device__ __forceinline__ double block_sum(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();  // red may still be in use by the previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double t = lane < nwarps ? red[lane] : 0.0;
        t = warp_sum(t);
        if (lane == 0) red[32] = t;
    }
    __syncthreads();
    return red[32];
}

__global__ void __launch_bounds__(kXformThreads) select_transform_kernel(
    const float* __restrict__ rewards, int N, const int32_t* __restrict__ idx, int P, int K, int global_std,
    double inv_k, double inv_total, float* __restrict__ r_out) {
    __shared__ double red[33];
    grid_dep_wait();  // idx is complete
    const int lane = threadIdx.x & 31;

    double inv_z_all = 0.0;
    if (global_std) {
        // Global mean, then mean squared deviation, over all P*K selected rewards: the
        // CTA's threads gather them through idx (kKeep each kept in registers for the
        // second pass), all loads of a round in flight together.
        const int64_t total = (int64_t)P * K;
        const int64_t step = blockDim.x;
        float keep[kKeep];
        double acc = 0.0;
#pragma unroll
        for (int u = 0; u < kKeep; ++u) {
            const int64_t e = threadIdx.x + u * step;
            keep[u] = e < total ? rewards[(e / K) * N + idx[e]] : 0.0f;
            acc += (double)keep[u];
        }
        for (int64_t e = threadIdx.x + kKeep * step; e < total; e += step)
            acc += (double)rewards[(e / K) * N + idx[e]];
        const double mean = div_by(block_sum(acc, red), (double)total, inv_total);
        acc = 0.0;
#pragma unroll
        for (int u = 0; u < kKeep; ++u) {
            const double dv = (double)keep[u] - mean;
            if (threadIdx.x + u * step < total) acc += dv * dv;
        }
        for (int64_t e = threadIdx.x + kKeep * step; e < total; e += step) {
            const double dv = (double)rewards[(e / K) * N + idx[e]] - mean;
            acc += dv * dv;
        }
        const double z = sqrt(div_by(block_sum(acc, red), (double)total, inv_total));
        inv_z_all = z > 0.0 ? 1.0 / z : 0.0;
    }
    if (threadIdx.x >= 32) return;  // one warp per prompt from here on

    for (int64_t p = blockIdx.x; p < P; p += gridDim.x) {
        const float* rw = rewards + p * N;
        const int32_t* ip = idx + p * K;
        float* rp = r_out + p * K;
        double sum = 0.0;
        for (int t = lane; t < K; t += 32) sum += (double)rw[ip[t]];
        const double mu = div_by(warp_sum(sum), (double)K, inv_k);
        double inv_z = inv_z_all;
        if (!global_std) {
            double ss = 0.0;
            for (int t = lane; t < K; t += 32) {
                const double dv = (double)rw[ip[t]] - mu;
                ss += dv * dv;
            }
            const double z = sqrt(div_by(warp_sum(ss), (double)K, inv_k));
            inv_z = z > 0.0 ? 1.0 / z : 0.0;
        }
        for (int t = lane; t < K; t += 32) {
            double r = 0.5;
            if (inv_z > 0.0) {
                double u = ((double)rw[ip[t]] - mu) * inv_z;
                u = u < -1.0 ? -1.0 : (u > 1.0 ? 1.0 : u);
                r = 0.5 + 0.5 * u;
            }
            rp[t] = (float)r;
        }
    }
}

}  // namespace

cudaError_t launch_select(const LaunchCtx& ctx, const float* rewards, int P, int N, int K,
                          int global_std, int32_t* idx, float* r_out) {
    if (N > kMaxN) return cudaErrorInvalidValue;
    const int threads = N >= kRankThreads ? kRankThreads : (N + 31) / 32 * 32;
    select_rank_kernel<<<(unsigned)P, threads, 0, ctx.stream>>>(rewards, N, K, idx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || r_out == nullptr) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // Every CTA gathers all P * K selected rewards for the global statistics: at most
    // one CTA per SM keeps that redundant work to one pass per SM.
    cfg.gridDim = dim3((unsigned)(P < ctx.num_sms ? P : ctx.num_sms));
    cfg.blockDim = dim3(kXformThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // The reciprocals of the means' divisors, for div_by (fp64 divisions on the host).
    const double inv_k = 1.0 / (double)K, inv_total = 1.0 / ((double)P * (double)K);
    return cudaLaunchKernelEx(&cfg, select_transform_kernel, rewards, N, static_cast<const int32_t*>(idx),
                              P, K, global_std, inv_k, inv_total, r_out);
}

}  // namespace nvfp4rl
