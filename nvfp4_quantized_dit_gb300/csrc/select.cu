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
// One CTA; warp w handles prompts w, w + nwarps, ...  Each lane ranks its rewards
// against the prompt's N rewards staged in shared memory:
//   rank_top(i) = #{j : v_j > v_i or (v_j == v_i and j < i)}
//   rank_bot(i) = #{j : v_j < v_i or (v_j == v_i and j < i)}
// and seed i goes to slot rank_top(i) (if < K/2) and K/2 + rank_bot(i) (if < K/2).
// The transform is done in fp64 with the selected raw rewards parked in r_out.
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__global__ void __launch_bounds__(1024) select_kernel(const float* __restrict__ rewards, int P,
                                                      int N, int K, int global_std,
                                                      int32_t* __restrict__ idx,
                                                      float* __restrict__ r_out) {
    extern __shared__ float vals[];  // [nwarps][N]
    __shared__ double red[32];
    __shared__ double s_mean;
    __shared__ double s_z;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int half = K >> 1;
    float* v = vals + warp * N;

    for (int p = warp; p < P; p += nwarps) {
        const float* row = rewards + (int64_t)p * N;
        for (int j = lane; j < N; j += 32) v[j] = row[j];
        __syncwarp();
        for (int i = lane; i < N; i += 32) {
            const float vi = v[i];
            int rt = 0, rb = 0;
            for (int j = 0; j < N; ++j) {
                const float vj = v[j];
                rt += (vj > vi) || (vj == vi && j < i);
                rb += (vj < vi) || (vj == vi && j < i);
            }
            if (rt < half) {
                idx[(int64_t)p * K + rt] = i;
                if (r_out) r_out[(int64_t)p * K + rt] = vi;
            }
            if (rb < half) {
                idx[(int64_t)p * K + half + rb] = i;
                if (r_out) r_out[(int64_t)p * K + half + rb] = vi;
            }
        }
        __syncwarp();
    }
    if (r_out == nullptr) return;
    __syncthreads();  // every selected raw reward is in r_out (written by this CTA)

    const int64_t total = (int64_t)P * K;
    if (global_std) {
        // Global mean, then mean squared deviation, over all P*K selected rewards.
        double acc = 0.0;
        for (int64_t e = threadIdx.x; e < total; e += blockDim.x) acc += (double)r_out[e];
        acc = warp_sum(acc);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w = 0; w < nwarps; ++w) t += red[w];
            s_mean = t / (double)total;
        }
        __syncthreads();
        const double mean = s_mean;
        acc = 0.0;
        for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
            const double dv = (double)r_out[e] - mean;
            acc += dv * dv;
        }
        acc = warp_sum(acc);
        __syncthreads();
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w = 0; w < nwarps; ++w) t += red[w];
            s_z = sqrt(t / (double)total);
        }
        __syncthreads();
    }

    for (int p = warp; p < P; p += nwarps) {
        float* rp = r_out + (int64_t)p * K;
        double sum = 0.0;
        for (int t = lane; t < K; t += 32) sum += (double)rp[t];
        const double mu = warp_sum(sum) / (double)K;
        double z;
        if (global_std) {
            z = s_z;
        } else {
            double ss = 0.0;
            for (int t = lane; t < K; t += 32) {
                const double dv = (double)rp[t] - mu;
                ss += dv * dv;
            }
            z = sqrt(warp_sum(ss) / (double)K);
        }
        __syncwarp();
        for (int t = lane; t < K; t += 32) {
            double r = 0.5;
            if (z > 0.0) {
                double u = ((double)rp[t] - mu) / z;
                u = u < -1.0 ? -1.0 : (u > 1.0 ? 1.0 : u);
                r = 0.5 + 0.5 * u;
            }
            rp[t] = (float)r;
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_select(const LaunchCtx& ctx, const float* rewards, int P, int N, int K,
                          int global_std, int32_t* idx, float* r_out) {
    int warps = P < 32 ? (P < 1 ? 1 : P) : 32;
    const size_t smem = (size_t)warps * N * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<1, warps * 32, smem, ctx.stream>>>(rewards, P, N, K, global_std, idx, r_out);
    return cudaGetLastError();
}

}  // namespace nvfp4rl
