// Tensor-core GEMMs on the 5th-generation (tcgen05) tensor cores of sm_103a.
//
//  * NVFP4:  Y = bf16( s_a[m] * s_w * sum_k (e2m1(qa) sfa)(e2m1(qw) sfw) + bias[n] )
//            with tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X: E2M1
//            operands packed two per byte, one E4M3 scale per 16 K-elements read
//            from tensor memory.  This is the FP4 linear layer of the
//            NVFP4-quantized solver (Sol-RL project page, "Two-Stage Pipeline",
//            Stage 1: "up to 4x TFLOPs vs. BF16").
//  * BF16:   Y = bf16( X W^T + bias ) with kind::f16 (Stage 2's BF16 layers).
//
// One persistent CTA per SM, 192 threads:
//   warp 0       TMA producer: A/B tiles (128-byte swizzle) and, for NVFP4, the
//                scale tiles (bulk copies) into a 4-stage shared-memory ring;
//   warp 1       allocates 512 tensor-memory columns; lane 0 issues the MMAs
//                (scale tiles first go shared -> tensor memory with tcgen05.cp);
//   warps 2..5   epilogue: tensor memory -> registers (tcgen05.ld), scale, bias,
//                bf16, staged through shared memory into coalesced global stores.
// Tile 128 x 256 (M x N), 128 bytes of K per stage row (256 E2M1 or 64 BF16
// elements), fp32 accumulator in tensor-memory columns 0..255.  NVFP4 scale
// tiles for stage s live in columns 256 + 48 s (A: 4 per MMA, B: 8 per MMA).
//
// Every mbarrier wait is bounded (common.cuh: mbar_wait); on expiry the kernel
// records NVFP4_ERR_TIMEOUT, drains its own copies and MMAs (again bounded),
// frees tensor memory and returns.
#include "common.cuh"

namespace nvfp4rl {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kATileBytes = BM * 128;    // 16 KB
constexpr uint32_t kBTileBytes = BN * 128;    // 32 KB
constexpr uint32_t kSFAStageBytes = 4 * 512;  // 128 rows x 4 K-chunks of 64
constexpr uint32_t kSFBStageBytes = 8 * 512;  // 256 rows x 4 K-chunks of 64
constexpr uint32_t kEpiWarpBytes = 32 * 64;   // 32 rows x 32 bf16
constexpr uint32_t kEpiBytes = 4 * kEpiWarpBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;
constexpr uint32_t kSfTmemPerStage = 48;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s for copies already in flight

template <bool kFP4>
struct Cfg {
    static constexpr uint32_t kStageBytes =
        kATileBytes + kBTileBytes + (kFP4 ? kSFAStageBytes + kSFBStageBytes : 0u);
    static constexpr uint32_t kBarrierBytes = 256;
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarrierBytes;
};
static_assert(Cfg<true>::kSmemBytes <= 232448, "shared memory budget");
static_assert(Cfg<true>::kStageBytes % 1024 == 0 && Cfg<false>::kStageBytes % 1024 == 0,
              "stages must keep 1024-byte alignment for the 128-byte swizzle");

// Instruction descriptors (tcgen05, 32 bits): bits 4-5 accumulator format
// (1 = f32), 7-9 A format, 10-12 B format, 15/16 A/B major (0 = K-major),
// 17-22 N >> 3, 24-28 M >> 4.  For the block-scaled kinds bit 23 selects the
// scale type (0 = UE4M3) and the E2M1 format code is 1.
constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t idesc_nvfp4() {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | (0u << 23) |
           ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

struct GemmArgs {
    const uint8_t* a_sf;
    const uint8_t* b_sf;
    const float* a_srow;
    const float* w_st;
    const __nv_bfloat16* bias;
    __nv_bfloat16* Y;
    int M, N, K;
    int* status;
};

template <bool kFP4>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
    using C = Cfg<kFP4>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi = smem + kStages * C::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi + kEpiBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tmem_full = empty + kStages;
    uint64_t* tmem_empty = tmem_full + 1;
    uint64_t* drain = tmem_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = args.M, N = args.N, K = args.K;
    const int num_m = (M + BM - 1) / BM;
    const int num_n = (N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    // MMA steps along K: 64 E2M1 (32 bytes) or 16 BF16 (32 bytes) each; 4 per stage.
    const int k_steps = kFP4 ? K / 64 : (K + 15) / 16;
    const int num_kb = (k_steps + 3) / 4;
    const int sf_row_tiles_b = (N + 127) / 128;
    const int k_chunks = K / 64;  // 512-byte scale tiles per 128-row tile (NVFP4)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m_blk = tile % num_m;
                const int n_blk = tile / num_m;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, args.status, abort_flag,
                                   kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * C::kStageBytes;
                    uint8_t* sb = sa + kATileBytes;
                    uint32_t bytes = kATileBytes + kBTileBytes;
                    const int nk = min(4, k_steps - kb * 4);
                    int nb = 0;
                    if (kFP4) {
                        nb = (2 * n_blk + 1 < sf_row_tiles_b) ? 2 : 1;
                        bytes += (uint32_t)nk * 512u * (uint32_t)(1 + nb);
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    const int x = kFP4 ? kb * 128 : kb * 64;
                    tma_load_2d(&tmap_a, &full[stage], sa, x, m_blk * BM);
                    tma_load_2d(&tmap_b, &full[stage], sb, x, n_blk * BN);
                    if (kFP4) {
                        uint8_t* sfa = sb + kBTileBytes;
                        uint8_t* sfb = sfa + kSFAStageBytes;
                        const uint8_t* src_a =
                            args.a_sf + ((size_t)m_blk * k_chunks + (size_t)kb * 4) * 512;
                        bulk_load(sfa, src_a, (uint32_t)nk * 512u, &full[stage]);
                        for (int h = 0; h < nb; ++h) {
                            const uint8_t* src_b =
                                args.b_sf +
                                ((size_t)(2 * n_blk + h) * k_chunks + (size_t)kb * 4) * 512;
                            bulk_load(sfb + h * 2048, src_b, (uint32_t)nk * 512u, &full[stage]);
                        }
                    }
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA exits.
                for (int s = 0; s < kStages; ++s)
                    if (issued & (1u << s)) {
                        int dummy_flag = 0;
                        mbar_wait(&full[s], (last_parity >> s) & 1u, args.status, &dummy_flag,
                                  kDrainLimitNs);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = kFP4 ? idesc_nvfp4() : idesc_bf16();
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            bool any_mma = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(tmem_empty, acc_phase ^ 1u, args.status, abort_flag,
                               kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, args.status, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int nk = min(4, k_steps - kb * 4);
                    const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t sb = sa + kATileBytes;
                    const uint32_t sf_col = kSfTmemBase + (uint32_t)stage * kSfTmemPerStage;
                    if (kFP4) {
                        const uint32_t sfa = sb + kBTileBytes;
                        const uint32_t sfb = sfa + kSFAStageBytes;
                        for (int kk = 0; kk < nk; ++kk) {
                            tmem_cp_32x128b_x4(tmem_base + sf_col + 4 * kk,
                                               smem_desc(sfa + kk * 512, 128, 128, kLayoutNone));
                            tmem_cp_32x128b_x4(tmem_base + sf_col + 16 + 8 * kk,
                                               smem_desc(sfb + kk * 512, 128, 128, kLayoutNone));
                            tmem_cp_32x128b_x4(
                                tmem_base + sf_col + 16 + 8 * kk + 4,
                                smem_desc(sfb + 2048 + kk * 512, 128, 128, kLayoutNone));
                        }
                    }
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, kLayoutSw128);
                        const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, kLayoutSw128);
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        if (kFP4)
                            mma_nvfp4(tmem_base, ad, bd, idesc, tmem_base + sf_col + 4 * kk,
                                      tmem_base + sf_col + 16 + 8 * kk, acc);
                        else
                            mma_bf16(tmem_base, ad, bd, idesc, acc);
                    }
                    any_mma = true;
                    mma_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tmem_full);
                acc_phase ^= 1u;
            }
            if (*abort_flag && any_mma) {
                // Let every MMA this thread issued finish before tensor memory is freed.
                mma_commit(drain);
                int dummy_flag = 0;
                mbar_wait(drain, 0, args.status, &dummy_flag, kDrainLimitNs);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
        uint8_t* stg = epi + (warp - 2) * kEpiWarpBytes;
        uint32_t acc_phase = 0;
        const float w_scale = kFP4 ? *args.w_st : 1.0f;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int m_blk = tile % num_m;
            const int n_blk = tile / num_m;
            bool ok = mbar_wait(tmem_full, acc_phase, args.status, abort_flag, kWaitLimitNs);
            // tcgen05.ld is .sync.aligned: reconverge the warp and agree on the outcome.
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            const int row = m_blk * BM + quarter * 32 + lane;
            const int n0 = n_blk * BN;
            float scale = 1.0f;
            if (kFP4) scale = (row < M ? args.a_srow[row] : 0.0f) * w_scale;
            uint32_t packed[128];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // 8 bias values (one 16-byte load, warp-uniform address) per 8 columns.
                    uint4 braw = make_uint4(0, 0, 0, 0);
                    const int col = n0 + c * 32 + q * 8;
                    if (args.bias != nullptr && col < N)
                        braw = __ldg(reinterpret_cast<const uint4*>(args.bias + col));
                    const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = q * 4 + u;
                        packed[c * 16 + i] = pack_bf16x2(
                            fmaf(__uint_as_float(v[2 * i]), scale, __uint_as_float(bw[u] << 16)),
                            fmaf(__uint_as_float(v[2 * i + 1]), scale,
                                 __uint_as_float(bw[u] & 0xFFFF0000u)));
                    }
                }
            }
            // The accumulator is in registers: hand tensor memory back to the MMA warp.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                // Row `lane` of the 32x32 bf16 chunk -> staging (16-byte pieces XOR-swizzled
                // by row), then 8 rows x 64 bytes per store instruction.
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 val = make_uint4(packed[c * 16 + 4 * j], packed[c * 16 + 4 * j + 1],
                                                 packed[c * 16 + 4 * j + 2],
                                                 packed[c * 16 + 4 * j + 3]);
                    *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ (lane & 3)) * 16)) = val;
                }
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int rr = it * 8 + (lane >> 2);
                    const int ch = lane & 3;
                    const uint4 val =
                        *reinterpret_cast<const uint4*>(stg + rr * 64 + ((ch ^ (rr & 3)) * 16));
                    const int grow = m_blk * BM + quarter * 32 + rr;
                    const int gcol = n0 + c * 32 + ch * 8;
                    if (grow < M && gcol < N)
                        *reinterpret_cast<uint4*>(args.Y + (size_t)grow * N + gcol) = val;
                }
                __syncwarp();
            }
            acc_phase ^= 1u;
        }
    }

    // ------------------------------------------------ teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status, &abort_flag, limit_ns);
    __syncthreads();
}

template <bool kFP4>
cudaError_t run_gemm(const LaunchCtx& ctx, const CUtensorMap& ta, const CUtensorMap& tb,
                     const GemmArgs& args) {
    // Set on every call: the attribute belongs to the current device's context.
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<kFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg<kFP4>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)((args.M + BM - 1) / BM) * ((args.N + BN - 1) / BN);
    const int grid = (int)(tiles < ctx.num_sms ? tiles : ctx.num_sms);
    gemm_kernel<kFP4><<<grid, kThreads, Cfg<kFP4>::kSmemBytes, ctx.stream>>>(ta, tb, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_nvfp4(const LaunchCtx& ctx, const CUtensorMap& tmap_a,
                              const CUtensorMap& tmap_b, const uint8_t* a_sf, const uint8_t* w_sf,
                              const float* a_srow, const float* w_st, const __nv_bfloat16* bias,
                              __nv_bfloat16* Y, int64_t M, int64_t N, int64_t K) {
    GemmArgs a{a_sf, w_sf, a_srow, w_st, bias, Y, (int)M, (int)N, (int)K, ctx.status};
    return run_gemm<true>(ctx, tmap_a, tmap_b, a);
}

cudaError_t launch_gemm_bf16(const LaunchCtx& ctx, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const __nv_bfloat16* bias,
                             __nv_bfloat16* Y, int64_t M, int64_t N, int64_t K) {
    GemmArgs a{nullptr, nullptr, nullptr, nullptr, bias, Y, (int)M, (int)N, (int)K, ctx.status};
    return run_gemm<false>(ctx, tmap_a, tmap_b, a);
}

cudaError_t launch_test_wait_timeout(const LaunchCtx& ctx, int64_t timeout_ns) {
    wait_timeout_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, (uint64_t)timeout_ns);
    return cudaGetLastError();
}

}  // namespace nvfp4rl
