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
// Persistent kernel on CTA pairs (clusters of two): each pair computes a 256 x 256
// tile with 2-CTA MMAs (tcgen05 cta_group::2, M = 256).  Each CTA loads its own 128
// rows of A and one half of B's 256 rows; the even CTA issues the MMAs for both.
//
// The even CTA's first 128 rows of B are output columns 256 nb .. +127 and the odd
// CTA's the next 128.  One accumulator of 256 columns per CTA: the MMAs of the next
// tile wait until the epilogue has moved it to registers (it is released before the
// conversion and the stores).
//
// Warps (NVFP4: 16 = four role-uniform warp groups, so that registers can be moved
// to the epilogue with setmaxnreg; BF16: 10):
//   warp 0       TMA producer (both CTAs): A, this CTA's half of B and, for NVFP4,
//                the scale tiles of this stage into a shared-memory ring; A/B
//                completion is counted on the even CTA's barriers, the scale tiles
//                on this CTA's own;
//   warp 1       allocates 512 tensor-memory columns in both CTAs (collectively);
//                lane 0 of the even CTA issues the MMAs and releases each stage
//                to both CTAs;
//   epilogue     NVFP4 warps 8..15, BF16 warps 2..9 (both CTAs), two warps per
//                tensor-memory lane quarter (quarter = warp % 4),
//                128 columns each: tensor memory -> registers (tcgen05.ld, all
//                issued before one wait), release of the accumulator, then scale,
//                bias, bf16, and 32x32 chunks stored by TMA from a swizzled
//                shared-memory staging ring (asynchronous, clipped at M and N);
//   warps 4..7   NVFP4 only (both CTAs), one per lane quarter: copy each stage's
//                scale bytes from shared memory into registers and write them into
//                this CTA's tensor memory with tcgen05.st (four warps writing their
//                own lane quarters in parallel), then signal the even CTA.
// Per CTA: fp32 accumulator in tensor-memory columns 0..255 (its 128 rows x 256);
// NVFP4 scales for stage s in columns 256 + 48 s: A at +4 kk for K-step kk (4
// columns: lane l, column c holds the 4 scales of row l + 32 c), B at +16 + 8 kk
// (8 columns: lane l, column c holds the scales of B row l + 32 c).  Each lane
// quarter holds the same scale data (the MMA reads its own quarter).  These are the
// 512-byte chunks of the 128x4 blocked scale layout, row l of a chunk per lane.
//
// Every mbarrier wait is bounded (common.cuh: mbar_wait); on expiry the kernel
// records NVFP4_ERR_TIMEOUT, drains its own copies and MMAs (again bounded),
// frees tensor memory and returns.
#include "common.cuh"
#include "gemm_epilogue.cuh"

namespace nvfp4rl {
namespace {

constexpr int BM = 128;        // rows of A / D per CTA
constexpr int BN = 256;        // columns of D per pair (rows of B)
constexpr int kPair = 2;       // CTAs per cluster (one 2-CTA MMA)
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 4;
constexpr int kSfWarp0 = 4;  // NVFP4: scale writers are warp group 1
constexpr uint32_t kATileBytes = BM * 128;            // 16 KB: 128 rows x 128 B
constexpr uint32_t kBHalfBytes = (BN / kPair) * 128;  // 16 KB: this CTA's 128 rows of B
constexpr uint32_t kSFAStageBytes = 4 * 512;          // 128 rows x 4 K-chunks of 64
constexpr uint32_t kSFBStageBytes = 8 * 512;          // 256 rows x 4 K-chunks of 64
constexpr uint32_t kChunkBytes = 32 * 64;             // 32 rows x 32 bf16, one TMA store
constexpr uint32_t kBiasBytes = 256;                   // 128 bias values per epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = 256;
constexpr uint32_t kSfTmemPerStage = 48;
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kEvenCta = 0x1;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s for copies already in flight

template <bool kFP4>
struct Cfg {
    // NVFP4 stages carry A, B and the scale tiles (38 KB); BF16 stages A and B (32 KB),
    // one more of them thanks to a single epilogue staging chunk per warp.
    static constexpr int kStages = kFP4 ? 5 : 6;
    static constexpr int kEpiWarp0 = kFP4 ? 8 : 2;  // first epilogue warp
    static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
    // A and B bytes this CTA loads per stage (the even CTA expects twice that), and for
    // NVFP4 its scale-tile bytes (expected on its own barrier).
    static constexpr uint32_t kABBytes = kATileBytes + kBHalfBytes;
    static constexpr uint32_t kSFBytes = kFP4 ? kSFAStageBytes + kSFBStageBytes : 0u;
    static constexpr uint32_t kStageBytes = kABBytes + kSFBytes;
    static constexpr int kEpiBufs = kFP4 ? 2 : 1;  // staging chunks per epilogue warp
    static constexpr uint32_t kEpiBytes = kEpiWarps * (kEpiBufs * kChunkBytes + kBiasBytes);
    static constexpr uint32_t kBarrierBytes = 256;
    static constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarrierBytes;
};
static_assert(Cfg<true>::kSmemBytes <= 232448 && Cfg<false>::kSmemBytes <= 232448,
              "shared memory budget");
static_assert(Cfg<true>::kStageBytes % 1024 == 0 && Cfg<false>::kStageBytes % 1024 == 0,
              "stages must keep 1024-byte alignment for the 128-byte swizzle");
static_assert(kSfTmemBase + Cfg<true>::kStages * kSfTmemPerStage <= kTmemCols, "tensor memory");
static_assert(kSfWarp0 % 4 == 0 && kSfWarps == 4 && Cfg<true>::kEpiWarp0 == kSfWarp0 + kSfWarps,
              "scale warps are one whole warp group covering the four lane quarters");
// NVFP4 register split (per thread; warp groups 0..3, launched with 65536 / 512 = 128):
// producer/MMA group, scale writers, two epilogue groups.  Must not exceed 4 x 128.
constexpr uint32_t kRegsCtl = 56, kRegsSf = 88, kRegsEpi = 184;
static_assert(kRegsCtl + kRegsSf + 2 * kRegsEpi <= 4 * 128, "setmaxnreg split over budget");

// Instruction descriptors (tcgen05, 32 bits): bits 4-5 accumulator format
// (1 = f32), 7-9 A format, 10-12 B format, 15/16 A/B major (0 = K-major),
// 17-22 N >> 3, 24-28 M >> 4 (M = 256 for the pair).  For the block-scaled kinds
// bit 23 selects the scale type (0 = UE4M3) and the E2M1 format code is 1.
constexpr uint32_t kMmaM = BM * kPair;
constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((kMmaM >> 4) << 24);
}
constexpr uint32_t idesc_nvfp4() {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | (0u << 23) | ((kMmaM >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

struct GemmArgs {
    const float* a_srow;
    const float* w_st;
    const __nv_bfloat16* bias;
    int M, N, K;
    int* status;
    uint64_t wait_limit_ns;  // bound of every wait (kWaitLimitNs; shorter in the test hook)
    int withhold_kb;         // test hook only: K-stage whose loads the first pair's even CTA
                             // never issues (on its first tile), or -1
    float* row_amax;         // optional: max |Y[m, :]| (of the bf16 values), atomicMax on the
                             // fp32 bits into a zeroed [M] array; nullptr: not computed
    const uint16_t* residual;  // kGemmEpiResidual only: [M, N] bf16 added to the bf16 output
};

// Pair tiles, grouped for L2 reuse: tiles are ordered in bands of kBandMp m-pairs
// (256 rows each); inside a band the m-pair varies fastest,
// then the n-block.  The clusters walk t = c, c + num_clusters, ..., so the tiles in
// flight at any time share a few m-pairs (their A rows are read from DRAM once) and
// sweep B band by band (B is re-read once per band), instead of re-reading A for
// every n-block.  Tile t covers m-blocks 2 mp + {0, 1} (one per CTA) and n-block nb.
// FLUX.1 up-projection: NVFP4 with bands of 4 ~2% faster than 8, 16 or 32 (its B,
// 21 MB, stays in L2; DRAM reads 119 MB against 254 MB with 16); BF16 with 16 (its
// 75.5 MB B does not stay in L2 over narrow bands: 2.8 GB of DRAM reads with 4).
template <bool kFP4>
struct Sched {
    static constexpr int kBandMp = kFP4 ? 4 : 16;
    int num_m, num_mp, num_n, total, first, step;
    __device__ Sched(int M, int N) {
        num_m = (M + BM - 1) / BM;
        num_mp = (num_m + kPair - 1) / kPair;
        num_n = (N + BN - 1) / BN;
        total = num_mp * num_n;
        first = (int)(blockIdx.x / kPair);
        step = (int)(gridDim.x / kPair);
    }
    __device__ __forceinline__ void tile(int t, int& mp, int& nb) const {
        const int band = t / (kBandMp * num_n);
        const int within = t - band * (kBandMp * num_n);
        const int rows = min(kBandMp, num_mp - band * kBandMp);  // m-pairs in this band
        mp = band * kBandMp + within % rows;
        nb = within / rows;
    }
};

// kEpi: 0, or kGemmEpiGelu / kGemmEpiResidual (the DiT block's epilogues, block.cuh).
template <bool kFP4, int kEpi = 0>
__global__ void __launch_bounds__(Cfg<kFP4>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_sfa,
                const __grid_constant__ CUtensorMap tmap_sfb,
                const __grid_constant__ CUtensorMap tmap_y, const GemmArgs args) {
    using C = Cfg<kFP4>;
    constexpr int S = C::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi = smem + S * C::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi + C::kEpiBytes);  // used in the even CTA
    uint64_t* empty = full + S;
    uint64_t* sf_full = empty + S;    // this CTA's scale tiles landed
    uint64_t* sfready = sf_full + S;  // scales of both CTAs in tensor memory (even CTA)
    uint64_t* tmem_full = sfready + S;
    uint64_t* tmem_empty = tmem_full + 1;  // used in the even CTA
    uint64_t* drain = tmem_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 (even, issues the MMAs) or 1
    const bool leader = rank == 0;
    const int M = args.M, N = args.N, K = args.K;
    const Sched<kFP4> sch(M, N);
    // MMA steps along K: 64 E2M1 (32 bytes) or 16 BF16 (32 bytes) each; 4 per stage.
    const int k_steps = kFP4 ? K / 64 : (K + 15) / 16;
    const int num_kb = (k_steps + 3) / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
            mbar_init(&sfready[s], kSfWarps * kPair);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kEpiWarps * kPair);  // the epilogue warps of both CTAs
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        if (kFP4) {
            prefetch_tmap(&tmap_sfa);
            prefetch_tmap(&tmap_sfb);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers and tensor memory exist from here on
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // NVFP4: each role's branch starts with its warp group's setmaxnreg (every warp of a
    // group executes the same one, converged).

    if (warp == 0) {
        if (kFP4) regs_decrease<kRegsCtl>();
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t full_even = map_to_rank(smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = sch.first; ok && t < sch.total; t += sch.step) {
                int mp, n_blk;
                sch.tile(t, mp, n_blk);
                const int m_blk = mp * kPair + (int)rank;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, args.status, abort_flag,
                                   args.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (kb == args.withhold_kb && leader && t == (int)(blockIdx.x / kPair) &&
                        blockIdx.x < kPair) {
                        // Test hook: this stage's copies are never issued (nor announced), so
                        // the pair's MMA issuer, scale writers and epilogue all run into their
                        // bounded waits.  Nothing is read or written out of place.
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    const uint32_t bar = full_even + 8u * (uint32_t)stage;
                    uint8_t* sa = smem + stage * C::kStageBytes;
                    uint8_t* sb = sa + kATileBytes;
                    if (kFP4) {
                        // Scale tiles first (small; the scale warps start on them while A and
                        // B are in flight): 4 chunks of 512 bytes along K per 128-row tile;
                        // chunks or tiles past the end arrive as zeros.
                        mbar_arrive_expect_tx(&sf_full[stage], C::kSFBytes);
                        uint8_t* sfa = sb + kBHalfBytes;
                        uint8_t* sfb = sfa + kSFAStageBytes;
                        tma_load_4d(&tmap_sfa, &sf_full[stage], sfa, 0, 0, kb * 4, m_blk);
                        tma_load_4d(&tmap_sfb, &sf_full[stage], sfb, 0, 0, kb * 4, 2 * n_blk);
                        tma_load_4d(&tmap_sfb, &sf_full[stage], sfb + 2048, 0, 0, kb * 4,
                                    2 * n_blk + 1);
                    }
                    if (leader) mbar_arrive_expect_tx(&full[stage], kPair * C::kABBytes);
                    const int x = kFP4 ? kb * 128 : kb * 64;
                    tma_load_2d_pair(&tmap_a, bar, sa, x, m_blk * BM);
                    tma_load_2d_pair(&tmap_b, bar, sb, x, n_blk * BN + (int)rank * (BN / kPair));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok && !*abort_flag) {
                // Tail: wait until the last fill of every stage has been released, so no
                // release from the pair's MMAs is still in flight towards this CTA at exit.
                for (int i = 0; i < S; ++i) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, args.status, abort_flag,
                                   args.wait_limit_ns))
                        break;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Give copies already issued time to land before the pair tears down.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (kFP4) regs_decrease<kRegsCtl>();
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const uint32_t idesc = kFP4 ? idesc_nvfp4() : idesc_bf16();
            // Descriptors of stage 0, K-step 0; stage s adds kStageBytes >> 4 and K-step kk
            // adds 32 >> 4 = 2 to the start-address field (never carries: < 256 KB).
            const uint64_t a_desc0 = smem_desc(smem_u32(smem), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(smem_u32(smem) + kATileBytes, 16, 1024, kLayoutSw128);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            bool any_mma = false;
            for (int t = sch.first; ok && t < sch.total; t += sch.step) {
                // The accumulator must have been drained by the epilogue of both CTAs.
                if (!mbar_wait<true>(tmem_empty, acc_phase ^ 1u, args.status, abort_flag,
                                     args.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, args.status, abort_flag, args.wait_limit_ns) ||
                        (kFP4 && !mbar_wait<true>(&sfready[stage], phase, args.status, abort_flag,
                                                  args.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int nk = min(4, k_steps - kb * 4);
                    const uint64_t soff = (uint64_t)((stage * C::kStageBytes) >> 4);
                    const uint32_t sf_col = tmem_base + kSfTmemBase + (uint32_t)stage * kSfTmemPerStage;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (kk < nk) {
                            const uint64_t ad = a_desc0 + soff + 2 * kk;
                            const uint64_t bd = b_desc0 + soff + 2 * kk;
                            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                            if (kFP4)
                                mma_nvfp4_pair(tmem_base, ad, bd, idesc, sf_col + 4 * kk,
                                               sf_col + 16 + 8 * kk, acc);
                            else
                                mma_bf16_pair(tmem_base, ad, bd, idesc, acc);
                        }
                    }
                    any_mma = true;
                    mma_commit_pair_multicast(&empty[stage], kBothCtas);  // release to both CTAs
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(tmem_full, kBothCtas);
                acc_phase ^= 1u;
            }
            if (*abort_flag && any_mma) {
                // Let every MMA this thread issued finish before tensor memory is freed.
                mma_commit_pair_multicast(drain, kEvenCta);
                int dummy_flag = 0;
                mbar_wait(drain, 0, args.status, &dummy_flag, kDrainLimitNs);
            }
        }
    } else if (kFP4 && warp < kSfWarp0) {
        regs_decrease<kRegsCtl>();  // warps 2, 3: no role
    } else if (kFP4 && warp < C::kEpiWarp0) {
        regs_decrease<kRegsSf>();
        // ------------------------------------------------ scale writers (NVFP4, both CTAs)
        // Warp w writes tensor-memory lanes 32 (w % 4) .. +31; lane l of every quarter
        // takes row l of each 512-byte scale chunk (16 bytes: rows l + 32 c, c = 0..3).
        const uint32_t quarter = (uint32_t)(warp & 3);
        const uint32_t lane_base = tmem_base + ((quarter * 32u) << 16);
        const uint32_t sfready_even = map_to_rank(smem_u32(sfready), 0);
        int stage = 0;
        uint32_t phase = 0;
        for (int t = sch.first; t < sch.total; t += sch.step) {
            bool ok = true;
            for (int kb = 0; kb < num_kb; ++kb) {
                ok = mbar_wait(&sf_full[stage], phase, args.status, abort_flag, args.wait_limit_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.st is .sync.aligned
                if (!ok) break;
                const uint8_t* sfa = smem + stage * C::kStageBytes + kATileBytes + kBHalfBytes;
                const uint8_t* sfb = sfa + kSFAStageBytes;
                uint32_t ra[16], rb[32];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint4 a4 = *reinterpret_cast<const uint4*>(sfa + kk * 512 + lane * 16);
                    const uint4 b0 = *reinterpret_cast<const uint4*>(sfb + kk * 512 + lane * 16);
                    const uint4 b1 =
                        *reinterpret_cast<const uint4*>(sfb + 2048 + kk * 512 + lane * 16);
                    ra[4 * kk + 0] = a4.x;
                    ra[4 * kk + 1] = a4.y;
                    ra[4 * kk + 2] = a4.z;
                    ra[4 * kk + 3] = a4.w;
                    rb[8 * kk + 0] = b0.x;  // B rows 0..127 (the even CTA's half)
                    rb[8 * kk + 1] = b0.y;
                    rb[8 * kk + 2] = b0.z;
                    rb[8 * kk + 3] = b0.w;
                    rb[8 * kk + 4] = b1.x;  // B rows 128..255
                    rb[8 * kk + 5] = b1.y;
                    rb[8 * kk + 6] = b1.z;
                    rb[8 * kk + 7] = b1.w;
                }
                const uint32_t col = lane_base + kSfTmemBase + (uint32_t)stage * kSfTmemPerStage;
                tmem_st_32x32b_x16(col, ra);
                tmem_st_32x32b_x32(col + 16, rb);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(sfready_even + 8u * (uint32_t)stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp >= C::kEpiWarp0) {
        if (kFP4) regs_increase<kRegsEpi>();
        // ------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;                // tensor-memory lanes 32*quarter .. +31
        const int ew = warp - C::kEpiWarp0;
        const int half = ew / 4;                     // columns 128*half .. +127
        uint8_t* stg = epi + ew * C::kEpiBufs * kChunkBytes;  // 2048-byte aligned chunks
        uint8_t* sbias = epi + kEpiWarps * C::kEpiBufs * kChunkBytes + ew * kBiasBytes;
        uint32_t chunk_seq = 0;
        const uint32_t tmem_empty_even = map_to_rank(smem_u32(tmem_empty), 0);
        uint32_t acc_phase = 0;
        const float w_scale = kFP4 ? *args.w_st : 1.0f;
        for (int t = sch.first; t < sch.total; t += sch.step) {
            int mp, n_blk;
            sch.tile(t, mp, n_blk);
            const int m_blk = mp * kPair + (int)rank;
            const int row = m_blk * BM + quarter * 32 + lane;
            const int n0 = n_blk * BN + half * 128;
            // Fetch this tile's per-row scale and the warp's 128 bias values while the
            // MMAs run, so no global load sits between the accumulator and the stores.
            float scale = 1.0f;
            if (kFP4) scale = (row < M ? args.a_srow[row] : 0.0f) * w_scale;
            {
                uint2 b2 = make_uint2(0, 0);
                if (args.bias != nullptr && n0 + lane * 4 < N)
                    b2 = __ldg(reinterpret_cast<const uint2*>(args.bias + n0 + lane * 4));
                *reinterpret_cast<uint2*>(sbias + lane * 8) = b2;
            }
            __syncwarp();
            bool ok = mbar_wait(tmem_full, acc_phase, args.status, abort_flag, args.wait_limit_ns);
            // tcgen05.ld is .sync.aligned: reconverge the warp and agree on the outcome.
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            // All four 32-column loads in flight, one wait, then the accumulator is free.
            uint32_t v[4][32];
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tmem_empty_even);
            uint32_t ymax = 0u;  // largest bf16 magnitude of this row's 128 columns (bit pattern)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t packed[16];
                uint32_t rw[16];  // kGemmEpiResidual: this row's 32 residual values of the chunk
                if constexpr (kEpi == kGemmEpiResidual) {
                    const bool in = row < M && n0 + c * 32 < N;  // N % 32 == 0: whole chunks
                    const uint4* rp = reinterpret_cast<const uint4*>(args.residual + (int64_t)row * N + n0 + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 r4 = in ? __ldg(rp + q) : make_uint4(0, 0, 0, 0);
                        rw[4 * q] = r4.x;
                        rw[4 * q + 1] = r4.y;
                        rw[4 * q + 2] = r4.z;
                        rw[4 * q + 3] = r4.w;
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // 8 bias values per 8 columns (shared memory, broadcast to the warp).
                    const uint4 braw = *reinterpret_cast<const uint4*>(sbias + (c * 32 + q * 8) * 2);
                    const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = q * 4 + u;
                        float lo = fmaf(__uint_as_float(v[c][2 * i]), scale, __uint_as_float(bw[u] << 16));
                        float hi = fmaf(__uint_as_float(v[c][2 * i + 1]), scale, __uint_as_float(bw[u] & 0xFFFF0000u));
                        if constexpr (kEpi != 0) {
                            // The plain output's bf16 value first, as the separate pass reads it.
                            const uint32_t yb = pack_bf16x2(lo, hi);
                            lo = __uint_as_float(yb << 16);
                            hi = __uint_as_float(yb & 0xFFFF0000u);
                            if constexpr (kEpi == kGemmEpiGelu) {
                                const float2 g = gelu_f32x2(make_float2(lo, hi));
                                lo = g.x;
                                hi = g.y;
                            } else {
                                lo += __uint_as_float(rw[i] << 16);
                                hi += __uint_as_float(rw[i] & 0xFFFF0000u);
                            }
                        }
                        packed[i] = pack_bf16x2(lo, hi);
                    }
                }
                if (args.row_amax != nullptr) {
                    // Columns past N hold 0 (their accumulators and bias are 0).
#pragma unroll
                    for (int i = 0; i < 16; ++i) ymax = __vmaxu2(ymax, packed[i] & 0x7FFF7FFFu);
                }
                // Row `lane` of the 32x32 bf16 chunk -> staging chunk, 16-byte pieces placed
                // by the 64-byte swizzle of the Y tensor map (piece j of row r at
                // j ^ ((r >> 1) & 3)), then one TMA store of the chunk.
                uint8_t* buf = stg + (chunk_seq % C::kEpiBufs) * kChunkBytes;
                if (chunk_seq >= (uint32_t)C::kEpiBufs) {
                    if (lane == 0) bulk_wait_group_read<C::kEpiBufs - 1>();
                    __syncwarp();
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) =
                        make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                                   packed[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                const int sx = n0 + c * 32, sy = m_blk * BM + quarter * 32;
                if (lane == 0) {
                    // Partial boxes are clipped by TMA; a chunk wholly outside Y is not
                    // stored but still commits its (empty) group, so that every ring slot
                    // owns exactly one group and the wait above is exact.
                    if (sx < N && sy < M) tma_store_2d(&tmap_y, buf, sx, sy);
                    bulk_commit_group();
                }
                ++chunk_seq;
            }
            if (args.row_amax != nullptr && row < M) {
                // |bf16| bit patterns order like the values; as fp32 (<< 16) too.
                const uint32_t mx = max(ymax & 0xFFFFu, ymax >> 16);
                if (mx != 0u) atomicMax(reinterpret_cast<unsigned int*>(args.row_amax + row), mx << 16);
            }
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_group<0>();  // every store of this warp has completed
        __syncwarp();
    }

    // ------------------------------------------------ teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still signal or load towards it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
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

template <bool kFP4, int kEpi = 0>
cudaError_t run_gemm(const LaunchCtx& ctx, const CUtensorMap& ta, const CUtensorMap& tb,
                     const CUtensorMap& tsfa, const CUtensorMap& tsfb, const CUtensorMap& ty,
                     const GemmArgs& args) {
    static OccupancyCache occupancy;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(Cfg<kFP4>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<kFP4>::kSmemBytes;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Co-resident pairs (one CTA per SM), capped by the work available.
    cfg.gridDim = dim3((unsigned)(ctx.num_sms / kPair * kPair), 1, 1);
    int max_clusters = 0;
    const cudaError_t e = clusters_per_device(occupancy, ctx, gemm_kernel<kFP4, kEpi>, cfg, &max_clusters);
    if (e != cudaSuccess) return e;
    const int64_t num_m = (args.M + BM - 1) / BM;
    const int64_t pairs = (num_m + kPair - 1) / kPair * ((args.N + BN - 1) / BN);
    const int64_t clusters = pairs < max_clusters ? pairs : max_clusters;
    cfg.gridDim = dim3((unsigned)(clusters * kPair), 1, 1);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<kFP4, kEpi>, ta, tb, tsfa, tsfb, ty, args);
}

}  // namespace

cudaError_t launch_gemm_nvfp4(const LaunchCtx& ctx, const CUtensorMap& tmap_a,
                              const CUtensorMap& tmap_b, const CUtensorMap& tmap_sfa,
                              const CUtensorMap& tmap_sfb, const CUtensorMap& tmap_y,
                              const float* a_srow, const float* w_st, const __nv_bfloat16* bias,
                              int64_t M, int64_t N, int64_t K, int withhold_kb,
                              int64_t wait_limit_ns, float* row_amax) {
    GemmArgs a{a_srow, w_st, bias, (int)M, (int)N, (int)K, ctx.status,
               wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : kWaitLimitNs, withhold_kb, row_amax};
    return run_gemm<true>(ctx, tmap_a, tmap_b, tmap_sfa, tmap_sfb, tmap_y, a);
}

cudaError_t launch_gemm_bf16(const LaunchCtx& ctx, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                             const __nv_bfloat16* bias, int64_t M, int64_t N, int64_t K) {
    GemmArgs a{nullptr, nullptr, bias, (int)M, (int)N, (int)K, ctx.status, kWaitLimitNs, -1, nullptr};
    return run_gemm<false>(ctx, tmap_a, tmap_b, tmap_a, tmap_b, tmap_y, a);
}

cudaError_t launch_gemm_nvfp4_epi(const LaunchCtx& ctx, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                  const CUtensorMap& tmap_sfa, const CUtensorMap& tmap_sfb,
                                  const CUtensorMap& tmap_y, const float* a_srow, const float* w_st,
                                  const __nv_bfloat16* bias, int64_t M, int64_t N, int64_t K, int epi,
                                  const uint16_t* residual) {
    GemmArgs a{a_srow, w_st, bias, (int)M, (int)N, (int)K, ctx.status, kWaitLimitNs, -1, nullptr, residual};
    if (epi == kGemmEpiGelu) return run_gemm<true, kGemmEpiGelu>(ctx, tmap_a, tmap_b, tmap_sfa, tmap_sfb, tmap_y, a);
    if (epi == kGemmEpiResidual && residual != nullptr && N % 32 == 0)
        return run_gemm<true, kGemmEpiResidual>(ctx, tmap_a, tmap_b, tmap_sfa, tmap_sfb, tmap_y, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_test_wait_timeout(const LaunchCtx& ctx, int64_t timeout_ns) {
    wait_timeout_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, (uint64_t)timeout_ns);
    return cudaGetLastError();
}

}  // namespace nvfp4rl
