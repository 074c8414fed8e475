// Fused attention of the synthetic DiT block on the tcgen05 tensor cores.
//
// Per image b and head h (dh = D/H, 64 or 128), with q, k, v the head's columns of qkv:
//   L = bf16(q k^T)                       (fp32 accumulation, one rounding)
//   P = bf16(softmax(scale L))            (scale = fp32 1/sqrt(dh); exponentials in fp32)
//   O = bf16(P v)                         (fp32 accumulation)
// written straight into o [B*S, D] at columns h*dh.  P is normalised before it is
// rounded, as the definition has it, so the kernel walks the keys twice: pass 1
// forms every tile of L and keeps each row's maximum m and sum of exponentials
// (rescaled when m grows), pass 2 forms the tiles of L again (the same MMAs, so the
// same bits), turns them into P with the final m and 1/sum, and accumulates P v.
//
// One cluster of two CTAs per (image-head, 256 query rows); every MMA is a 2-CTA
// `cta_group::2` MMA (M = 256: each CTA's 128 query rows):
//   L tile   M = 256, N = 128 keys (64 per CTA), K = dh;   A = Q (shared memory),
//            B = K rows (shared memory)
//   O       M = 256, N = dh (dh/2 per CTA), K = 128 keys; A = P (tensor memory),
//            B = V^T rows (shared memory)
// Q and K tiles come from qkv by TMA (128-byte swizzle); V^T [B*H*dh, S] is written
// beforehand by the block's transpose kernel.  Keys past S (the last tile when
// S % 128 == 64) are masked: their logits count as -inf, their P as 0.
//
// Tensor memory per CTA (512 columns): L tiles in 0..127 and 128..255 (double
// buffer), P tiles in 256..319 and 320..383 (64 columns of bf16 pairs each), O in
// 384 .. 384 + dh - 1.
//
// Warps: 0 TMA producer (both CTAs: Q once, then K tiles for pass 1 and K, V tiles
// for pass 2); 1 tensor-memory allocation and, in the even CTA, the MMA issuer;
// 2..5 softmax and output (one row per thread: tensor-memory lane quarter = warp % 4).
// Every wait is bounded (mbar_wait); on expiry the kernel records NVFP4_ERR_TIMEOUT,
// lets its copies and MMAs land, frees tensor memory and returns.
#include "block.cuh"

namespace nvfp4rl {
namespace {

constexpr int kPairCtas = 2;
constexpr int kRowsCta = 128;    // query rows per CTA
constexpr int kTileKeys = 128;   // keys per L tile (64 per CTA)
constexpr int kStagesK = 4;
constexpr int kStagesV = 4;
constexpr int kSoftWarp0 = 2;
constexpr int kSoftWarps = 4;
constexpr int kAttnThreads = (kSoftWarp0 + kSoftWarps) * 32;
constexpr uint32_t kTmemColsAttn = 512;
constexpr uint32_t kColL = 0, kColP = 256, kColO = 384;
constexpr uint16_t kBoth = 0x3, kEven = 0x1;
constexpr uint64_t kAttnWaitNs = 4000000000ull;
constexpr uint64_t kAttnDrainNs = 200000000ull;

template <int kDh>
struct AttnCfg {
    static_assert(kDh == 64 || kDh == 128, "head width");
    static constexpr uint32_t kQSub = kRowsCta * 128;                 // one 64-column atom of Q
    static constexpr uint32_t kQBytes = kQSub * (kDh / 64);
    static constexpr uint32_t kKSub = (kTileKeys / kPairCtas) * 128;   // 64 keys x 64 columns
    static constexpr uint32_t kKBytes = kKSub * (kDh / 64);
    static constexpr uint32_t kVSub = (kDh / kPairCtas) * 128;         // dh/2 rows x 64 keys
    static constexpr uint32_t kVBytes = kVSub * (kTileKeys / 64);
    static constexpr uint32_t kBarBytes = 512;
    static constexpr uint32_t kSmemBytes =
        1024 + kQBytes + kStagesK * kKBytes + kStagesV * kVBytes + kBarBytes;
    // kind::f16, bf16 A and B, fp32 accumulator, both K-major, M = 256.
    static constexpr uint32_t idesc(uint32_t n) {
        return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(kRowsCta * kPairCtas >> 4) << 24);
    }
};
static_assert(AttnCfg<128>::kSmemBytes <= 232448, "shared memory budget");
static_assert(kColO + 128 <= kTmemColsAttn, "tensor memory budget");

struct AttnArgs {
    uint16_t* o;
    int S, D, H, nqb;   // nqb: 256-row query blocks per head
    float c;            // scale * log2(e)
    int* status;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair (round to nearest even) of two fp32 values: lo in bits 0..15.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The 128 logits of this thread's row in one L tile, rounded to bf16 (pairs), with
// the columns at and past `valid` set to -inf.
__device__ __forceinline__ void round_tile(const uint32_t (&v)[4][32], int valid, uint32_t (&lb)[64]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i)
            lb[c * 16 + i] = bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
    if (valid < kTileKeys) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
            if (2 * i >= valid) lb[i] = 0xFF80FF80u;  // both halves -inf (valid is even)
    }
}

template <int kDh>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnArgs args) {
    using C = AttnCfg<kDh>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sq = smem;
    uint8_t* sk = sq + C::kQBytes;
    uint8_t* sv = sk + kStagesK * C::kKBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sv + kStagesV * C::kVBytes);
    uint64_t* q_full = bars;
    uint64_t* k_full = q_full + 1;
    uint64_t* k_empty = k_full + kStagesK;
    uint64_t* v_full = k_empty + kStagesK;
    uint64_t* v_empty = v_full + kStagesV;
    uint64_t* s_full = v_empty + kStagesV;   // [2]
    uint64_t* s_empty = s_full + 2;          // [2], even CTA
    uint64_t* p_full = s_empty + 2;          // [2], even CTA
    uint64_t* p_free = p_full + 2;           // [2]
    uint64_t* o_full = p_free + 2;
    uint64_t* drain = o_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int S = args.S, D = args.D, H = args.H;
    const int item = (int)(blockIdx.x / kPairCtas);
    const int z = item / args.nqb, qb = item - z * args.nqb;
    const int b = z / H, h = z - b * H;
    const int n_tiles = (S + kTileKeys - 1) / kTileKeys;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], kSoftWarps * kPairCtas);
            mbar_init(&p_full[i], kSoftWarps * kPairCtas);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemColsAttn);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t q_full_e = map_to_rank(smem_u32(q_full), 0);
            const uint32_t k_full_e = map_to_rank(smem_u32(k_full), 0);
            const uint32_t v_full_e = map_to_rank(smem_u32(v_full), 0);
            const int row0 = b * S;
            const int qcol = h * kDh, kcol = D + h * kDh;
            bool ok = true;
            if (leader) mbar_arrive_expect_tx(q_full, kPairCtas * C::kQBytes);
#pragma unroll
            for (int i = 0; i < kDh / 64; ++i)
                tma_load_2d_pair(&tmap_q, q_full_e, sq + i * C::kQSub, qcol + 64 * i,
                                 row0 + qb * (kRowsCta * kPairCtas) + (int)rank * kRowsCta);
            int kc = 0, vc = 0;
            for (int pass = 0; ok && pass < 2; ++pass) {
                for (int j = 0; j < n_tiles; ++j) {
                    {
                        const int s = kc % kStagesK;
                        if (!mbar_wait(&k_empty[s], (uint32_t)(((kc / kStagesK) & 1) ^ 1), args.status, abort_flag,
                                       kAttnWaitNs)) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&k_full[s], kPairCtas * C::kKBytes);
                        uint8_t* dst = sk + s * C::kKBytes;
#pragma unroll
                        for (int i = 0; i < kDh / 64; ++i)
                            tma_load_2d_pair(&tmap_k, k_full_e + 8u * (uint32_t)s, dst + i * C::kKSub, kcol + 64 * i,
                                             row0 + j * kTileKeys + (int)rank * (kTileKeys / kPairCtas));
                        ++kc;
                    }
                    if (pass == 1) {
                        const int s = vc % kStagesV;
                        if (!mbar_wait(&v_empty[s], (uint32_t)(((vc / kStagesV) & 1) ^ 1), args.status, abort_flag,
                                       kAttnWaitNs)) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&v_full[s], kPairCtas * C::kVBytes);
                        uint8_t* dst = sv + s * C::kVBytes;
#pragma unroll
                        for (int i = 0; i < kTileKeys / 64; ++i)
                            tma_load_2d_pair(&tmap_v, v_full_e + 8u * (uint32_t)s, dst + i * C::kVSub,
                                             j * kTileKeys + 64 * i, z * kDh + (int)rank * (kDh / kPairCtas));
                        ++vc;
                    }
                }
            }
            if (ok && !*abort_flag) {
                // Tail: the releases of the last fills land before this CTA leaves.
                for (int i = (kc > kStagesK ? kc - kStagesK : 0); i < kc; ++i)
                    if (!mbar_wait(&k_empty[i % kStagesK], (uint32_t)((i / kStagesK) & 1), args.status, abort_flag,
                                   kAttnWaitNs))
                        break;
                for (int i = (vc > kStagesV ? vc - kStagesV : 0); i < vc; ++i)
                    if (!mbar_wait(&v_empty[i % kStagesV], (uint32_t)((i / kStagesV) & 1), args.status, abort_flag,
                                   kAttnWaitNs))
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
            const uint32_t idesc_l = C::idesc(kTileKeys), idesc_o = C::idesc(kDh);
            const uint64_t q_desc = smem_desc(smem_u32(sq), 16, 1024, kLayoutSw128);
            const uint64_t k_desc0 = smem_desc(smem_u32(sk), 16, 1024, kLayoutSw128);
            const uint64_t v_desc0 = smem_desc(smem_u32(sv), 16, 1024, kLayoutSw128);
            bool ok = mbar_wait(q_full, 0, args.status, abort_flag, kAttnWaitNs);
            bool any = false;
            int kc = 0, g = 0;
            // One L tile: wait for its K stage and a free L buffer, dh/16 MMAs, release.
            auto issue_l = [&]() -> bool {
                const int s = kc % kStagesK, lb = g & 1;
                if (!mbar_wait(&k_full[s], (uint32_t)((kc / kStagesK) & 1), args.status, abort_flag, kAttnWaitNs) ||
                    !mbar_wait<true>(&s_empty[lb], (uint32_t)(((g >> 1) & 1) ^ 1), args.status, abort_flag,
                                     kAttnWaitNs))
                    return false;
                tc_fence_after_sync();
                const uint64_t kd = k_desc0 + (uint64_t)((s * C::kKBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kDh / 16; ++kk) {
                    const uint64_t off = (uint64_t)((kk >> 2) * 0 + (kk & 3) * 2);
                    mma_bf16_pair(tmem_base + kColL + (uint32_t)(lb * kTileKeys),
                                  q_desc + (uint64_t)((kk >> 2) * (C::kQSub >> 4)) + off,
                                  kd + (uint64_t)((kk >> 2) * (C::kKSub >> 4)) + off, idesc_l, kk > 0 ? 1u : 0u);
                }
                any = true;
                mma_commit_pair_multicast(&k_empty[s], kBoth);
                mma_commit_pair_multicast(&s_full[lb], kBoth);
                ++kc;
                ++g;
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) ok = issue_l();  // pass 1
            if (ok) ok = issue_l();                                  // pass 2, tile 0
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !(ok = issue_l())) break;
                const int s = j % kStagesV, pb = j & 1;
                if (!mbar_wait(&v_full[s], (uint32_t)((j / kStagesV) & 1), args.status, abort_flag, kAttnWaitNs) ||
                    !mbar_wait<true>(&p_full[pb], (uint32_t)((j >> 1) & 1), args.status, abort_flag, kAttnWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t vd = v_desc0 + (uint64_t)((s * C::kVBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk)
                    mma_bf16_pair_ta(tmem_base + kColO, tmem_base + kColP + (uint32_t)(pb * 64) + 8u * (uint32_t)kk,
                                     vd + (uint64_t)((kk >> 2) * (C::kVSub >> 4) + (kk & 3) * 2), idesc_o,
                                     (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit_pair_multicast(&v_empty[s], kBoth);
                mma_commit_pair_multicast(&p_free[pb], kBoth);
            }
            if (ok) mma_commit_pair_multicast(o_full, kBoth);
            if (*abort_flag && any) {
                mma_commit_pair_multicast(drain, kEven);
                int dummy = 0;
                mbar_wait(drain, 0, args.status, &dummy, kAttnDrainNs);
            }
        }
    } else {
        // ------------------------------------------------ softmax and output (both CTAs)
        const int quarter = warp & 3;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_empty_e = map_to_rank(smem_u32(s_empty), 0);
        const uint32_t p_full_e = map_to_rank(smem_u32(p_full), 0);
        const float c = args.c;
        float m = -INFINITY, sum = 0.0f, inv = 0.0f;
        bool ok = true;
        for (int g = 0; ok && g < 2 * n_tiles; ++g) {
            const int j = g < n_tiles ? g : g - n_tiles;
            const int lb = g & 1;
            const int valid = min(kTileKeys, S - j * kTileKeys);
            ok = mbar_wait(&s_full[lb], (uint32_t)((g >> 1) & 1), args.status, abort_flag, kAttnWaitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld is .sync.aligned
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t v[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x32(lane_base + kColL + (uint32_t)(lb * kTileKeys + q * 32), v[q]);
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(s_empty_e + 8u * (uint32_t)lb);
            uint32_t lbits[64];
            round_tile(v, valid, lbits);
            if (g < n_tiles) {
                // Pass 1: running maximum and rescaled sum of exponentials.
                uint32_t mx2 = lbits[0];
#pragma unroll
                for (int i = 1; i < 64; ++i) mx2 = bmax2(mx2, lbits[i]);
                const float tmax = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
                const float m_new = fmaxf(m, tmax);
                const float mc = m_new * c;
                float acc = sum * ex2(fmaf(m, c, -mc));
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    acc += ex2(fmaf(__uint_as_float(lbits[i] << 16), c, -mc));
                    acc += ex2(fmaf(__uint_as_float(lbits[i] & 0xFFFF0000u), c, -mc));
                }
                sum = acc;
                m = m_new;
                if (g == n_tiles - 1) inv = 1.0f / sum;
            } else {
                // Pass 2: P = bf16(exp(scale (l - m)) / sum) into tensor memory.
                const float mc = m * c;
                uint32_t p[2][32];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float e0 = ex2(fmaf(__uint_as_float(lbits[i] << 16), c, -mc)) * inv;
                    const float e1 = ex2(fmaf(__uint_as_float(lbits[i] & 0xFFFF0000u), c, -mc)) * inv;
                    p[i >> 5][i & 31] = bf16x2(e0, e1);
                }
                const int pb = j & 1;
                ok = mbar_wait(&p_free[pb], (uint32_t)(((j >> 1) & 1) ^ 1), args.status, abort_flag, kAttnWaitNs);
                ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.st is .sync.aligned
                if (!ok) break;
                tc_fence_after_sync();
                tmem_st_32x32b_x32(lane_base + kColP + (uint32_t)(pb * 64), p[0]);
                tmem_st_32x32b_x32(lane_base + kColP + (uint32_t)(pb * 64 + 32), p[1]);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(p_full_e + 8u * (uint32_t)pb);
            }
        }
        if (ok) {
            ok = mbar_wait(o_full, 0, args.status, abort_flag, kAttnWaitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);
        }
        if (ok) {
            tc_fence_after_sync();
            uint32_t v[kDh / 32][32];
#pragma unroll
            for (int q = 0; q < kDh / 32; ++q) tmem_ld_32x32b_x32(lane_base + kColO + (uint32_t)(q * 32), v[q]);
            tmem_ld_wait();
            const int s = qb * (kRowsCta * kPairCtas) + (int)rank * kRowsCta + quarter * 32 + lane;
            if (s < S) {
                uint4* dst = reinterpret_cast<uint4*>(args.o + ((int64_t)b * S + s) * D + (int64_t)h * kDh);
#pragma unroll
                for (int q = 0; q < kDh / 32; ++q)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[q * 4 + i] = make_uint4(
                            bf16x2(__uint_as_float(v[q][8 * i + 0]), __uint_as_float(v[q][8 * i + 1])),
                            bf16x2(__uint_as_float(v[q][8 * i + 2]), __uint_as_float(v[q][8 * i + 3])),
                            bf16x2(__uint_as_float(v[q][8 * i + 4]), __uint_as_float(v[q][8 * i + 5])),
                            bf16x2(__uint_as_float(v[q][8 * i + 6]), __uint_as_float(v[q][8 * i + 7])));
            }
        }
    }

    // ------------------------------------------------ teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemColsAttn);
    }
}

template <int kDh>
cudaError_t run_attn(const LaunchCtx& ctx, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const AttnArgs& args, int64_t items) {
    static bool configured[kMaxDevices] = {};
    if (!configured[ctx.device]) {
        const cudaError_t e = cudaFuncSetAttribute(attn_kernel<kDh>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)AttnCfg<kDh>::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[ctx.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPairCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = AttnCfg<kDh>::kSmemBytes;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(items * kPairCtas), 1, 1);
    return cudaLaunchKernelEx(&cfg, attn_kernel<kDh>, tq, tk, tv, args);
}

}  // namespace

cudaError_t launch_attention(const LaunchCtx& ctx, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                             const CUtensorMap& tmap_vt, uint16_t* o, int64_t B, int64_t S, int64_t D, int64_t H,
                             float scale) {
    const int64_t dh = D / H;
    const int64_t nqb = (S + kRowsCta * kPairCtas - 1) / (kRowsCta * kPairCtas);
    const int64_t items = B * H * nqb;
    if (items <= 0 || items * kPairCtas > 0x7FFFFFFF) return cudaErrorInvalidValue;
    AttnArgs a{o, (int)S, (int)D, (int)H, (int)nqb, scale * 1.4426950408889634f, ctx.status};
    if (dh == 128) return run_attn<128>(ctx, tmap_q, tmap_k, tmap_vt, a, items);
    if (dh == 64) return run_attn<64>(ctx, tmap_q, tmap_k, tmap_vt, a, items);
    return cudaErrorInvalidValue;
}

}  // namespace nvfp4rl
