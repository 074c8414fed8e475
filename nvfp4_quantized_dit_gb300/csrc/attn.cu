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
// Persistent clusters of two CTAs (one per SM), each walking items (image-head, 256
// query rows); every MMA is a 2-CTA `cta_group::2` MMA (M = 256: each CTA's 128 query
// rows).  The next item's Q loads once the current item's last L tile is formed, and
// its first P v waits until the current item's O has been read out of tensor memory:
//   L tile   M = 256, N = 256 keys (128 per CTA), K = dh;  A = Q (shared memory),
//            B = K rows (shared memory)
//   O       M = 256, N = dh (dh/2 per CTA), K = 256 keys; A = P (tensor memory),
//            B = V^T rows (shared memory)
// Q and K tiles come from qkv by TMA (128-byte swizzle); V^T [B*H*dh, S] is written
// beforehand by the block's transpose kernel.  Keys past S (the last tile when
// S % 256 != 0) are masked: their logits count as -inf, their P as 0.
//
// Tensor memory per CTA (512 columns): the L tile in 0..255, P in 256..383 (bf16
// pairs), O in 384 .. 384 + dh - 1.  The L tile is read into registers at once, so
// the next tile's MMAs run while the softmax works on the last one.
//
// Warps: 0 TMA producer (both CTAs: Q once, then K tiles for pass 1 and K, V tiles
// for pass 2); 1 tensor-memory allocation and, in the even CTA, the MMA issuer;
// 2..17 softmax and output: one query row per thread (tensor-memory lane quarter =
// warp % 4), four warps per quarter, each with a quarter of the columns of every L
// tile and of O; the four partial maxima and sums of a row are combined once,
// between the passes.
// Every wait is bounded (mbar_wait); on expiry the kernel records NVFP4_ERR_TIMEOUT,
// lets its copies and MMAs land, frees tensor memory and returns.
#include "block.cuh"

namespace nvfp4rl {
namespace {

constexpr int kPairCtas = 2;
constexpr int kRowsCta = 128;    // query rows per CTA
constexpr int kTileKeys = 256;   // keys per L tile (128 per CTA)
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
constexpr int kSoftWarp0 = 2;
constexpr int kSoftWarps = 16;                   // four per tensor-memory lane quarter
constexpr int kSlices = kSoftWarps / 4;          // column slices of a tile, one per warp of a quarter
constexpr int kSliceCols = kTileKeys / kSlices;  // 64 logits of a row per warp and tile
constexpr int kChunk = 32;                       // columns per tensor-memory load
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
    static constexpr uint32_t kKSub = (kTileKeys / kPairCtas) * 128;   // 128 keys x 64 columns
    static constexpr uint32_t kKBytes = kKSub * (kDh / 64);
    static constexpr uint32_t kVSub = (kDh / kPairCtas) * 128;         // dh/2 rows x 64 keys
    static constexpr uint32_t kVBytes = kVSub * (kTileKeys / 64);
    // barriers; (m, sum) per item parity, slice and row
    static constexpr uint32_t kBarBytes = 512 + 2 * kSlices * 2 * kRowsCta * 4;
    static constexpr uint32_t kSmemBytes =
        1024 + kQBytes + kStagesK * kKBytes + kStagesV * kVBytes + kBarBytes;
    // kind::f16, bf16 A and B, fp32 accumulator, both K-major, M = 256.
    static constexpr uint32_t idesc(uint32_t n) {
        return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(kRowsCta * kPairCtas >> 4) << 24);
    }
};
static_assert(AttnCfg<128>::kSmemBytes <= 232448, "shared memory budget");
static_assert(kColO + 128 <= kTmemColsAttn, "tensor memory budget");
static_assert(32 * 8 + 8 <= 512, "barrier area");

struct AttnArgs {
    uint16_t* o;
    int S, D, H, nqb;   // nqb: 256-row query blocks per head
    int items;          // B * H * nqb
    float c;            // scale * log2(e)
    int* status;
    uint64_t wait_ns;   // bound of every wait (kAttnWaitNs; shorter in the test hook)
    int withhold;       // test hook only: K tile of pass 1 that the first pair never loads for its
                        // first item (nothing issued, nothing announced), or -1
};

// 2^x (hardware approximation; results below 2^-126 flush to zero, which changes no
// sum of exponentials that includes the row maximum's 1, nor any P that bf16 keeps
// above the products' rounding).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// kChunk logits of this thread's row (columns col .. col + kChunk - 1 of an L tile),
// rounded to bf16 (pairs) into lb, with the columns at and past `valid` set to -inf.
__device__ __forceinline__ void round_chunk(const uint32_t (&v)[kChunk], int col, int valid, uint32_t* lb) {
#pragma unroll
    for (int i = 0; i < kChunk / 2; ++i) lb[i] = bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    if (col + kChunk > valid) {
#pragma unroll
        for (int i = 0; i < kChunk / 2; ++i)
            if (col + 2 * i >= valid) lb[i] = 0xFF80FF80u;  // both halves -inf (valid is even)
    }
}

// The two fp32 values of a bf16 pair.
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

template <int kDh>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_qk, const __grid_constant__ CUtensorMap tmap_v,
                const AttnArgs args) {
    using C = AttnCfg<kDh>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sq = smem;
    uint8_t* sk = sq + C::kQBytes;
    uint8_t* sv = sk + kStagesK * C::kKBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sv + kStagesV * C::kVBytes);
    uint64_t* q_full = bars;                 // Q of the pair's current item has landed (even CTA)
    uint64_t* q_empty = q_full + 1;          // ... and its last L tile's MMAs have read it
    uint64_t* k_full = q_empty + 1;
    uint64_t* k_empty = k_full + kStagesK;
    uint64_t* v_full = k_empty + kStagesK;
    uint64_t* v_empty = v_full + kStagesV;
    uint64_t* s_full = v_empty + kStagesV;   // the L tile is in tensor memory
    uint64_t* s_empty = s_full + 1;          // ... and has been read (even CTA)
    uint64_t* p_full = s_empty + 1;          // P is in tensor memory (even CTA)
    uint64_t* p_free = p_full + 1;           // ... and has been read by the P v MMAs
    uint64_t* o_full = p_free + 1;           // the item's O is complete in tensor memory
    uint64_t* o_free = o_full + 1;           // ... and has been read out (even CTA)
    uint64_t* drain = o_free + 1;
    uint64_t* stats_ready = drain + 1;       // every softmax thread has written its (m, sum)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stats_ready + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // [item parity][slice][m|sum][row]
    float* row_stats = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int S = args.S, D = args.D, H = args.H;
    const int n_tiles = (S + kTileKeys - 1) / kTileKeys;
    // Items (image-head, 256 query rows) of this pair: first, first + step, ...
    const int first = (int)(blockIdx.x / kPairCtas), step = (int)(gridDim.x / kPairCtas);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_empty, kSoftWarps * kPairCtas);
        mbar_init(p_full, kSoftWarps * kPairCtas);
        mbar_init(p_free, 1);
        mbar_init(o_full, 1);
        mbar_init(o_free, kSoftWarps * kPairCtas);
        mbar_init(drain, 1);
        mbar_init(stats_ready, kSoftWarps * 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_qk);
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
            bool ok = true;
            int kc = 0, vc = 0, it = 0;
            for (int item = first; ok && item < args.items; item += step, ++it) {
                const int z = item / args.nqb, qb = item - z * args.nqb;
                const int b = z / H, h = z - b * H;
                const int row0 = b * S;
                const int qcol = h * kDh, kcol = D + h * kDh;
                // Q: once the previous item's last L tile has been formed.
                if (!mbar_wait(q_empty, (uint32_t)((it & 1) ^ 1), args.status, abort_flag, args.wait_ns)) break;
                if (leader) mbar_arrive_expect_tx(q_full, kPairCtas * C::kQBytes);
#pragma unroll
                for (int i = 0; i < kDh / 64; ++i)
                    tma_load_2d_pair(&tmap_qk, q_full_e, sq + i * C::kQSub, qcol + 64 * i,
                                     row0 + qb * (kRowsCta * kPairCtas) + (int)rank * kRowsCta);
                for (int pass = 0; ok && pass < 2; ++pass) {
                    for (int j = 0; j < n_tiles; ++j) {
                        if (pass == 0 && j == args.withhold && it == 0 && first == 0) {
                            // Test hook: this K tile is never loaded nor announced, so the pair's
                            // MMA issuer and softmax warps run into their bounded waits.
                            ++kc;
                            continue;
                        }
                        {
                            const int s = kc % kStagesK;
                            if (!mbar_wait(&k_empty[s], (uint32_t)(((kc / kStagesK) & 1) ^ 1), args.status,
                                           abort_flag, args.wait_ns)) {
                                ok = false;
                                break;
                            }
                            if (leader) mbar_arrive_expect_tx(&k_full[s], kPairCtas * C::kKBytes);
                            uint8_t* dst = sk + s * C::kKBytes;
#pragma unroll
                            for (int i = 0; i < kDh / 64; ++i)
                                tma_load_2d_pair(&tmap_qk, k_full_e + 8u * (uint32_t)s, dst + i * C::kKSub,
                                                 kcol + 64 * i,
                                                 row0 + j * kTileKeys + (int)rank * (kTileKeys / kPairCtas));
                            ++kc;
                        }
                        if (pass == 1) {
                            const int s = vc % kStagesV;
                            if (!mbar_wait(&v_empty[s], (uint32_t)(((vc / kStagesV) & 1) ^ 1), args.status,
                                           abort_flag, args.wait_ns)) {
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
            }
            if (ok && !*abort_flag) {
                // Tail: the releases of the last fills land before this CTA leaves.
                for (int i = (kc > kStagesK ? kc - kStagesK : 0); i < kc; ++i)
                    if (!mbar_wait(&k_empty[i % kStagesK], (uint32_t)((i / kStagesK) & 1), args.status, abort_flag,
                                   args.wait_ns))
                        break;
                for (int i = (vc > kStagesV ? vc - kStagesV : 0); i < vc; ++i)
                    if (!mbar_wait(&v_empty[i % kStagesV], (uint32_t)((i / kStagesV) & 1), args.status, abort_flag,
                                   args.wait_ns))
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
            bool ok = true, any = false;
            // Running counts over the pair's items: K stages, L tiles, P tiles, V stages.
            int kc = 0, g = 0, pj = 0, vc = 0, it = 0;
            // One L tile: wait for its K stage and for the previous tile to have been read,
            // dh/16 MMAs, release the stage, announce the tile.
            auto issue_l = [&]() -> bool {
                const int s = kc % kStagesK;
                if (!mbar_wait(&k_full[s], (uint32_t)((kc / kStagesK) & 1), args.status, abort_flag, args.wait_ns) ||
                    !mbar_wait<true>(s_empty, (uint32_t)((g & 1) ^ 1), args.status, abort_flag, args.wait_ns))
                    return false;
                tc_fence_after_sync();
                const uint64_t kd = k_desc0 + (uint64_t)((s * C::kKBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kDh / 16; ++kk)
                    mma_bf16_pair(tmem_base + kColL,
                                  q_desc + (uint64_t)((kk >> 2) * (C::kQSub >> 4) + (kk & 3) * 2),
                                  kd + (uint64_t)((kk >> 2) * (C::kKSub >> 4) + (kk & 3) * 2), idesc_l, kk > 0 ? 1u : 0u);
                any = true;
                mma_commit_pair_multicast(&k_empty[s], kBoth);
                mma_commit_pair_multicast(s_full, kBoth);
                ++kc;
                ++g;
                return true;
            };
            for (int item = first; ok && item < args.items; item += step, ++it) {
                if (!(ok = mbar_wait(q_full, (uint32_t)(it & 1), args.status, abort_flag, args.wait_ns))) break;
                // L tiles of both passes in order; in pass 2 tile j + 1 is queued before the
                // P v of tile j, so it is ready when the softmax is.  After the item's last L
                // tile Q is released to the producer (the next item's Q loads meanwhile).
                for (int j = 0; ok && j < n_tiles + 1; ++j) ok = issue_l();
                if (ok && n_tiles == 1) mma_commit_pair_multicast(q_empty, kBoth);
                for (int j = 0; ok && j < n_tiles; ++j, ++pj, ++vc) {
                    if (j + 1 < n_tiles) {
                        if (!(ok = issue_l())) break;
                        if (j + 2 == n_tiles) mma_commit_pair_multicast(q_empty, kBoth);
                    }
                    const int s = vc % kStagesV;
                    if (!mbar_wait(&v_full[s], (uint32_t)((vc / kStagesV) & 1), args.status, abort_flag, args.wait_ns) ||
                        !mbar_wait<true>(p_full, (uint32_t)(pj & 1), args.status, abort_flag, args.wait_ns) ||
                        // The first P v of an item overwrites O: the previous item's O must
                        // have been read out.
                        (j == 0 && !mbar_wait<true>(o_free, (uint32_t)((it & 1) ^ 1), args.status, abort_flag,
                                                    args.wait_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t vd = v_desc0 + (uint64_t)((s * C::kVBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileKeys / 16; ++kk)
                        mma_bf16_pair_ta(tmem_base + kColO, tmem_base + kColP + 8u * (uint32_t)kk,
                                         vd + (uint64_t)((kk >> 2) * (C::kVSub >> 4) + (kk & 3) * 2), idesc_o,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair_multicast(&v_empty[s], kBoth);
                    mma_commit_pair_multicast(p_free, kBoth);
                }
                if (ok) mma_commit_pair_multicast(o_full, kBoth);
            }
            if (*abort_flag && any) {
                mma_commit_pair_multicast(drain, kEven);
                int dummy = 0;
                mbar_wait(drain, 0, args.status, &dummy, kAttnDrainNs);
            }
        }
    } else {
        // ------------------------------------------------ softmax and output (both CTAs)
        // Warp w: tensor-memory lanes 32 (w % 4) .. +31 (one query row per thread) and
        // column slice (w - 2) / 4 of every L tile and of O.
        const int quarter = warp & 3, slice = (warp - kSoftWarp0) / 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_empty_e = map_to_rank(smem_u32(s_empty), 0);
        const uint32_t p_full_e = map_to_rank(smem_u32(p_full), 0);
        const uint32_t o_free_e = map_to_rank(smem_u32(o_free), 0);
        const float c = args.c;
        const float2 c2 = make_float2(c, c);
        const int col0 = slice * kSliceCols;
        bool ok = true;
        int gg = 0, pj = 0, it = 0;  // running counts: L tiles, P tiles, items
        for (int item = first; ok && item < args.items; item += step, ++it) {
            const int z = item / args.nqb, qb = item - z * args.nqb;
            const int b = z / H, h = z - b * H;
            float* stats = row_stats + (it & 1) * (kSlices * 2 * kRowsCta);
            float m = -INFINITY, sum = 0.0f, mc2 = 0.0f;
            for (int g = 0; ok && g < 2 * n_tiles; ++g, ++gg) {
                const int j = g < n_tiles ? g : g - n_tiles;
                const int valid = min(kTileKeys, S - j * kTileKeys);
                ok = mbar_wait(s_full, (uint32_t)(gg & 1), args.status, abort_flag, args.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld is .sync.aligned
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t lbits[kSliceCols / 2];
#pragma unroll
                for (int ch = 0; ch < kSliceCols / kChunk; ++ch) {
                    uint32_t v[kChunk];
                    tmem_ld_32x32b_x32(lane_base + kColL + (uint32_t)(col0 + ch * kChunk), v);
                    tmem_ld_wait();
                    round_chunk(v, col0 + ch * kChunk, valid, lbits + ch * (kChunk / 2));
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(s_empty_e);
                if (g < n_tiles) {
                    // Pass 1: running maximum and rescaled sum of exponentials (packed pairs,
                    // four partial sums, so that the additions do not form one chain).
                    uint32_t mx2 = lbits[0];
#pragma unroll
                    for (int i = 1; i < kSliceCols / 2; ++i) mx2 = bmax2(mx2, lbits[i]);
                    const float tmax = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
                    const float m_new = fmaxf(m, tmax);
                    // A slice whose columns so far were all masked (m_new = -inf) keeps sum = 0:
                    // with the offset 0 every term is 2^-inf = 0 (no inf - inf).
                    const float mc = m_new == -INFINITY ? 0.0f : m_new * c;
                    const float2 nmc = make_float2(-mc, -mc);
                    float2 acc[4] = {make_float2(sum * ex2(fmaf(m, c, -mc)), 0.0f), make_float2(0.0f, 0.0f),
                                     make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
                    for (int i = 0; i < kSliceCols / 2; ++i) {
                        const float2 a = __ffma2_rn(unpack_bf16x2(lbits[i]), c2, nmc);
                        acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(ex2(a.x), ex2(a.y)));
                    }
                    const float2 s01 = __fadd2_rn(acc[0], acc[1]), s23 = __fadd2_rn(acc[2], acc[3]);
                    const float2 s4 = __fadd2_rn(s01, s23);
                    sum = s4.x + s4.y;
                    m = m_new;
                    if (g == n_tiles - 1) {
                        // The row's slices: combine their (m, sum) through shared memory (one
                        // buffer per item parity, so a warp ahead on the next item cannot
                        // overwrite values another warp still reads).
                        stats[(slice * 2 + 0) * kRowsCta + row] = m;
                        stats[(slice * 2 + 1) * kRowsCta + row] = sum;
                        mbar_arrive(stats_ready);
                        ok = mbar_wait(stats_ready, (uint32_t)(it & 1), args.status, abort_flag, args.wait_ns);
                        ok = __all_sync(0xFFFFFFFFu, ok);
                        if (!ok) break;
                        float ms[kSlices], ss[kSlices], mm = -INFINITY;
#pragma unroll
                        for (int k = 0; k < kSlices; ++k) {
                            ms[k] = stats[(k * 2 + 0) * kRowsCta + row];
                            ss[k] = stats[(k * 2 + 1) * kRowsCta + row];
                            mm = fmaxf(mm, ms[k]);
                        }
                        float total = 0.0f;
#pragma unroll
                        for (int k = 0; k < kSlices; ++k) total += ss[k] * ex2(fmaf(ms[k], c, -mm * c));
                        // P = exp(scale (l - m)) / sum = 2^(l c - (m c + log2(sum))).
                        mc2 = fmaf(mm, c, lg2(total));
                    }
                } else {
                    // Pass 2: P = bf16(exp(scale (l - m)) / sum) into tensor memory.
                    const float2 nmc = make_float2(-mc2, -mc2);
                    uint32_t p[kSliceCols / 2];
#pragma unroll
                    for (int i = 0; i < kSliceCols / 2; ++i) {
                        const float2 a = __ffma2_rn(unpack_bf16x2(lbits[i]), c2, nmc);
                        p[i] = bf16x2(ex2(a.x), ex2(a.y));
                    }
                    ok = mbar_wait(p_free, (uint32_t)((pj & 1) ^ 1), args.status, abort_flag, args.wait_ns);
                    ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.st is .sync.aligned
                    if (!ok) break;
                    tc_fence_after_sync();
                    tmem_st_32x32b_x32(lane_base + kColP + (uint32_t)(slice * (kSliceCols / 2)), p);
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(p_full_e);
                    ++pj;
                }
            }
            if (ok) {
                ok = mbar_wait(o_full, (uint32_t)(it & 1), args.status, abort_flag, args.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);
            }
            if (!ok) break;
            // O: this warp's dh / 4 columns of its 32 rows; then O's columns are free for
            // the next item's P v.
            constexpr int kOCols = kDh / kSlices;
            tc_fence_after_sync();
            uint32_t v[kOCols];
            const uint32_t oaddr = lane_base + kColO + (uint32_t)(slice * kOCols);
            if constexpr (kOCols == 32) {
                tmem_ld_32x32b_x32(oaddr, v);
            } else {
                tmem_ld_32x32b_x16(oaddr, v);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(o_free_e);
            const int s = qb * (kRowsCta * kPairCtas) + (int)rank * kRowsCta + row;
            if (s < S) {
                uint4* dst = reinterpret_cast<uint4*>(args.o + ((int64_t)b * S + s) * D + (int64_t)h * kDh +
                                                      slice * kOCols);
#pragma unroll
                for (int i = 0; i < kOCols / 8; ++i)
                    dst[i] = make_uint4(bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                                        bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                                        bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                                        bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
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
cudaError_t run_attn(const LaunchCtx& ctx, const CUtensorMap& tqk, const CUtensorMap& tv, const AttnArgs& args) {
    static OccupancyCache occupancy;
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
    // Persistent: the co-resident pairs (one CTA per SM), each walking its items.
    cfg.gridDim = dim3((unsigned)(ctx.num_sms / kPairCtas * kPairCtas), 1, 1);
    int max_clusters = 0;
    const cudaError_t e = clusters_per_device(occupancy, ctx, attn_kernel<kDh>, cfg, &max_clusters);
    if (e != cudaSuccess) return e;
    const int pairs = args.items < max_clusters ? args.items : max_clusters;
    cfg.gridDim = dim3((unsigned)(pairs * kPairCtas), 1, 1);
    return cudaLaunchKernelEx(&cfg, attn_kernel<kDh>, tqk, tv, args);
}

}  // namespace

cudaError_t launch_attention(const LaunchCtx& ctx, const CUtensorMap& tmap_qk, const CUtensorMap& tmap_vt,
                             uint16_t* o, int64_t B, int64_t S, int64_t D, int64_t H, float scale, int withhold,
                             int64_t wait_limit_ns) {
    const int64_t dh = D / H;
    const int64_t nqb = (S + kRowsCta * kPairCtas - 1) / (kRowsCta * kPairCtas);
    const int64_t items = B * H * nqb;
    if (items <= 0 || items > 0x7FFFFFFF) return cudaErrorInvalidValue;
    AttnArgs a{o, (int)S, (int)D, (int)H, (int)nqb, (int)items, scale * 1.4426950408889634f, ctx.status,
               wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : kAttnWaitNs, withhold};
    if (dh == 128) return run_attn<128>(ctx, tmap_qk, tmap_vt, a);
    if (dh == 64) return run_attn<64>(ctx, tmap_qk, tmap_vt, a);
    return cudaErrorInvalidValue;
}

}  // namespace nvfp4rl
