/*
 * CPU oracle for the NVFP4 FP4-explore hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * restatement of what the hot path computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  The CUDA library never
 * links, loads or calls it, and the two share no code, header, table or
 * constant generator.  Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math),
 * so every float operation below is one IEEE-754 binary32 operation with
 * round-to-nearest-even, exactly as written.
 *
 * Sources (page title, section):
 *   [SOL]  "Sol-RL: FP4 Explore, BF16 Train" project page, "Two-Stage Pipeline":
 *          Stage 1 samples N = 96 noises, runs an NVFP4-quantized solver and keeps
 *          the top/bottom-K most contrastive seeds; Stage 2 regenerates K = 24 seeds
 *          in BF16, updates the policy, then re-quantizes the weights to NVFP4.
 *   [AIT]  AI Trends summary "FP4 탐색, BF16 학습: 효율적인 롤아웃 스케일링을 통한
 *          확산 강화 학습", paragraph on the pipeline (weights quantized to NVFP4,
 *          top K/2 and bottom K/2 seeds) and paragraph on training stability
 *          (LoRA rank 32; updated weights re-quantized in real time).
 *   [NFT]  "DiffusionNFT" (VeRL-Omni documentation), "Algorithm": the reward
 *          transform r = 1/2 + 1/2 clip((r_raw - E[r_raw]) / Z, -1, 1), Z a standard
 *          deviation taken over the prompt's group or the global batch, global by
 *          default.
 *   [MX]   OCP Microscaling Formats specification, FP4 E2M1 element type.
 *   [FP8]  OCP 8-bit floating point specification, E4M3 (bias 7, max 448,
 *          S.1111.111 is NaN, no infinities).
 *
 * The pages name NVFP4 but do not define its encoding.  The convention used here:
 *   s   = amax / (6 * 448)                   fp32 (per tensor for weights, per row
 *                                            for activations)
 *   sf  = RNE_E4M3_sat(block_amax / (6 s))   one per 16 consecutive K-elements
 *   q   = RNE_E2M1_sat(x / (sf s))           sign kept, saturating at 6
 *
 * Readings where the pages are silent (the numbers skip readings that concern only
 * the CUDA library or the synthetic inputs):
 *   R1  Scale arithmetic is IEEE fp32: d = 6*s, v = bamax / d (a division, not a
 *       reciprocal multiply), den = sff * s formed first, then q = x / den.
 *   R2  Merge: c = alpha / r (fp32); acc = fmaf chain over j = 0..r-1 of
 *       B[n,j]*A[j,k] starting from +0; w' = fmaf(c, acc, W[n,k]).
 *   R3  s = 0 gives sf = 0 for every block; a block whose den = sff*s is 0 emits
 *       code 0x0 for all its elements.
 *   R7  Code nibbles: byte k/2 holds code(k even) in bits 0..3, code(k odd) in
 *       bits 4..7.  Scales are emitted row-major [rows, K/16] here.
 *   R9  Selection: top K/2 by (value desc, index asc), then bottom K/2 by
 *       (value asc, index asc); -0 == +0.
 *   R10 Transform: mean over the K selected rewards of the prompt; Z is the
 *       population standard deviation of all P*K selected rewards (global) or of
 *       the prompt's K (per prompt); Z == 0 gives r = 1/2.  Accumulation in fp64,
 *       r rounded to fp32 once.
 *   R15 The synthetic DiT block ([SOL] Stage 1 runs the NVFP4-quantized solver
 *       over the DiT's linears; the block below is a FLUX-shaped stand-in):
 *       tensors between the steps are bf16, each rounded once to nearest-even
 *       from the exact value of its step: the NVFP4 and BF16 products (exact
 *       sums), the attention logits, the softmax probabilities, the GELU
 *       (tanh form) and the residual sums.  The softmax scale is the fp32 value of
 *       1/sqrt(dh), applied to the bf16 logits.  See orc_bf16_rne and the block
 *       functions at the end.
 *   R16 The GELU's tanh form is evaluated through the exact identity
 *       (1 + tanh t)/2 = 1/(1 + e^(-2t)), the exponential of a non-positive
 *       argument (the direct form cancels below x = -7).
 *
 * Every function is pinned by tests/test_oracle_*.py against closed forms,
 * brute force or a library routine; none is "parity unpinned".
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SHAPE 2

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ formats */

/* [MX] E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: 0.m x 2^(1-1). */
double orc_e2m1_decode(int code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* [FP8] E4M3: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * Exponent field 0 is subnormal: 0.mmm x 2^(1-7).  S.1111.111 is NaN. */
double orc_e4m3_decode(int code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, 1 - 7) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Non-negative codes of each format in increasing value order (code order is
 * value order for both formats), filled from the decoders above. */
static double g_e2m1_pos[8];
static double g_e4m3_pos[127]; /* 0x00..0x7E; 0x7F is NaN */
static int g_tables_ready = 0;

static void ensure_tables(void) {
    if (g_tables_ready) return;
#ifdef _OPENMP
#pragma omp critical(orc_tables)
#endif
    {
        if (!g_tables_ready) {
            for (int c = 0; c < 8; ++c) g_e2m1_pos[c] = orc_e2m1_decode(c);
            for (int c = 0; c < 127; ++c) g_e4m3_pos[c] = orc_e4m3_decode(c);
            g_tables_ready = 1;
        }
    }
}

/* Round mag >= 0 to the nearest of vals[0..n-1] (increasing), ties to the code
 * with an even mantissa (code bit 0 == 0); anything above vals[n-1] saturates
 * to n-1.  For the two neighbours that decide, mag - vals[c] is exact in double
 * (mag has 24 significant bits and sits within a few binades of vals[c]); when
 * mag is far below vals[1] the winner is code 0 regardless. */
static int round_nearest_even(double mag, const double* vals, int n) {
    if (!(mag > vals[0])) return 0;
    if (mag >= vals[n - 1]) return n - 1;
    int lo = 0, hi = n - 1; /* vals[lo] <= mag < vals[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (vals[mid] <= mag) lo = mid; else hi = mid;
    }
    double dlo = mag - vals[lo];
    double dhi = vals[hi] - mag;
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return (lo & 1) == 0 ? lo : hi;
}

/* RNE to E2M1 with the sign bit copied from q, saturating at 6. */
int orc_e2m1_rne_sat(float q) {
    ensure_tables();
    int mag = round_nearest_even(fabs((double)q), g_e2m1_pos, 8);
    return mag | (signbit(q) ? 8 : 0);
}

/* RNE to E4M3 for v >= 0, saturating at 448 (code 0x7E). */
int orc_e4m3_rne_sat(float v) {
    ensure_tables();
    return round_nearest_even((double)v, g_e4m3_pos, 127);
}

void orc_e2m1_rne_sat_array(const float* q, int64_t n, uint8_t* out) {
    ensure_tables();
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_rne_sat(q[i]);
}

void orc_e4m3_rne_sat_array(const float* v, int64_t n, uint8_t* out) {
    ensure_tables();
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_rne_sat(v[i]);
}

/* ------------------------------------------------------------------ merge */

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* LoRA merge W' = W + (alpha / r) * B * A with rank r ([AIT]: r = 32), reading
 * R2.  W is [N,K] bf16 (w_dtype 0) or fp32 (w_dtype 1); A is [r,K]; B is [N,r].
 * r == 0 or a NULL factor means no merge: W' = W.  out is [N,K] fp32. */
void orc_merge(const void* W, int w_dtype, const float* A, const float* B, int r,
               float alpha, int64_t N, int64_t K, float* out) {
    const int merge = (r > 0 && A != NULL && B != NULL);
    const float c = merge ? alpha / (float)r : 0.0f;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            float w = (w_dtype == 0) ? bf16_bits_to_float(((const uint16_t*)W)[n * K + k])
                                     : ((const float*)W)[n * K + k];
            if (!merge) { out[n * K + k] = w; continue; }
            float acc = 0.0f;
            for (int j = 0; j < r; ++j) acc = fmaf(B[n * r + j], A[(int64_t)j * K + k], acc);
            out[n * K + k] = fmaf(c, acc, w);
        }
    }
}

/* ------------------------------------------------------------------ quantize */

/* Quantize rows [r0, r1) of x [rows,K] with second-level scale s, readings R1/R3/R7. */
static void quantize_rows(const float* x, int64_t r0, int64_t r1, int64_t K, float s,
                          uint8_t* codes, uint8_t* sf) {
    const int64_t nblk = K / 16;
    for (int64_t row = r0; row < r1; ++row) {
        for (int64_t b = 0; b < nblk; ++b) {
            const float* blk = x + row * K + b * 16;
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(blk[i]));
            const float d = 6.0f * s;
            const int sfc = (d == 0.0f) ? 0 : orc_e4m3_rne_sat(bamax / d);
            const float sff = (float)orc_e4m3_decode(sfc);
            const float den = sff * s;
            sf[row * nblk + b] = (uint8_t)sfc;
            for (int i = 0; i < 16; i += 2) {
                int c0 = (den == 0.0f) ? 0 : orc_e2m1_rne_sat(blk[i] / den);
                int c1 = (den == 0.0f) ? 0 : orc_e2m1_rne_sat(blk[i + 1] / den);
                codes[(row * K + b * 16 + i) / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}

/* NVFP4-quantize x [rows,K] (K % 16 == 0).
 *   scope 0: one scale for the whole tensor (weights; s_out[0]),
 *   scope 1: one scale per row (activations, "per token"; s_out[rows]).
 * codes [rows, K/2], sf [rows, K/16] row-major. */
int orc_quantize(const float* x, int64_t rows, int64_t K, int scope, uint8_t* codes,
                 uint8_t* sf, float* s_out) {
    if (K % 16 != 0 || rows < 0) return ORC_ERR_SHAPE;
    ensure_tables();
    if (scope == 0) {
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * K; ++i) amax = fmaxf(amax, fabsf(x[i]));
        const float s = amax / 2688.0f;
        s_out[0] = s;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t row = 0; row < rows; ++row) quantize_rows(x, row, row + 1, K, s, codes, sf);
    } else {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t row = 0; row < rows; ++row) {
            float amax = 0.0f;
            for (int64_t k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(x[row * K + k]));
            const float s = amax / 2688.0f;
            s_out[row] = s;
            quantize_rows(x, row, row + 1, K, s, codes, sf);
        }
    }
    return ORC_OK;
}

/* Dequantize: x_hat = e2m1(code) * e4m3(sf) * s, in double; exact (2 + 4 + 24
 * significant bits).  scope as in orc_quantize.  out [rows, K]. */
void orc_dequantize(const uint8_t* codes, const uint8_t* sf, const float* s, int scope,
                    int64_t rows, int64_t K, double* out) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t row = 0; row < rows; ++row) {
        const double srow = (double)(scope == 0 ? s[0] : s[row]);
        for (int64_t k = 0; k < K; ++k) {
            const uint8_t byte = codes[(row * K + k) / 2];
            const int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
            const double sff = orc_e4m3_decode(sf[row * (K / 16) + k / 16]);
            out[row * K + k] = orc_e2m1_decode(code) * sff * srow;
        }
    }
}

/* ------------------------------------------------------------------ GEMMs */

/* NVFP4 GEMM: y[m,n] = sum_k a_hat[m,k] * w_hat[n,k] + bias[n], in double,
 * sequential in k, for the sampled rows m = rows[i].  a_* hold per-row scales
 * (activations), w_s is the per-tensor weight scale.  Also returns the
 * tolerance denominator S[m,n] = sum_k |a_hat * w_hat|.  y, S are [nrows, N]. */
void orc_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_s,
                    const uint8_t* w_codes, const uint8_t* w_sf, float w_s,
                    const uint16_t* bias, int64_t M, int64_t N, int64_t K,
                    const int64_t* rows, int64_t nrows, double* y, double* S) {
    (void)M;
    double* w_hat = (double*)malloc(sizeof(double) * (size_t)(N * K));
    orc_dequantize(w_codes, w_sf, &w_s, 0, N, K, w_hat);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t m = rows[i];
        double* a_hat = (double*)malloc(sizeof(double) * (size_t)K);
        orc_dequantize(a_codes + m * (K / 2), a_sf + m * (K / 16), a_s + m, 1, 1, K, a_hat);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, sabs = 0.0;
            const double* wr = w_hat + n * K;
            for (int64_t k = 0; k < K; ++k) {
                const double p = a_hat[k] * wr[k];
                acc += p;
                sabs += fabs(p);
            }
            if (bias) acc += (double)bf16_bits_to_float(bias[n]);
            y[i * N + n] = acc;
            S[i * N + n] = sabs;
        }
        free(a_hat);
    }
    free(w_hat);
}

/* Second, independent evaluation of the same sum with integers only:
 *   2 * e2m1(code) is an integer in {0,1,2,3,4,6,8,12} (times the sign) and
 *   2^9 * e4m3(sf) is an integer <= 229376, so
 *   sum_k a_hat * w_hat = a_s * w_s * 2^-20 * T,
 *   T = sum_blocks Ia * Iw * sum_{16} (2 qa)(2 qw)      (exact in int64 for K <= 12288).
 * Returns T[nrows, N] (no bias).  The integer decodings below are written from
 * the bit layouts directly and do not call the double decoders. */
static int64_t e2m1_times2(int code) {
    const int e = (code >> 1) & 3, m = code & 1;
    int64_t v = (e == 0) ? m : ((int64_t)(2 + m) << (e - 1)); /* 2 * 1.m * 2^(e-1) */
    return (code & 8) ? -v : v;
}

static int64_t e4m3_times512(int code) {
    const int e = (code >> 3) & 15, m = code & 7;
    return (e == 0) ? m : ((int64_t)(8 + m) << (e - 1)); /* 2^9 * 1.mmm * 2^(e-7) */
}

void orc_gemm_nvfp4_exact(const uint8_t* a_codes, const uint8_t* a_sf,
                          const uint8_t* w_codes, const uint8_t* w_sf,
                          int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                          int64_t* T) {
    const int64_t nblk = K / 16;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t m = rows[i];
        for (int64_t n = 0; n < N; ++n) {
            int64_t total = 0;
            for (int64_t b = 0; b < nblk; ++b) {
                int64_t inner = 0;
                for (int t = 0; t < 16; ++t) {
                    const int64_t k = b * 16 + t;
                    const uint8_t ab = a_codes[m * (K / 2) + k / 2];
                    const uint8_t wb = w_codes[n * (K / 2) + k / 2];
                    const int ac = (k % 2 == 0) ? (ab & 15) : (ab >> 4);
                    const int wc = (k % 2 == 0) ? (wb & 15) : (wb >> 4);
                    inner += e2m1_times2(ac) * e2m1_times2(wc);
                }
                total += e4m3_times512(a_sf[m * nblk + b]) * e4m3_times512(w_sf[n * nblk + b]) * inner;
            }
            T[i * N + n] = total;
        }
    }
}

/* BF16 GEMM: y[m,n] = sum_k x[m,k] * w[n,k] + bias[n] in double (bf16 products
 * are exact in double), sequential in k, for the sampled rows; S as above. */
void orc_gemm_bf16(const uint16_t* x, const uint16_t* w, const uint16_t* bias, int64_t M,
                   int64_t N, int64_t K, const int64_t* rows, int64_t nrows, double* y,
                   double* S) {
    (void)M;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t m = rows[i];
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = (double)bf16_bits_to_float(x[m * K + k]) *
                                 (double)bf16_bits_to_float(w[n * K + k]);
                acc += p;
                sabs += fabs(p);
            }
            if (bias) acc += (double)bf16_bits_to_float(bias[n]);
            y[i * N + n] = acc;
            S[i * N + n] = sabs;
        }
    }
}

/* ------------------------------------------------------------------ selection */

typedef struct {
    float v;
    int i;
} orc_pair;

static int by_value_desc(const void* pa, const void* pb) {
    const orc_pair* a = (const orc_pair*)pa;
    const orc_pair* b = (const orc_pair*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

static int by_value_asc(const void* pa, const void* pb) {
    const orc_pair* a = (const orc_pair*)pa;
    const orc_pair* b = (const orc_pair*)pb;
    if (a->v < b->v) return -1;
    if (a->v > b->v) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

/* Contrastive filter ([SOL] Stage 1, [AIT] top K/2 and bottom K/2) and the
 * reward transform ([NFT] "Algorithm"), readings R9/R10.
 * rewards [P,N]; idx [P,K]: slots 0..K/2-1 the top seeds in descending order,
 * slots K/2..K-1 the bottom seeds in ascending order; r_out [P,K] or NULL. */
int orc_select_contrastive(const float* rewards, int P, int N, int K, int global_std,
                           int32_t* idx, float* r_out) {
    if (P < 0 || N <= 0 || K <= 0 || (K % 2) != 0 || K > N) return ORC_ERR_SHAPE;
    const int half = K / 2;
    orc_pair* pairs = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)N);
    for (int p = 0; p < P; ++p) {
        for (int j = 0; j < N; ++j) { pairs[j].v = rewards[(int64_t)p * N + j]; pairs[j].i = j; }
        qsort(pairs, (size_t)N, sizeof(orc_pair), by_value_desc);
        for (int t = 0; t < half; ++t) idx[(int64_t)p * K + t] = pairs[t].i;
        qsort(pairs, (size_t)N, sizeof(orc_pair), by_value_asc);
        for (int t = 0; t < half; ++t) idx[(int64_t)p * K + half + t] = pairs[t].i;
    }
    free(pairs);
    if (r_out == NULL || P == 0) return ORC_OK;

    /* selected raw rewards x[p,t] in slot order */
    double* x = (double*)malloc(sizeof(double) * (size_t)P * K);
    double* mu = (double*)malloc(sizeof(double) * (size_t)P);
    double* z = (double*)malloc(sizeof(double) * (size_t)P);
    for (int p = 0; p < P; ++p)
        for (int t = 0; t < K; ++t)
            x[(int64_t)p * K + t] = (double)rewards[(int64_t)p * N + idx[(int64_t)p * K + t]];
    for (int p = 0; p < P; ++p) {
        double sum = 0.0;
        for (int t = 0; t < K; ++t) sum += x[(int64_t)p * K + t];
        mu[p] = sum / K;
    }
    if (global_std) {
        double sum = 0.0;
        for (int64_t i = 0; i < (int64_t)P * K; ++i) sum += x[i];
        const double mean = sum / ((double)P * K);
        double ss = 0.0;
        for (int64_t i = 0; i < (int64_t)P * K; ++i) ss += (x[i] - mean) * (x[i] - mean);
        const double zg = sqrt(ss / ((double)P * K));
        for (int p = 0; p < P; ++p) z[p] = zg;
    } else {
        for (int p = 0; p < P; ++p) {
            double ss = 0.0;
            for (int t = 0; t < K; ++t) {
                const double dv = x[(int64_t)p * K + t] - mu[p];
                ss += dv * dv;
            }
            z[p] = sqrt(ss / K);
        }
    }
    for (int p = 0; p < P; ++p) {
        for (int t = 0; t < K; ++t) {
            double r = 0.5;
            if (z[p] > 0.0) {
                double u = (x[(int64_t)p * K + t] - mu[p]) / z[p];
                if (u < -1.0) u = -1.0;
                if (u > 1.0) u = 1.0;
                r = 0.5 + 0.5 * u;
            }
            r_out[(int64_t)p * K + t] = (float)r;
        }
    }
    free(x);
    free(mu);
    free(z);
    return ORC_OK;
}

/* ------------------------------------------------------------------ DiT block (R15) */

/* Nearest bf16 to x, ties to even: 8 significant bits over the fp32 exponent
 * range (below 2^-126 a fixed quantum of 2^-133, the bf16 subnormals); values
 * that round above the largest finite bf16, (2 - 2^-7) 2^127, give infinity.
 * Returns the bf16 bit pattern.  The rounding is one operation on the exact
 * double: x / quantum is exact (a power of two), nearbyint rounds it to an
 * integer with ties to even (the default rounding mode). */
uint16_t orc_bf16_rne(double x) {
    if (x != x) return 0x7FC0;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    (void)frexp(a, &e); /* a = f 2^e, f in [0.5, 1): the leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < -126) lead = -126;
    const double quantum = ldexp(1.0, lead - 7);
    const double v = nearbyint(a / quantum) * quantum;
    if (v > 3.3895313892515355e38) return sign | 0x7F80;
    const float f = (float)v; /* exact: at most 8 significant bits in range */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)(u >> 16);
}

void orc_bf16_rne_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(x[i]);
}

/* Attention probabilities: per row of bf16 logits L [rows, cols],
 * P = bf16(softmax(scale * L)), the softmax exact in double (the maximum
 * subtracted first, which leaves it unchanged). */
void orc_softmax_bf16(const uint16_t* L, int64_t rows, int64_t cols, double scale, uint16_t* P) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < rows; ++i) {
        const uint16_t* l = L + i * cols;
        double m = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) m = fmax(m, (double)bf16_bits_to_float(l[j]));
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j) sum += exp(scale * ((double)bf16_bits_to_float(l[j]) - m));
        for (int64_t j = 0; j < cols; ++j)
            P[i * cols + j] = orc_bf16_rne(exp(scale * ((double)bf16_bits_to_float(l[j]) - m)) / sum);
    }
}

/* GELU in its tanh form, g(x) = x/2 (1 + tanh(t)), t = sqrt(2/pi) (x + 0.044715 x^3),
 * in double; and its bf16 version on bf16 inputs.  It is evaluated through the exact
 * identity (1 + tanh(t)) / 2 = 1 / (1 + e^(-2t)), with the exponential taken of a
 * non-positive argument: 1 + tanh(t) itself cancels for t << 0 (x below about -5),
 * where g is small but not zero. */
static double gelu_f64_one(double v) {
    const double k = sqrt(2.0 / (4.0 * atan(1.0)));
    const double t2 = 2.0 * k * (v + 0.044715 * v * v * v);
    const double sig = t2 >= 0.0 ? 1.0 / (1.0 + exp(-t2)) : exp(t2) / (1.0 + exp(t2));
    return v * sig;
}

void orc_gelu_f64(const double* x, int64_t n, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = gelu_f64_one(x[i]);
}

void orc_gelu_bf16(const uint16_t* x, int64_t n, uint16_t* y) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) y[i] = orc_bf16_rne(gelu_f64_one((double)bf16_bits_to_float(x[i])));
}

/* Residual sum of two bf16 tensors, bf16(a + b) (the sum is exact in double). */
void orc_add_bf16(const uint16_t* a, const uint16_t* b, int64_t n, uint16_t* y) {
    for (int64_t i = 0; i < n; ++i)
        y[i] = orc_bf16_rne((double)bf16_bits_to_float(a[i]) + (double)bf16_bits_to_float(b[i]));
}
