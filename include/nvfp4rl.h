/*
 * nvfp4rl — C ABI of the NVFP4 FP4-explore hot path (GB300, sm_103a).
 *
 * Five calls implement the data path of Sol-RL's "FP4 Explore, BF16 Train"
 * iteration:
 *   nvfp4_requant       LoRA-merge the DiT weights and re-quantize them to NVFP4
 *                       after a policy update (Sol-RL project page, "Two-Stage
 *                       Pipeline", Stage 2: "re-quantize weights to NVFP4 for the
 *                       next iteration"; AI Trends summary, paragraph on training
 *                       stability: LoRA rank 32, re-quantized in real time with
 *                       no compile step).
 *   nvfp4_act_quant     quantize BF16 activations to NVFP4, one scale per token,
 *                       for the NVFP4-quantized solver (Sol-RL project page,
 *                       "Two-Stage Pipeline", Stage 1); nvfp4_act_quant_tensor is
 *                       the variant with one scale for the whole tensor.
 *   nvfp4_gemm          the block-scaled FP4 linear layer of that solver (same
 *                       section: "up to 4x TFLOPs vs. BF16").
 *   bf16_gemm           the BF16 linear layer of Stage 2 (regeneration of the
 *                       selected seeds), used for the FP4 / BF16 ratio.
 *   select_contrastive  keep the top K/2 and bottom K/2 seeds of N proxy rewards
 *                       per prompt (Sol-RL project page, "Two-Stage Pipeline",
 *                       Stage 1; AI Trends summary, paragraph on the pipeline)
 *                       and apply the DiffusionNFT reward transform ("DiffusionNFT",
 *                       VeRL-Omni documentation, "Algorithm").
 *
 * NVFP4 convention.  The pages name NVFP4 without defining its encoding; this
 * library uses the two-level scheme
 *     s    = amax / (6 * 448)                      fp32; per tensor for weights,
 *                                                  per row ("per token") for
 *                                                  activations
 *     sf   = RNE_E4M3_sat(block_amax / (6 * s))    one E4M3 scale per 16
 *                                                  consecutive K-elements
 *     code = RNE_E2M1_sat(x / (sf * s))            E2M1, sign kept, saturating
 * with every scale operation an IEEE fp32 operation (round to nearest even):
 * d = 6*s; v = block_amax / d (a true division); den = sf*s; q = x / den.  A
 * zero s gives sf = 0 everywhere; a block whose den is 0 emits code 0x0.
 *
 * Data layouts (all row-major, K innermost).
 *   codes  [rows, K/2] bytes: byte k/2 holds the code of element k (even) in
 *          bits 0..3 and of element k+1 in bits 4..7.  E2M1 code: bit 3 sign,
 *          bits 2..1 exponent (bias 1), bit 0 mantissa.
 *   sf     nvfp4_sf_bytes(rows, K) bytes in the 128x4 blocked layout that the
 *          tensor cores read: tile (R, C) covers rows 128R..128R+127 and 16-element
 *          K-blocks 4C..4C+3 and is 512 contiguous bytes; tiles are stored
 *          R-major (tile index R * K/64 + C); inside a tile the byte of (row, kblk)
 *          is at (row % 32) * 16 + ((row / 32) % 4) * 4 + kblk % 4.  Rows from
 *          `rows` up to the next multiple of 128 are padding and are written as 0.
 *          E4M3 scale byte: sign 0, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 *   s      fp32: one value (weights) or one per row (activations).
 *
 * Conventions shared by every call.
 *   - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *     caller; the library never allocates, frees or retains them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call only enqueues work on it and returns; outputs are
 *     valid once the stream reaches that point.  No call synchronizes.
 *   - Arguments are validated before any CUDA call: NULL required pointers give
 *     NVFP4_ERR_NULL, bad sizes NVFP4_ERR_SHAPE, device pointers not 16-byte
 *     aligned NVFP4_ERR_ALIGN (4-byte for fp32 scalars and vectors).  A current
 *     device that is not compute capability 10.3 gives NVFP4_ERR_ARCH; a failed
 *     CUDA call or launch gives NVFP4_ERR_CUDA.  Nothing is launched on error.
 *   - Device-side failures never trap: every wait inside a kernel is bounded, and
 *     a kernel that gives up records NVFP4_ERR_TIMEOUT in a device status word
 *     read by nvfp4_device_status().
 *   - No C++ exception crosses this interface.
 *   - Sizes: 1 <= K, K % 64 == 0 for the NVFP4 calls; rows (M, N) may be 0 (the
 *     call is then a no-op) and need not be multiples of anything except where
 *     stated.
 */
#ifndef NVFP4RL_H
#define NVFP4RL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_NULL = 1,
    NVFP4_ERR_SHAPE = 2,
    NVFP4_ERR_ALIGN = 3,
    NVFP4_ERR_ARCH = 4,
    NVFP4_ERR_CUDA = 5,
    NVFP4_ERR_TIMEOUT = 6
} nvfp4_status;

enum { NVFP4_W_BF16 = 0, NVFP4_W_FP32 = 1 };

/* Size in bytes of a scale-factor buffer for a [rows, K] NVFP4 tensor. */
static inline size_t nvfp4_sf_bytes(int64_t rows, int64_t K) {
    return (size_t)((rows + 127) / 128) * 128u * (size_t)(K / 16);
}

/* Byte offset of the scale of (row, kblk) in that buffer (kblk = k / 16). */
static inline size_t nvfp4_sf_offset(int64_t row, int64_t kblk, int64_t K) {
    return (size_t)(((row / 128) * (K / 64) + kblk / 4) * 512 + (row % 32) * 16 +
                    ((row / 32) % 4) * 4 + kblk % 4);
}

/*
 * nvfp4_requant — W' = W + (alpha / r) * B * A, then per-tensor NVFP4.
 *   W      device, [N, K], bf16 (w_dtype NVFP4_W_BF16) or fp32 (NVFP4_W_FP32).
 *   A      device, [r, K] fp32, or NULL;  B  device, [N, r] fp32, or NULL.
 *          r == 0 or A == NULL or B == NULL quantizes W without a merge.
 *          0 <= r <= 64.  The merge is, per element, acc = +0 followed by
 *          acc = fma(B[n,j], A[j,k], acc) for j = 0..r-1 in order, then
 *          w' = fma(alpha / r, acc, W[n,k]) (fp32, alpha / r rounded once).
 *   codes  device, [N, K/2] bytes (out).
 *   sf     device, nvfp4_sf_bytes(N, K) bytes (out, padding rows written 0).
 *   s_t    device, one fp32 (out): amax(|W'|) / 2688.  Also used as the amax
 *          accumulator while the call runs, so it must not alias other buffers.
 *   workspace, workspace_bytes
 *          device scratch owned by the caller, or NULL / 0.  With bf16 W, r == 32
 *          and a 16-byte aligned B, a 256-byte aligned workspace of at least
 *          nvfp4_requant_workspace_bytes(...) bytes selects the tensor-core merge;
 *          otherwise the merge runs on CUDA cores.  Both give identical results.
 *          The workspace must not be used by anything else until the call's
 *          work on `stream` has completed; its contents are not needed afterwards.
 *   K % 64 == 0, K <= 1 << 20, N < 2^31.
 * CUDA-core path: a memset and three kernels: exact amax|W'| (W read once; only the
 * elements whose |W| a Cauchy-Schwarz bound on the LoRA term leaves in reach of the
 * maximum are merged), merge + quantize (every element merged once), and a
 * one-thread finalize of s_t.  Tensor-core path: a kernel that splits A and B into
 * bf16 pairs (into the workspace), then one persistent kernel with the merge as a
 * bf16 GEMM and every decision certified against a rigorous bound or recomputed by
 * the fp32 chain: an amax phase over W, a grid-wide barrier (every CTA resident; a
 * bounded wait), a quantize phase over W again (from L2), and the finalize.  Inputs
 * must be finite.
 */
nvfp4_status nvfp4_requant(const void* W, int w_dtype, const float* A, const float* B, int r,
                           float alpha, int64_t N, int64_t K, uint8_t* codes, uint8_t* sf,
                           float* s_t, void* workspace, size_t workspace_bytes, void* stream);

/*
 * nvfp4_requant_workspace_bytes — bytes of workspace that select nvfp4_requant's
 * tensor-core merge for these arguments, or 0 when that path does not apply
 * (w_dtype other than NVFP4_W_BF16, r != 32, or invalid sizes).  Host only.
 */
size_t nvfp4_requant_workspace_bytes(int w_dtype, int r, int64_t N, int64_t K);

/*
 * nvfp4_act_quant — per-row ("per token") NVFP4 of BF16 activations.
 *   X      device, [M, K] bf16.
 *   codes  device, [M, K/2] bytes (out).
 *   sf     device, nvfp4_sf_bytes(M, K) bytes (out, padding rows written 0).
 *   s_row  device, [M] fp32 (out): amax(|X[m,:]|) / 2688.
 *   K % 64 == 0, K <= 32768, M < 2^31.  X must be finite.  One kernel, one
 *   pass over X.
 */
nvfp4_status nvfp4_act_quant(const void* X, int64_t M, int64_t K, uint8_t* codes, uint8_t* sf,
                             float* s_row, void* stream);

/*
 * nvfp4_act_quant_tensor — NVFP4 of BF16 activations with one scale for the whole
 * tensor instead of one per row (a variant of the per-token reading; the same
 * convention as the weights: s = amax(|X|) / 2688).
 *   X      device, [M, K] bf16, finite.
 *   codes  device, [M, K/2] bytes (out).
 *   sf     device, nvfp4_sf_bytes(M, K) bytes (out, padding rows written 0).
 *   s_t    device, one fp32 (out); also the amax accumulator while the call runs.
 *          Required even when M == 0 (it is then set to 0; X, codes, sf may be NULL).
 *   K % 64 == 0, K <= 32768, M < 2^31.  Two passes over X: a memset, an amax kernel,
 *   nvfp4_act_quant's kernel with the tensor's amax given for every row, and a
 *   one-thread kernel that turns amax into s_t.  Gives the
 *   same codes, scales and s_t as nvfp4_requant with no LoRA factors on X.
 *   To use the result as nvfp4_gemm's activations, pass an [M] fp32 vector holding s_t
 *   in every entry as a_srow (the GEMM reads one scale per row; s_t alone is a single
 *   float and must not be passed there).
 */
nvfp4_status nvfp4_act_quant_tensor(const void* X, int64_t M, int64_t K, uint8_t* codes, uint8_t* sf,
                                    float* s_t, void* stream);

/*
 * nvfp4_act_quant_prescaled — nvfp4_act_quant for activations whose per-row amax is
 * already known, e.g. written by nvfp4_gemm_rowamax when it produced X (the per-token
 * quantization of the NVFP4-quantized solver's next linear, Sol-RL project page,
 * "Two-Stage Pipeline", Stage 1).  With row_amax[m] == max_k |X[m,k]| the codes, scales
 * and s_row are identical to nvfp4_act_quant(X); a row_amax below a row's true amax
 * makes its largest elements saturate (E4M3 scale and E2M1 code clamp).
 *   X         device, [M, K] bf16, finite.
 *   row_amax  device, [M] fp32 (in), each >= 0.
 *   codes     device, [M, K/2] bytes (out).
 *   sf        device, nvfp4_sf_bytes(M, K) bytes (out, padding rows written 0).
 *   s_row     device, [M] fp32 (out): row_amax[m] / 2688.
 *   K % 64 == 0, K <= 32768, M < 2^31.  One kernel: nvfp4_act_quant's, with each row's
 *   scale from row_amax instead of a reduction over the row (X is still read once).
 */
nvfp4_status nvfp4_act_quant_prescaled(const void* X, int64_t M, int64_t K, const float* row_amax,
                                       uint8_t* codes, uint8_t* sf, float* s_row, void* stream);

/*
 * nvfp4_gemm — Y = bf16_RNE( s_a[m] * s_w * sum_k a_hat[m,k] * w_hat[n,k] + bias[n] ),
 * where a_hat = e2m1(code) * e4m3(sf) of the activations and w_hat likewise of
 * the weights; the sum runs on the tensor cores (tcgen05 block-scaled FP4 MMA)
 * with fp32 accumulation.
 *   a_codes, a_sf, a_srow   device, activations as written by nvfp4_act_quant:
 *                           [M, K/2], nvfp4_sf_bytes(M, K), [M] fp32.
 *   w_codes, w_sf, w_st     device, weights as written by nvfp4_requant:
 *                           [N, K/2], nvfp4_sf_bytes(N, K), one fp32.
 *   bias                    device, [N] bf16, or NULL for none.
 *   Y                       device, [M, N] bf16 (out).
 *   K % 64 == 0, N % 8 == 0, M, N < 2^31.
 */
nvfp4_status nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                        const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * nvfp4_gemm_rowamax — nvfp4_gemm that also writes each output row's amax,
 *   y_row_amax[m] = max_n |Y[m,n]| (of the bf16 values, exactly; 0 when N == 0),
 * for the per-token quantization of the next linear (nvfp4_act_quant_prescaled), so
 * that it needs no pass of its own over Y to find the row scales.  The epilogue of
 * every output tile max-reduces its rows into y_row_amax (atomicMax on the fp32 bits;
 * every value is >= 0, so the result is exact and order-free), which the call first
 * zeroes (a memset on `stream`).
 *   y_row_amax  device, [M] fp32 (out), 4-byte aligned.
 *   Other arguments, limits and errors as nvfp4_gemm; Y is bit-identical to its Y.
 */
nvfp4_status nvfp4_gemm_rowamax(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                                const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                                const void* bias, void* Y, float* y_row_amax, int64_t M, int64_t N,
                                int64_t K, void* stream);

/*
 * bf16_gemm — Y = bf16_RNE( X * W^T + bias ), bf16 operands, fp32 accumulation on
 * the tensor cores (tcgen05 kind::f16).
 *   X [M, K] bf16, W [N, K] bf16, bias [N] bf16 or NULL, Y [M, N] bf16 (out); device.
 *   K % 8 == 0, N % 8 == 0, M, N < 2^31.
 */
nvfp4_status bf16_gemm(const void* X, const void* W, const void* bias, void* Y, int64_t M,
                       int64_t N, int64_t K, void* stream);

/*
 * select_contrastive — contrastive filter plus the DiffusionNFT reward transform.
 *   rewards  device, [P, N] fp32 proxy rewards (finite).
 *   idx      device, [P, K] int32 (out): slots 0..K/2-1 hold the seeds of the K/2
 *            largest rewards ordered by (reward descending, seed ascending); slots
 *            K/2..K-1 the seeds of the K/2 smallest, by (reward ascending, seed
 *            ascending).  -0 and +0 compare equal.
 *   r_out    device, [P, K] fp32 (out), or NULL to skip the transform:
 *            r = 1/2 + 1/2 clip((x - mean_p) / Z, -1, 1) where x is the selected
 *            raw reward, mean_p the mean of prompt p's K selected rewards, and Z the
 *            population standard deviation of all P*K selected rewards
 *            (global_std = 1, the default of the page) or of prompt p's K
 *            (global_std = 0); Z == 0 gives r = 1/2.  Accumulated in fp64.
 *   0 < K <= N, K even, N <= 1024, 0 <= P < 2^31.  Two kernels: the ranks (one
 *   CTA per prompt) and, with r_out, the transform (one CTA per prompt, at most
 *   one per SM, started by programmatic dependent launch).
 */
nvfp4_status select_contrastive(const float* rewards, int P, int N, int K, int global_std,
                                int32_t* idx, float* r_out, void* stream);

/*
 * nvfp4_requant_noalloc — nvfp4_requant without a caller workspace.  The Sol-RL
 * pages have no counterpart: this is a library convenience for callers that
 * cannot hand over scratch memory.  Same arguments, results and errors as
 * nvfp4_requant; where the tensor-core merge applies, its workspace is a fixed
 * scratch array that the library reserves in device memory when it is loaded
 * (NVFP4_NOALLOC_SCRATCH_BYTES per device), instead of caller memory.  The call
 * itself allocates and frees nothing.
 *   - Size limit: returns NVFP4_ERR_SHAPE when nvfp4_requant_workspace_bytes(...)
 *     (256 K + 4 N + 16 K / 128 bytes, N rounded up to 256, each piece rounded up
 *     to 256 bytes) exceeds NVFP4_NOALLOC_SCRATCH_BYTES: e.g. K = 16384 fits up to
 *     N = 2^20 rows, K = 32768 up to 15360 rows, K = 65536 never.
 *   - One scratch per device, shared by every call: two calls whose work can
 *     overlap on the device (different streams without ordering between them)
 *     race on it.  Order them (one stream, or events).
 *   - Arguments are checked first, then the device's architecture, exactly as in
 *     nvfp4_requant; only then does the first call on each device look up the
 *     scratch's address (a runtime query, cached afterwards), so make that first
 *     call outside any stream capture.
 */
#define NVFP4_NOALLOC_SCRATCH_BYTES ((size_t)8 * 1024 * 1024 + (size_t)64 * 1024)
nvfp4_status nvfp4_requant_noalloc(const void* W, int w_dtype, const float* A, const float* B,
                                   int r, float alpha, int64_t N, int64_t K, uint8_t* codes,
                                   uint8_t* sf, float* s_t, void* stream);

/* ---------------------------------------------------------------- synthetic DiT block
 *
 * A FLUX-shaped transformer block with NVFP4 linears, standing in for one block of the
 * NVFP4-quantized solver that explores the seeds (Sol-RL project page, "Two-Stage
 * Pipeline", Stage 1; the pages give no block layout, so this is the plain reading):
 * with x [T, D] bf16, T = B*S tokens (B images of S tokens), H heads of dh = D/H,
 *   qkv = lin(x, qkv)                                 [T, 3D]: q | k | v, head h in
 *                                                     columns h*dh .. of each part
 *   o   = attention(qkv): per image and head, P = bf16(softmax(bf16(q k^T) / sqrt(dh)))
 *         over the image's S keys, O = bf16(P v)      [T, D]
 *   h1  = bf16(lin(o, o) + x)
 *   out = bf16(lin(gelu(lin(h1, up)), dn) + h1)       gelu: tanh form, bf16 out
 * where lin(a, w) = nvfp4_gemm(nvfp4_act_quant(a), w) + bias (bf16 out), and w are
 * weights as written by nvfp4_requant: qkv [3D, D], o [D, D], up [4D, D], dn [D, 4D].
 * Every intermediate is bf16, rounded once to nearest-even.  The softmax scale is the
 * fp32 value of 1/sqrt(dh); P is normalised before it is rounded.  The attention runs
 * as one fused tensor-core kernel per call (two passes over the keys: the row maxima
 * and sums, then P and P v), after a per-head transpose of v.
 * Shapes: D % 64 == 0, H divides D with dh = D/H equal to 64 or 128, S % 64 == 0,
 * B*H <= 65535, T < 2^31.
 */
typedef struct {
    const uint8_t* codes; /* [N, K/2] E2M1 codes (nvfp4_requant) */
    const uint8_t* sf;    /* nvfp4_sf_bytes(N, K) bytes, blocked layout */
    const float* s_t;     /* one fp32 */
    const void* bias;     /* [N] bf16, or NULL */
} nvfp4_linear_weights;

/* Bytes of device workspace nvfp4_dit_block needs (host only; 0 for invalid shapes). */
size_t nvfp4_dit_block_workspace_bytes(int64_t B, int64_t S, int64_t D, int64_t H);

/*
 * nvfp4_dit_block — the block above.
 *   x          device, [B*S, D] bf16.
 *   w          host array of 4 nvfp4_linear_weights (device pointers): qkv, o, up, dn.
 *   out        device, [B*S, D] bf16 (out); may not alias x.
 *   workspace  device, >= nvfp4_dit_block_workspace_bytes(...) bytes, 256-byte aligned;
 *              owned by the caller, not used by anything else until the call's work on
 *              `stream` is done.
 * Errors as the calls it makes (NVFP4_ERR_SHAPE for the shape rules above, _NULL,
 * _ALIGN, _ARCH, _CUDA).  Enqueues 10 kernels (the GELU and both residual adds run in
 * the epilogues of the GEMMs that produce their inputs); allocates nothing.
 */
nvfp4_status nvfp4_dit_block(const void* x, int64_t B, int64_t S, int64_t D, int64_t H,
                             const nvfp4_linear_weights* w, void* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* The block's attention alone: qkv [B*S, 3D] bf16 -> o [B*S, D] bf16 (o may not alias
 * qkv), with a device workspace of nvfp4_dit_attention_workspace_bytes(B, S, D, H)
 * bytes (256-byte aligned; it holds v transposed per head), shape rules as the block.
 * Enqueues two kernels; allocates nothing. */
size_t nvfp4_dit_attention_workspace_bytes(int64_t B, int64_t S, int64_t D, int64_t H);
nvfp4_status nvfp4_dit_attention(const void* qkv, int64_t B, int64_t S, int64_t D, int64_t H, void* o,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* The block's streaming steps on bf16 tensors (n % 8 == 0, cols % 8 == 0, 16-byte
 * aligned; results rounded to nearest-even):
 *   bf16_softmax_rows  P = softmax(scale * L) per row of L [rows, cols] (fp32 exp);
 *                      P may alias L.
 *   bf16_gelu          y = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) (fp32); y may
 *                      alias x.
 *   bf16_add           y = a + b (fp32 sum); y may alias a or b. */
nvfp4_status bf16_softmax_rows(const void* L, int64_t rows, int64_t cols, float scale, void* P,
                               void* stream);
nvfp4_status bf16_gelu(const void* x, int64_t n, void* y, void* stream);
nvfp4_status bf16_add(const void* a, const void* b, int64_t n, void* y, void* stream);

/* ---------------------------------------------------------------- diagnostics */

/*
 * nvfp4_requant_exact_counts — how much of the last tensor-core nvfp4_requant that
 * used this workspace went through the exact fp32 chain instead of a certified
 * tensor-core decision (a diagnostic; the Sol-RL pages have no counterpart).
 *   workspace, workspace_bytes, N, K  as passed to that nvfp4_requant call (the
 *            counts live in the workspace; 256-byte aligned, at least
 *            nvfp4_requant_workspace_bytes(NVFP4_W_BF16, 32, N, K) bytes).
 *   counts   host, 2 x uint32 (out): [0] quantize-phase elements merged by the chain
 *            (listed elements, plus 16 per block recomputed whole); [1] amax-phase
 *            candidates merged by the chain.
 * Reads the counts with a device-to-host copy ordered after the work already on
 * `stream`, and waits for it.  Meaningless after a call that took the CUDA-core
 * path or failed.  NVFP4_ERR_NULL / _ALIGN / _SHAPE for bad arguments.
 */
nvfp4_status nvfp4_requant_exact_counts(const void* workspace, size_t workspace_bytes, int64_t N,
                                        int64_t K, uint32_t* counts, void* stream);

/* Human-readable name of a status code (static storage). */
const char* nvfp4_status_string(nvfp4_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int nvfp4_version(void);

/*
 * Reads the device status word of the current device (NVFP4_OK, or
 * NVFP4_ERR_TIMEOUT if some kernel gave up on a bounded wait since the last
 * clear) into *out (host).  clear != 0 resets it afterwards.  Synchronizes the
 * device.  Returns NVFP4_ERR_CUDA if the device cannot be read.
 */
nvfp4_status nvfp4_device_status(int* out, int clear);

/* ---------------------------------------------------------------- test hooks
 * Exported for the test-suite: each runs, over n independent elements, the very
 * device function the quantizers use, so that their rounding can be checked
 * exhaustively.  All buffers are device memory; n >= 0.
 */

/* codes[i] = RNE_E2M1_sat(q[i]) (sign kept), one code per byte. */
nvfp4_status nvfp4_test_e2m1(const float* q, uint8_t* codes, int64_t n, void* stream);

/* codes[i] = RNE_E4M3_sat(v[i]) for v[i] >= 0. */
nvfp4_status nvfp4_test_e4m3(const float* v, uint8_t* codes, int64_t n, void* stream);

/* out[i] = the value of E4M3 code codes[i] (0 <= code <= 0x7E), as the
 * quantizers decode a block scale before dividing by it. */
nvfp4_status nvfp4_test_e4m3_decode(const uint8_t* codes, float* out, int64_t n, void* stream);

/* codes[i] = RNE_E2M1_sat(fl32(x[i] / den[i])) for den[i] > 0, through the
 * quantizers' reciprocal fast path with its exact-division fallback. */
nvfp4_status nvfp4_test_e2m1_quotient(const float* x, const float* den, uint8_t* codes,
                                      int64_t n, void* stream);

/* codes[i] = RNE_E4M3_sat(fl32(v[i] / d[i])) for v[i] >= 0, d[i] > 0, through the
 * quantizers' reciprocal fast path with its exact-division fallback. */
nvfp4_status nvfp4_test_e4m3_quotient(const float* v, const float* d, uint8_t* codes, int64_t n,
                                      void* stream);

/*
 * out[n, k] = W'[n, k] (fp32, device, [N, K]): the merged weights exactly as
 * nvfp4_requant computes them before quantizing (its second kernel, writing the
 * merged values instead of codes).  Arguments and limits as nvfp4_requant;
 * out must be 16-byte aligned.
 */
nvfp4_status nvfp4_test_merge(const void* W, int w_dtype, const float* A, const float* B, int r,
                              float alpha, int64_t N, int64_t K, float* out, void* stream);

/*
 * Launches one CTA that waits on a shared-memory barrier nothing will ever
 * complete, through the same bounded wait the GEMM pipelines use, with a limit
 * of timeout_ns (1e3 .. 1e10).  The kernel must give up, record
 * NVFP4_ERR_TIMEOUT in the device status word and exit; the context stays
 * usable.
 */
nvfp4_status nvfp4_test_wait_timeout(int64_t timeout_ns, void* stream);

/*
 * nvfp4_gemm (no bias) with one K-stage (256 K-elements) of one CTA pair left
 * unloaded on purpose: the pair's even CTA skips the copies of stage withhold_kb
 * (0 <= withhold_kb < K / 256) on its first tile and never announces them, and every
 * wait of the kernel is bounded by timeout_ns (1e6 .. 1e9) instead of the usual 4 s.
 * The pair's MMA issuer, scale writers and epilogue must all give up, record
 * NVFP4_ERR_TIMEOUT, let their own copies and MMAs land, free tensor memory and
 * exit; Y is then incomplete.  Nothing is read or written out of bounds.  Exists to
 * exercise the GEMM's abort path without faulting anything.
 */
nvfp4_status nvfp4_test_gemm_withhold(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                                      const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                                      void* Y, int64_t M, int64_t N, int64_t K, int withhold_kb,
                                      int64_t timeout_ns, void* stream);

/*
 * nvfp4_dit_attention with one K tile (256 keys) of pass 1 left unloaded on purpose:
 * both CTAs of the first CTA pair skip the copies of tile withhold_tile
 * (0 <= withhold_tile < ceil(S / 256)) for their first item and never announce them,
 * and every wait of the kernel is bounded by timeout_ns (1e6 .. 1e9) instead of the
 * usual 4 s.  The pair's MMA issuer, producer and softmax warps must all give up,
 * record NVFP4_ERR_TIMEOUT, let their own copies and MMAs land, free tensor memory and
 * exit; o is then incomplete.  Nothing is read or written out of bounds.  Exists to
 * exercise the attention's abort path without faulting anything.
 */
nvfp4_status nvfp4_test_attention_withhold(const void* qkv, int64_t B, int64_t S, int64_t D, int64_t H, void* o,
                                           void* workspace, size_t workspace_bytes, int withhold_tile,
                                           int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4RL_H */
