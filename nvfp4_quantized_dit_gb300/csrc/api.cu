// extern "C" entry points of libnvfp4rl (declared and documented in nvfp4rl.h).
//
// Every call validates its arguments before touching CUDA, resolves the current
// device (cached: compute capability, SM count, the address of the device status
// word), encodes TMA tensor maps where a GEMM needs them, and enqueues kernels on
// the caller's stream.  No call allocates, frees or synchronizes (except
// nvfp4_device_status, documented as synchronizing).
#include <cudaTypedefs.h>

#include <mutex>

#include "block.cuh"
#include "common.cuh"

namespace nvfp4rl {

// Device status word: 0, or the first failure a kernel recorded (NVFP4_ERR_TIMEOUT).
__device__ int g_status_word = 0;

// Scratch of nvfp4_requant_noalloc (reserved with the module; one per device).
__device__ __align__(256) uint8_t g_noalloc_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

namespace {

struct DeviceInfo {
    bool checked = false;
    bool arch_ok = false;
    int num_sms = 0;
    int* status = nullptr;
};

DeviceInfo g_devices[kMaxDevices];
void* g_noalloc_addr[kMaxDevices];  // address of g_noalloc_scratch per device, once looked up
std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

nvfp4_status resolve(void* stream, LaunchCtx* ctx) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return NVFP4_ERR_CUDA;
        }
        d.arch_ok = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.arch_ok) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
                cudaGetLastError();
                return NVFP4_ERR_CUDA;
            }
            d.status = static_cast<int*>(p);
        }
        d.checked = true;
    }
    if (!d.arch_ok) return NVFP4_ERR_ARCH;
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->status = d.status;
    ctx->num_sms = d.num_sms;
    ctx->device = dev;
    cudaGetLastError();  // start from a clean error state
    return NVFP4_OK;
}

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

bool encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            cudaGetLastError();
            return false;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return true;
}

// 2-D row-major tensor [rows, inner] with a (box_inner x box_rows) box.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if (!encoder(&enc)) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The bf16 output Y [M, N] as 32 x 32 store boxes with the 64-byte swizzle.
bool encode_out(CUtensorMap* map, void* Y, int64_t M, int64_t N) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, (uint64_t)N, (uint64_t)M,
                     (uint64_t)N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Scale-factor buffer of a [rows, K] NVFP4 tensor viewed as 4-D bytes
// {256, 2, K/64, ceil(rows/128)}: one 512-byte tile per (K-chunk of 64, 128-row
// tile), loaded four K-chunks (2 KB) at a time; tiles or chunks past the end arrive
// as zeros.
bool encode_sf(CUtensorMap* map, const void* base, int64_t rows, int64_t K) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if (!encoder(&enc)) return false;
    const cuuint64_t dims[4] = {256, 2, (cuuint64_t)(K / 64), (cuuint64_t)((rows + 127) / 128)};
    const cuuint64_t strides[3] = {256, 512, (cuuint64_t)(K / 64) * 512};
    const cuuint32_t box[4] = {256, 2, 4, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

}  // namespace
}  // namespace nvfp4rl

namespace nvfp4rl {
// Defined in quant.cu (the per-tensor activation variant).
cudaError_t launch_act_quant_tensor(const LaunchCtx& ctx, const __nv_bfloat16* X, int64_t M, int64_t K,
                                    uint8_t* codes, uint8_t* sf, float* s_t);
}  // namespace nvfp4rl

using namespace nvfp4rl;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_NULL: return "NVFP4_ERR_NULL";
        case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE";
        case NVFP4_ERR_ALIGN: return "NVFP4_ERR_ALIGN";
        case NVFP4_ERR_ARCH: return "NVFP4_ERR_ARCH";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    }
    return "NVFP4_ERR_UNKNOWN";
}

int nvfp4_version(void) { return 100; }

nvfp4_status nvfp4_requant_exact_counts(const void* workspace, size_t workspace_bytes, int64_t N,
                                        int64_t K, uint32_t* counts, void* stream) {
    if (workspace == nullptr || counts == nullptr) return NVFP4_ERR_NULL;
    if (misaligned(workspace, 256)) return NVFP4_ERR_ALIGN;
    if (N <= 0 || N > kMaxRows || K <= 0 || K % 64 != 0 || K > (1 << 20)) return NVFP4_ERR_SHAPE;
    const size_t need = requant_tc_workspace_bytes(NVFP4_W_BF16, 32, N, K);
    if (need == 0 || workspace_bytes < need) return NVFP4_ERR_SHAPE;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    const RequantTcLayout ws = requant_tc_layout(const_cast<void*>(workspace), N, K);
    cudaError_t e = cudaMemcpyAsync(counts, ws.counter + 3, 2 * sizeof(uint32_t), cudaMemcpyDeviceToHost, ctx.stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx.stream);
    return from_cuda(e);
}

size_t nvfp4_requant_workspace_bytes(int w_dtype, int r, int64_t N, int64_t K) {
    if (N < 0 || N > kMaxRows || K <= 0 || K % 64 != 0 || K > (1 << 20)) return 0;
    return requant_tc_workspace_bytes(w_dtype, r, N, K);
}

// nvfp4_requant's argument checks (no CUDA call); both requant entry points run them
// before resolving the device.
static nvfp4_status check_requant(const void* W, int w_dtype, const float* A, const float* B, int r,
                                  int64_t N, int64_t K, const uint8_t* codes, const uint8_t* sf,
                                  const float* s_t) {
    if (w_dtype != NVFP4_W_BF16 && w_dtype != NVFP4_W_FP32) return NVFP4_ERR_SHAPE;
    if (r < 0 || r > 64 || N < 0 || N > kMaxRows || K <= 0 || K % 64 != 0 || K > (1 << 20))
        return NVFP4_ERR_SHAPE;
    if (s_t == nullptr) return NVFP4_ERR_NULL;
    if (misaligned(s_t, 4)) return NVFP4_ERR_ALIGN;
    const bool merge = r > 0 && A != nullptr && B != nullptr;
    if (N > 0) {
        if (W == nullptr || codes == nullptr || sf == nullptr) return NVFP4_ERR_NULL;
        if (misaligned(W, 16) || misaligned(codes, 16) || misaligned(sf, 16)) return NVFP4_ERR_ALIGN;
        if (merge && (misaligned(A, 16) || misaligned(B, 4))) return NVFP4_ERR_ALIGN;
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_requant(const void* W, int w_dtype, const float* A, const float* B, int r,
                           float alpha, int64_t N, int64_t K, uint8_t* codes, uint8_t* sf,
                           float* s_t, void* workspace, size_t workspace_bytes, void* stream) {
    nvfp4_status st = check_requant(W, w_dtype, A, B, r, N, K, codes, sf, s_t);
    if (st != NVFP4_OK) return st;
    const bool merge = r > 0 && A != nullptr && B != nullptr;
    LaunchCtx ctx;
    st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    if (N == 0) return from_cuda(cudaMemsetAsync(s_t, 0, sizeof(float), ctx.stream));
    const float c = merge ? alpha / static_cast<float>(r) : 0.0f;
    const size_t need = merge ? requant_tc_workspace_bytes(w_dtype, r, N, K) : 0;
    if (need > 0 && workspace != nullptr && workspace_bytes >= need && !misaligned(workspace, 256) &&
        !misaligned(B, 16)) {
        const RequantTcLayout ws = requant_tc_layout(workspace, N, K);
        RequantTcMaps m;
        if (!encode_2d(&m.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)K, (uint64_t)N,
                       (uint64_t)K * 2, 64, 128) ||
            !encode_2d(&m.ap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws.ap, 128, (uint64_t)K, 256, 64, 64))
            return NVFP4_ERR_CUDA;
        return from_cuda(launch_requant_tc(ctx, m, W, A, B, workspace, c, N, K, codes, sf, s_t));
    }
    return from_cuda(launch_requant(ctx, W, w_dtype, merge ? A : nullptr, merge ? B : nullptr,
                                    merge ? r : 0, c, N, K, codes, sf, s_t));
}

nvfp4_status nvfp4_requant_noalloc(const void* W, int w_dtype, const float* A, const float* B,
                                   int r, float alpha, int64_t N, int64_t K, uint8_t* codes,
                                   uint8_t* sf, float* s_t, void* stream) {
    // The same checks, in the same order, as nvfp4_requant (arguments, then the device's
    // architecture) before the scratch's address is looked up.
    nvfp4_status st = check_requant(W, w_dtype, A, B, r, N, K, codes, sf, s_t);
    if (st != NVFP4_OK) return st;
    const bool merge = r > 0 && A != nullptr && B != nullptr;
    const size_t need = merge ? nvfp4_requant_workspace_bytes(w_dtype, r, N, K) : 0;
    if (need > NVFP4_NOALLOC_SCRATCH_BYTES) return NVFP4_ERR_SHAPE;
    LaunchCtx ctx;
    st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    void* scratch = nullptr;
    if (need > 0 && N > 0) {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_noalloc_addr[ctx.device] == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return NVFP4_ERR_CUDA;
            }
            g_noalloc_addr[ctx.device] = p;
        }
        scratch = g_noalloc_addr[ctx.device];
    }
    return nvfp4_requant(W, w_dtype, A, B, r, alpha, N, K, codes, sf, s_t, scratch,
                         scratch != nullptr ? NVFP4_NOALLOC_SCRATCH_BYTES : 0, stream);
}

nvfp4_status nvfp4_act_quant(const void* X, int64_t M, int64_t K, uint8_t* codes, uint8_t* sf,
                             float* s_row, void* stream) {
    if (M < 0 || M > kMaxRows || K <= 0 || K % 64 != 0 || K > 32768) return NVFP4_ERR_SHAPE;
    if (M == 0) return NVFP4_OK;
    if (X == nullptr || codes == nullptr || sf == nullptr || s_row == nullptr) return NVFP4_ERR_NULL;
    if (misaligned(X, 16) || misaligned(codes, 16) || misaligned(sf, 16) || misaligned(s_row, 4))
        return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_act_quant(ctx, static_cast<const __nv_bfloat16*>(X), M, K, codes, sf,
                                      s_row));
}

nvfp4_status nvfp4_act_quant_prescaled(const void* X, int64_t M, int64_t K, const float* row_amax,
                                       uint8_t* codes, uint8_t* sf, float* s_row, void* stream) {
    if (M < 0 || M > kMaxRows || K <= 0 || K % 64 != 0 || K > 32768) return NVFP4_ERR_SHAPE;
    if (M == 0) return NVFP4_OK;
    if (!X || !row_amax || !codes || !sf || !s_row) return NVFP4_ERR_NULL;
    if (misaligned(X, 16) || misaligned(codes, 16) || misaligned(sf, 16) || misaligned(row_amax, 4) ||
        misaligned(s_row, 4))
        return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_act_quant_prescaled(ctx, static_cast<const __nv_bfloat16*>(X), M, K, row_amax,
                                                codes, sf, s_row));
}

nvfp4_status nvfp4_act_quant_tensor(const void* X, int64_t M, int64_t K, uint8_t* codes, uint8_t* sf,
                                    float* s_t, void* stream) {
    if (M < 0 || M > kMaxRows || K <= 0 || K % 64 != 0 || K > 32768) return NVFP4_ERR_SHAPE;
    if (s_t == nullptr) return NVFP4_ERR_NULL;  // written even for an empty tensor (s_t = 0)
    if (misaligned(s_t, 4)) return NVFP4_ERR_ALIGN;
    if (M > 0) {
        if (X == nullptr || codes == nullptr || sf == nullptr) return NVFP4_ERR_NULL;
        if (misaligned(X, 16) || misaligned(codes, 16) || misaligned(sf, 16)) return NVFP4_ERR_ALIGN;
    }
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    if (M == 0) return from_cuda(cudaMemsetAsync(s_t, 0, sizeof(float), ctx.stream));
    return from_cuda(
        launch_act_quant_tensor(ctx, static_cast<const __nv_bfloat16*>(X), M, K, codes, sf, s_t));
}

static nvfp4_status gemm_nvfp4_call(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                                    const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                                    const void* bias, void* Y, int64_t M, int64_t N, int64_t K,
                                    void* stream, int withhold_kb, int64_t wait_limit_ns,
                                    float* row_amax = nullptr, bool want_amax = false, int epi = 0,
                                    const uint16_t* residual = nullptr) {
    if (M < 0 || N < 0 || M > kMaxRows || N > kMaxRows || K <= 0 || K % 64 != 0 ||
        K > (1 << 24) || N % 8 != 0)
        return NVFP4_ERR_SHAPE;
    if (want_amax) {
        if (M > 0 && row_amax == nullptr) return NVFP4_ERR_NULL;
        if (misaligned(row_amax, 4)) return NVFP4_ERR_ALIGN;
    }
    if (M == 0) return NVFP4_OK;
    if (N > 0) {
        if (!a_codes || !a_sf || !a_srow || !w_codes || !w_sf || !w_st || !Y) return NVFP4_ERR_NULL;
        if (misaligned(a_codes, 16) || misaligned(a_sf, 16) || misaligned(w_codes, 16) ||
            misaligned(w_sf, 16) || misaligned(Y, 16) || misaligned(a_srow, 4) ||
            misaligned(w_st, 4) || (bias && misaligned(bias, 16)))
            return NVFP4_ERR_ALIGN;
        if (epi == kGemmEpiResidual && (!residual || misaligned(residual, 16) || N % 32 != 0))
            return NVFP4_ERR_SHAPE;
    }
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    if (want_amax) {
        // The epilogue max-reduces into zeros (an empty row's amax is 0).
        const cudaError_t e = cudaMemsetAsync(row_amax, 0, (size_t)M * sizeof(float), ctx.stream);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (N == 0) return NVFP4_OK;
    CUtensorMap ta, tb, tsa, tsb, ty;
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, (uint64_t)K / 2, (uint64_t)M,
                   (uint64_t)K / 2, 128, 128) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_codes, (uint64_t)K / 2, (uint64_t)N,
                   (uint64_t)K / 2, 128, 128) ||
        !encode_sf(&tsa, a_sf, M, K) || !encode_sf(&tsb, w_sf, N, K) || !encode_out(&ty, Y, M, N))
        return NVFP4_ERR_CUDA;
    if (epi != 0)
        return from_cuda(launch_gemm_nvfp4_epi(ctx, ta, tb, tsa, tsb, ty, a_srow, w_st,
                                               static_cast<const __nv_bfloat16*>(bias), M, N, K, epi, residual));
    return from_cuda(launch_gemm_nvfp4(ctx, ta, tb, tsa, tsb, ty, a_srow, w_st,
                                       static_cast<const __nv_bfloat16*>(bias), M, N, K, withhold_kb,
                                       wait_limit_ns, want_amax ? row_amax : nullptr));
}

nvfp4_status nvfp4_gemm_rowamax(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                                const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                                const void* bias, void* Y, float* y_row_amax, int64_t M, int64_t N,
                                int64_t K, void* stream) {
    return gemm_nvfp4_call(a_codes, a_sf, a_srow, w_codes, w_sf, w_st, bias, Y, M, N, K, stream, -1, 0,
                           y_row_amax, true);
}

nvfp4_status nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                        const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* stream) {
    return gemm_nvfp4_call(a_codes, a_sf, a_srow, w_codes, w_sf, w_st, bias, Y, M, N, K, stream, -1, 0);
}

nvfp4_status nvfp4_test_gemm_withhold(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_srow,
                                      const uint8_t* w_codes, const uint8_t* w_sf, const float* w_st,
                                      void* Y, int64_t M, int64_t N, int64_t K, int withhold_kb,
                                      int64_t timeout_ns, void* stream) {
    if (withhold_kb < 0 || (int64_t)withhold_kb * 256 >= K || timeout_ns < 1000000 ||
        timeout_ns > 1000000000LL)
        return NVFP4_ERR_SHAPE;
    return gemm_nvfp4_call(a_codes, a_sf, a_srow, w_codes, w_sf, w_st, nullptr, Y, M, N, K, stream,
                           withhold_kb, timeout_ns);
}

nvfp4_status bf16_gemm(const void* X, const void* W, const void* bias, void* Y, int64_t M,
                       int64_t N, int64_t K, void* stream) {
    if (M < 0 || N < 0 || M > kMaxRows || N > kMaxRows || K <= 0 || K % 8 != 0 ||
        K > (1 << 24) || N % 8 != 0)
        return NVFP4_ERR_SHAPE;
    if (M == 0 || N == 0) return NVFP4_OK;
    if (!X || !W || !Y) return NVFP4_ERR_NULL;
    if (misaligned(X, 16) || misaligned(W, 16) || misaligned(Y, 16) || (bias && misaligned(bias, 16)))
        return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    CUtensorMap ta, tb, ty;
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)K, (uint64_t)M,
                   (uint64_t)K * 2, 64, 128) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)K, (uint64_t)N,
                   (uint64_t)K * 2, 64, 128) ||
        !encode_out(&ty, Y, M, N))
        return NVFP4_ERR_CUDA;
    return from_cuda(launch_gemm_bf16(ctx, ta, tb, ty, static_cast<const __nv_bfloat16*>(bias), M,
                                      N, K));
}

// ------------------------------------------------------------------ synthetic DiT block

static size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static bool block_shape_ok(int64_t B, int64_t S, int64_t D, int64_t H) {
    if (B <= 0 || S <= 0 || D <= 0 || H <= 0) return false;
    if (D % 64 != 0 || D % H != 0 || S % 64 != 0) return false;
    const int64_t dh = D / H;
    if (dh != 64 && dh != 128) return false;
    if (B * S > kMaxRows || B * H > 65535 || S > (1 << 20) || 4 * D > (1 << 20)) return false;
    return true;
}

// Attention scratch: V^T [B*H, dh, S] (the only operand the fused kernel does not read
// from qkv directly).
static size_t attn_bytes(int64_t B, int64_t S, int64_t D) { return up256((size_t)B * S * D * 2); }

size_t nvfp4_dit_attention_workspace_bytes(int64_t B, int64_t S, int64_t D, int64_t H) {
    if (!block_shape_ok(B, S, D, H)) return 0;
    return attn_bytes(B, S, D);
}

// The attention of the block: v transposed per head, then the fused two-pass kernel
// (attn.cu), which reads q and k from qkv and writes o in the [B*S, D] layout.
static nvfp4_status attention_run(const LaunchCtx& ctx, const uint16_t* qkv, int64_t B, int64_t S, int64_t D,
                                  int64_t H, uint16_t* o, uint16_t* Vt, int withhold = -1, int64_t wait_limit_ns = 0) {
    const int64_t dh = D / H, T = B * S;
    CUtensorMap tqk, tv;
    if (!encode_2d(&tqk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)(3 * D), (uint64_t)T, (uint64_t)(3 * D) * 2,
                   64, 128) ||
        !encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Vt, (uint64_t)S, (uint64_t)(B * H * dh), (uint64_t)S * 2,
                   64, (uint32_t)(dh / 2)))
        return NVFP4_ERR_CUDA;
    cudaError_t e = launch_heads_vt(ctx, qkv, B, S, D, H, Vt);
    if (e != cudaSuccess) return from_cuda(e);
    const float scale = 1.0f / sqrtf((float)dh);
    return from_cuda(launch_attention(ctx, tqk, tv, o, B, S, D, H, scale, withhold, wait_limit_ns));
}

static nvfp4_status dit_attention_call(const void* qkv, int64_t B, int64_t S, int64_t D, int64_t H, void* o,
                                       void* workspace, size_t workspace_bytes, void* stream, int withhold,
                                       int64_t wait_limit_ns) {
    if (!block_shape_ok(B, S, D, H)) return NVFP4_ERR_SHAPE;
    if (!qkv || !o || !workspace) return NVFP4_ERR_NULL;
    if (misaligned(qkv, 16) || misaligned(o, 16) || misaligned(workspace, 256)) return NVFP4_ERR_ALIGN;
    if (workspace_bytes < attn_bytes(B, S, D)) return NVFP4_ERR_SHAPE;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return attention_run(ctx, static_cast<const uint16_t*>(qkv), B, S, D, H, static_cast<uint16_t*>(o),
                         static_cast<uint16_t*>(workspace), withhold, wait_limit_ns);
}

nvfp4_status nvfp4_dit_attention(const void* qkv, int64_t B, int64_t S, int64_t D, int64_t H, void* o,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    return dit_attention_call(qkv, B, S, D, H, o, workspace, workspace_bytes, stream, -1, 0);
}

nvfp4_status nvfp4_test_attention_withhold(const void* qkv, int64_t B, int64_t S, int64_t D, int64_t H, void* o,
                                           void* workspace, size_t workspace_bytes, int withhold_tile,
                                           int64_t timeout_ns, void* stream) {
    const int64_t n_tiles = (S + 255) / 256;
    if (withhold_tile < 0 || withhold_tile >= n_tiles || timeout_ns < 1000000 || timeout_ns > 1000000000LL)
        return NVFP4_ERR_SHAPE;
    return dit_attention_call(qkv, B, S, D, H, o, workspace, workspace_bytes, stream, withhold_tile, timeout_ns);
}

// Block scratch: R1 [3 T D] holds qkv, then o; R2 [4 T D] holds the attention's V^T,
// then the GELU output of the up-projection; h1 [T D]; the activation quantization of a
// D-wide tensor (x, o, h1 in turn) and of the 4D-wide GELU output.
struct BlockLayout {
    uint16_t *r1, *r2, *h1;
    uint8_t *qa_codes, *qa_sf, *qb_codes, *qb_sf;
    float *qa_s, *qb_s;
    size_t bytes;
};
static BlockLayout block_layout(void* base, int64_t B, int64_t S, int64_t D) {
    BlockLayout l;
    const int64_t T = B * S;
    const size_t td = up256((size_t)T * D * 2);
    size_t off = 0;
    uint8_t* p = static_cast<uint8_t*>(base);
    auto take = [&](size_t n) {
        uint8_t* q = p + off;
        off += up256(n);
        return q;
    };
    l.r1 = reinterpret_cast<uint16_t*>(take(3 * td));
    l.r2 = reinterpret_cast<uint16_t*>(take(4 * td));
    l.h1 = reinterpret_cast<uint16_t*>(take(td));
    l.qa_codes = take((size_t)T * D / 2);
    l.qa_sf = take(nvfp4_sf_bytes(T, D));
    l.qa_s = reinterpret_cast<float*>(take((size_t)T * 4));
    l.qb_codes = take((size_t)T * 4 * D / 2);
    l.qb_sf = take(nvfp4_sf_bytes(T, 4 * D));
    l.qb_s = reinterpret_cast<float*>(take((size_t)T * 4));
    l.bytes = off;
    return l;
}

size_t nvfp4_dit_block_workspace_bytes(int64_t B, int64_t S, int64_t D, int64_t H) {
    if (!block_shape_ok(B, S, D, H)) return 0;
    return block_layout(nullptr, B, S, D).bytes;
}

nvfp4_status nvfp4_dit_block(const void* x, int64_t B, int64_t S, int64_t D, int64_t H,
                             const nvfp4_linear_weights* w, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (!block_shape_ok(B, S, D, H)) return NVFP4_ERR_SHAPE;
    if (!x || !w || !out || !workspace) return NVFP4_ERR_NULL;
    for (int i = 0; i < 4; ++i)
        if (!w[i].codes || !w[i].sf || !w[i].s_t) return NVFP4_ERR_NULL;
    if (misaligned(x, 16) || misaligned(out, 16) || misaligned(workspace, 256)) return NVFP4_ERR_ALIGN;
    const BlockLayout l = block_layout(workspace, B, S, D);
    if (workspace_bytes < l.bytes) return NVFP4_ERR_SHAPE;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    const int64_t T = B * S;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    uint16_t *qkv = l.r1, *o = l.r1, *u = l.r2;
    // lin(in) = nvfp4_gemm(nvfp4_act_quant(in)) + bias, with the GEMM epilogue's GELU or
    // residual add where the block applies one to the linear's output (the same bits as
    // the separate passes: bf16 output first, then the operation, then bf16).
    auto lin = [&](const uint16_t* in, int64_t K, uint8_t* c, uint8_t* sf, float* s, const nvfp4_linear_weights& wi,
                   int64_t N, uint16_t* y, int epi, const uint16_t* residual) {
        nvfp4_status r = nvfp4_act_quant(in, T, K, c, sf, s, stream);
        if (r != NVFP4_OK) return r;
        return gemm_nvfp4_call(c, sf, s, wi.codes, wi.sf, wi.s_t, wi.bias, y, T, N, K, stream, -1, 0, nullptr,
                               false, epi, residual);
    };
    if ((st = lin(xb, D, l.qa_codes, l.qa_sf, l.qa_s, w[0], 3 * D, qkv, 0, nullptr)) != NVFP4_OK) return st;
    if ((st = attention_run(ctx, qkv, B, S, D, H, o, l.r2)) != NVFP4_OK) return st;
    if ((st = lin(o, D, l.qa_codes, l.qa_sf, l.qa_s, w[1], D, l.h1, kGemmEpiResidual, xb)) != NVFP4_OK) return st;
    if ((st = lin(l.h1, D, l.qa_codes, l.qa_sf, l.qa_s, w[2], 4 * D, u, kGemmEpiGelu, nullptr)) != NVFP4_OK)
        return st;
    return lin(u, 4 * D, l.qb_codes, l.qb_sf, l.qb_s, w[3], D, static_cast<uint16_t*>(out), kGemmEpiResidual, l.h1);
}

nvfp4_status bf16_softmax_rows(const void* L, int64_t rows, int64_t cols, float scale, void* P,
                               void* stream) {
    if (rows < 0 || cols <= 0 || cols % 8 != 0 || rows > kMaxRows || cols > (1 << 24)) return NVFP4_ERR_SHAPE;
    if (rows == 0) return NVFP4_OK;
    if (!L || !P) return NVFP4_ERR_NULL;
    if (misaligned(L, 16) || misaligned(P, 16)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_softmax_rows(ctx, static_cast<const uint16_t*>(L), rows, cols, scale,
                                         static_cast<uint16_t*>(P)));
}

nvfp4_status bf16_gelu(const void* x, int64_t n, void* y, void* stream) {
    if (n < 0 || n % 8 != 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!x || !y) return NVFP4_ERR_NULL;
    if (misaligned(x, 16) || misaligned(y, 16)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_gelu(ctx, static_cast<const uint16_t*>(x), n, static_cast<uint16_t*>(y)));
}

nvfp4_status bf16_add(const void* a, const void* b, int64_t n, void* y, void* stream) {
    if (n < 0 || n % 8 != 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!a || !b || !y) return NVFP4_ERR_NULL;
    if (misaligned(a, 16) || misaligned(b, 16) || misaligned(y, 16)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    const nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_add(ctx, static_cast<const uint16_t*>(a), static_cast<const uint16_t*>(b), n,
                                static_cast<uint16_t*>(y)));
}

nvfp4_status select_contrastive(const float* rewards, int P, int N, int K, int global_std,
                                int32_t* idx, float* r_out, void* stream) {
    if (P < 0 || N < 1 || N > 1024 || K <= 0 || K % 2 != 0 || K > N) return NVFP4_ERR_SHAPE;
    if (P == 0) return NVFP4_OK;
    if (rewards == nullptr || idx == nullptr) return NVFP4_ERR_NULL;
    if (misaligned(rewards, 4) || misaligned(idx, 4) || (r_out && misaligned(r_out, 4)))
        return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_select(ctx, rewards, P, N, K, global_std ? 1 : 0, idx, r_out));
}

nvfp4_status nvfp4_device_status(int* out, int clear) {
    if (out == nullptr) return NVFP4_ERR_NULL;
    LaunchCtx ctx;
    nvfp4_status st = resolve(nullptr, &ctx);
    if (st != NVFP4_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_CUDA;
    }
    if (cudaMemcpyFromSymbol(out, g_status_word, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_test_e2m1(const float* q, uint8_t* codes, int64_t n, void* stream) {
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!q || !codes) return NVFP4_ERR_NULL;
    if (misaligned(q, 4)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_e2m1(ctx, q, codes, n));
}

nvfp4_status nvfp4_test_e4m3(const float* v, uint8_t* codes, int64_t n, void* stream) {
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!v || !codes) return NVFP4_ERR_NULL;
    if (misaligned(v, 4)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_e4m3(ctx, v, codes, n));
}

nvfp4_status nvfp4_test_e4m3_decode(const uint8_t* codes, float* out, int64_t n, void* stream) {
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!codes || !out) return NVFP4_ERR_NULL;
    if (misaligned(out, 4)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_e4m3_decode(ctx, codes, out, n));
}

nvfp4_status nvfp4_test_e2m1_quotient(const float* x, const float* den, uint8_t* codes, int64_t n,
                                      void* stream) {
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!x || !den || !codes) return NVFP4_ERR_NULL;
    if (misaligned(x, 4) || misaligned(den, 4)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_e2m1_quotient(ctx, x, den, codes, n));
}

nvfp4_status nvfp4_test_e4m3_quotient(const float* v, const float* d, uint8_t* codes, int64_t n,
                                      void* stream) {
    if (n < 0) return NVFP4_ERR_SHAPE;
    if (n == 0) return NVFP4_OK;
    if (!v || !d || !codes) return NVFP4_ERR_NULL;
    if (misaligned(v, 4) || misaligned(d, 4)) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_e4m3_quotient(ctx, v, d, codes, n));
}

nvfp4_status nvfp4_test_merge(const void* W, int w_dtype, const float* A, const float* B, int r,
                              float alpha, int64_t N, int64_t K, float* out, void* stream) {
    if (w_dtype != NVFP4_W_BF16 && w_dtype != NVFP4_W_FP32) return NVFP4_ERR_SHAPE;
    if (r < 0 || r > 64 || N < 0 || N > kMaxRows || K <= 0 || K % 64 != 0 || K > (1 << 20))
        return NVFP4_ERR_SHAPE;
    if (N == 0) return NVFP4_OK;
    if (W == nullptr || out == nullptr) return NVFP4_ERR_NULL;
    const bool merge = r > 0 && A != nullptr && B != nullptr;
    if (misaligned(W, 16) || misaligned(out, 16)) return NVFP4_ERR_ALIGN;
    if (merge && (misaligned(A, 16) || misaligned(B, 4))) return NVFP4_ERR_ALIGN;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    if (st != NVFP4_OK) return st;
    const float c = merge ? alpha / static_cast<float>(r) : 0.0f;
    return from_cuda(launch_test_merge(ctx, W, w_dtype, merge ? A : nullptr, merge ? B : nullptr,
                                       merge ? r : 0, c, N, K, out));
}

nvfp4_status nvfp4_test_wait_timeout(int64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return NVFP4_ERR_SHAPE;
    LaunchCtx ctx;
    nvfp4_status st = resolve(stream, &ctx);
    return st != NVFP4_OK ? st : from_cuda(launch_test_wait_timeout(ctx, timeout_ns));
}

}  // extern "C"
