// The NVFP4 GEMM's epilogue variants used by the synthetic DiT block (gemm.cu), and the
// GELU they share with the block's GELU kernel (block.cu), so both give the same bits.
#pragma once
#include "common.cuh"

namespace nvfp4rl {

// The NVFP4 GEMM (gemm.cu) with one of the block's epilogues applied to each output
// y = bf16(acc * s_a * s_w + bias) before it is stored: kGemmEpiGelu stores bf16(gelu(y)),
// kGemmEpiResidual stores bf16(y + residual[m, n]) (residual [M, N] bf16, N % 32 == 0,
// 16-byte aligned).  Same results as the plain GEMM followed by launch_gelu / launch_add.
constexpr int kGemmEpiGelu = 1, kGemmEpiResidual = 2;
cudaError_t launch_gemm_nvfp4_epi(const LaunchCtx&, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                  const CUtensorMap& tmap_sfa, const CUtensorMap& tmap_sfb,
                                  const CUtensorMap& tmap_y, const float* a_srow, const float* w_st,
                                  const __nv_bfloat16* bias, int64_t M, int64_t N, int64_t K, int epi,
                                  const uint16_t* residual);

#if defined(__CUDACC__)
// GELU of two fp32 values in its tanh form, g(x) = x (1 + tanh(t)) / 2 with
// t = sqrt(2/pi) (x + 0.044715 x^3), through the identity (1 + tanh(t)) / 2 =
// 1 / (1 + e^(-2t)) evaluated without cancellation: u = e^(-2|t|) in (0, 1],
// r = 1 / (1 + u), and the logistic value is r for t >= 0 and u r for t < 0.
// ex2.approx (no flush to zero: the function's tail reaches bf16's subnormal range near
// x = -10) and rcp.approx (of a value in (1, 2]) each err by a few ulps of fp32, far
// below bf16's rounding step; the rest is packed fp32 arithmetic, each lane rounded as
// the scalar operation would be.  Shared by the GELU kernel and the GEMM epilogue, so
// both give the same bits.
__device__ __forceinline__ float2 gelu_f32x2(float2 v) {
    // 2t log2(e) = 2 sqrt(2/pi) log2(e) (v + 0.044715 v^3)
    const float2 p = __ffma2_rn(__fmul2_rn(make_float2(0.044715f, 0.044715f), v), __fmul2_rn(v, v), v);
    const float2 t2 = __fmul2_rn(make_float2(2.3022082f, 2.3022082f), p);
    float2 u, r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(u.x) : "f"(-fabsf(t2.x)));
    asm("ex2.approx.f32 %0, %1;" : "=f"(u.y) : "f"(-fabsf(t2.y)));
    const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), u);
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(d.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(d.y));
    const float2 ur = __fmul2_rn(u, r);
    return __fmul2_rn(v, make_float2(t2.x >= 0.0f ? r.x : ur.x, t2.y >= 0.0f ? r.y : ur.y));
}
#endif

}  // namespace nvfp4rl
