// Launch functions of the synthetic DiT block's kernels: the v transpose, the row
// softmax, the GELU and the residual add (block.cu), and the fused attention
// (attn.cu).  Each enqueues one kernel on ctx.stream and returns the launch error;
// arguments are checked by the caller (api.cu).
#pragma once
#include "common.cuh"
#include "gemm_epilogue.cuh"

namespace nvfp4rl {

cudaError_t launch_heads_vt(const LaunchCtx&, const uint16_t* qkv, int64_t B, int64_t S, int64_t D, int64_t H,
                            uint16_t* Vt);
// The fused attention (attn.cu): Q and K tiles from qkv [B*S, 3D] (tmap_qk: 64 x 128
// boxes, 128-byte swizzle), V^T [B*H*dh, S] (tmap_vt: 64 x dh/2 boxes), o [B*S, D]
// written at columns h*dh; dh = D/H is 64 or 128.
// withhold >= 0 and wait_limit_ns > 0 only from the test hook (nvfp4_test_attention_withhold).
cudaError_t launch_attention(const LaunchCtx&, const CUtensorMap& tmap_qk, const CUtensorMap& tmap_vt, uint16_t* o,
                             int64_t B, int64_t S, int64_t D, int64_t H, float scale, int withhold = -1,
                             int64_t wait_limit_ns = 0);
cudaError_t launch_softmax_rows(const LaunchCtx&, const uint16_t* L, int64_t rows, int64_t cols, float scale,
                                uint16_t* P);
cudaError_t launch_gelu(const LaunchCtx&, const uint16_t* x, int64_t n, uint16_t* y);
cudaError_t launch_add(const LaunchCtx&, const uint16_t* a, const uint16_t* b, int64_t n, uint16_t* y);


}  // namespace nvfp4rl
