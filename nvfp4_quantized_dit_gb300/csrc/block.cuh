// Launch functions of the synthetic DiT block's streaming kernels (block.cu): head split
// and merge, the attention softmax, the GELU and the residual add.  Each enqueues one
// kernel on ctx.stream and returns the launch error; arguments are checked by the
// caller (api.cu).
#pragma once
#include "common.cuh"

namespace nvfp4rl {

cudaError_t launch_heads_split(const LaunchCtx&, const uint16_t* qkv, int64_t B, int64_t S, int64_t D,
                               int64_t H, uint16_t* Q, uint16_t* K, uint16_t* Vt);
cudaError_t launch_heads_merge(const LaunchCtx&, const uint16_t* O, int64_t B, int64_t S, int64_t D,
                               int64_t H, uint16_t* o);
cudaError_t launch_softmax_rows(const LaunchCtx&, const uint16_t* L, int64_t rows, int64_t cols, float scale,
                                uint16_t* P);
cudaError_t launch_gelu(const LaunchCtx&, const uint16_t* x, int64_t n, uint16_t* y);
cudaError_t launch_add(const LaunchCtx&, const uint16_t* a, const uint16_t* b, int64_t n, uint16_t* y);

}  // namespace nvfp4rl
