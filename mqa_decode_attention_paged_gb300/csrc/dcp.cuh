// Local step of the DCP all-gather-lse / reduce-scatter-output merge (dcp.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mqa {

// in: bf16 [B, H, D] (this rank's shard output); lses: fp32 [G, B, H];
// dst: [G, B, H / G, D], fp32 if f32 else bf16; lse: fp32 [B, H] or null.
// H a multiple of G, D a multiple of 8, pointers 16-byte aligned.
cudaError_t dcp_scale(const __nv_bfloat16* in, const float* lses, void* dst, float* lse, int G, int rank, int B,
                      int H, int D, bool f32, cudaStream_t stream);

}  // namespace mqa
