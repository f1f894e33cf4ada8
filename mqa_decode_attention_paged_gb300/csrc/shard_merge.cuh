// Merge of sequence-shard results (shard_merge.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mqa {

// outs: bf16 [G, rows, R], lses: fp32 [G, rows]; out: bf16 [rows, R], lse:
// fp32 [rows] or null.  R a multiple of 8, pointers 16-byte aligned.
cudaError_t shard_merge(const __nv_bfloat16* outs, const float* lses, __nv_bfloat16* out, float* lse, int G,
                        long long rows, int R, cudaStream_t stream);

}  // namespace mqa
