// Test hook of the bf16 GQA stage-1 kernel (gqa_mma.cu).
#pragma once

#include "args.cuh"

namespace mqa {

// gqa_mma_stage1 with the producer of unit `withhold` never filling or
// announcing its first tile: its consumers' bounded wait runs out and the
// kernel reports MQA_ERR_DEVICE_TIMEOUT and returns (failure detection
// tested without a fault or a hang).
cudaError_t gqa_mma_stage1_withheld(const GqaArgs& a, int D, int grid, int withhold, cudaStream_t stream);

}  // namespace mqa
