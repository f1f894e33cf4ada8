// Stage 1 of GQA paged decode over 8-bit caches (gqa_q8.cu).
#pragma once

#include "args.cuh"

namespace mqa {

// Cache formats served by gqa_q8_stage1 (the values of mqa_kv_dtype):
//   1  e4m3 codes, one k_scale / v_scale for the whole cache;
//   2  e4m3 codes, per (token, KV head) row: D codes + its fp32 scale;
//   3  int8 codes, per (token, KV head) row: D codes + its fp32 scale;
//   4  int4 codes, per (token, KV head) row: D / 2 bytes of codes (element 2i
//      in the low nibble of byte i) + its fp32 scale.
// out_scale multiplies the output (v_scale for format 1, 1 otherwise); the
// softmax scale in a.sl2 already holds k_scale for format 1.
cudaError_t gqa_q8_stage1(const GqaArgs& a, float out_scale, int D, int kind, int grid, cudaStream_t stream);
size_t gqa_q8_smem_bytes(int D, int kind, int hkv, int q_per_kv, int batch);
// Blocks of the kernel resident per SM (2 for up to 8 query heads per KV
// head, else 1): the balanced plan should make that many units per SM.
int gqa_q8_ctas_per_sm(int q_per_kv);

}  // namespace mqa
