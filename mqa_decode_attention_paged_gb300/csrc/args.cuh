// Kernel argument blocks, passed by value to the stage-1 and stage-2
// kernels and filled in by the C ABI layer (api.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "plan.cuh"

namespace mqa {

// Upper bound on balanced-mode work units (the merge stages one weight per
// unit in shared memory).
constexpr int kMaxMergeUnits = 1024;

// Largest batch whose page prefix the stage-1 kernels keep in shared memory.
constexpr int kMaxBatchSmem = 2048;

struct MlaArgs {
    // 3D tiled view of the cache whose box is box_rows whole cache rows
    // (bf16: 64-element panels with the 128-byte swizzle; e4m3: unswizzled).
    CUtensorMap tmap;
    int box_rows;
    const __nv_bfloat16* q;
    const uint8_t* kv;
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;    // [slots, H, R]
    float* ws_lse;  // [slots, H]
    int* status;
    float sl2;        // scale * k_scale(fp8) * log2(e)
    float out_scale;  // k_scale for fp8, 1 for bf16
    int H, num_blocks;
    // multi-token decode: the H rows are q_len query tokens x heads
    // (token-major); row r (token i = r / heads) sees the first
    // len - q_len + i + 1 tokens of its request.  q_len = 1: plain decode.
    int q_len, heads;
    // sparse decode (indices != null): request b attends the positions
    // indices[b * topk + e]; the plan runs over the topk entries in "pages"
    // of one pipeline tile (plan.fixed_len = topk) and a selected position's
    // row is found through block_table (row stride bt_stride) with pages of
    // cache_page tokens
    const int32_t* indices;
    int topk, cache_page, bt_stride;
    // test hook of the bounded waits (-1 in every product call): the producer
    // of work unit `withhold` fills and announces none of its tiles
    int withhold;
    Plan plan;
};

// H = 128 tensor-core MLA path (2-CTA clusters split by feature columns).
struct MlaTcArgs {
    // The cache (bf16, or e4m3 unswizzled): with box_rows == 64 as a 3D
    // tensor {64, num_blocks * page, D / 64} with box {64, 64, R / 128}
    // (kv_pair_map[0]: one rank's kv_c panels of a 64-token pair), else as a
    // 2D tensor {D, num_blocks * page} with box {64, box_rows} (kv_map); the
    // rope halves as a 2D tensor with box {32, box_rows} (kv_rope_map).  bf16
    // panels use the 128-byte swizzle, bf16 rope halves the 64-byte one.
    CUtensorMap kv_map;
    CUtensorMap kv_pair_map[2];
    CUtensorMap kv_rope_map;
    int box_rows;
    const __nv_bfloat16* q;  // [B, H, D]
    const uint8_t* kv;       // cache rows of D bf16 values
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;
    float* ws_lse;
    int* status;
    float sl2;
    float out_scale;
    int H, num_blocks;
    int q_len, heads;  // multi-token decode rows, as in MlaArgs
    int withhold;      // test hook, as in MlaArgs (-1 in every product call)
    // test hook (-1 in every product call): softmax warp give_up % 16 of unit
    // give_up / 16 gives up before its first pair as if a wait had expired
    int give_up;
    Plan plan;
};

struct GqaArgs {
    const __nv_bfloat16* q;
    const uint8_t* kv;
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;
    float* ws_lse;
    int* status;
    float sl2;
    int Hq, Hkv, num_blocks;
    Plan plan;
};

struct MergeArgs {
    const float* ws_o;    // [slots, H, R]
    const float* ws_lse;  // [slots, H]
    const int32_t* seq_lens;
    __nv_bfloat16* out;   // [B, H, R]
    float* lse;           // [B, H] or null
    int* status;
    float out_scale;
    int H, R;
    Plan plan;
};

cudaError_t mla_mma_stage1(const MlaArgs& a, int D, bool fp8, int grid, cudaStream_t stream);
size_t mla_mma_smem_bytes(int D, bool fp8, int batch);
int mla_mma_tile();
// entries per pipeline tile of the sparse (index-gather) kernel
int mla_mma_sparse_tile(bool fp8);
cudaError_t gqa_mma_stage1(const GqaArgs& a, int D, int grid, cudaStream_t stream);
cudaError_t mla_tc_stage1(const MlaTcArgs& a, int D, bool fp8, int clusters, cudaStream_t stream);
int mla_tc_tile();
constexpr int kMaxBatchTc = 512;  // page prefix of the H = 128 path lives in smem
size_t gqa_mma_smem_bytes(int D, int hkv, int batch);
cudaError_t lse_merge(const MergeArgs& a, cudaStream_t stream);

}  // namespace mqa
