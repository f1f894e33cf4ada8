// C ABI entry points: argument validation, work decomposition and launches.
// See include/mqa_decode.h for the contract of every function.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "plan.cuh"
#include "../../include/mqa_decode_testing.h"

#include "args.cuh"
#include "gqa_q8.cuh"
#include "shard_merge.cuh"
#include "dcp.cuh"
#include "gqa_test.cuh"

namespace {

// Last CUDA error seen by this thread inside the library (for diagnostics).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

mqa_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = e;
    return MQA_ERR_CUDA;
}

constexpr int kMaxBatch = mqa::kMaxBatchSmem;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Test hooks run only when MQA_ENABLE_TEST_HOOKS is "1" (mqa_decode_testing.h).
bool test_hooks_enabled() {
    const char* v = std::getenv("MQA_ENABLE_TEST_HOOKS");
    return v && v[0] == '1' && v[1] == '\0';
}

int sm_count_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

size_t partial_bytes(int batch, int heads, int width, int splits) {
    if (batch <= 0 || heads <= 0 || width <= 0 || splits <= 0) return 0;
    if (splits == 1) return 0;
    return static_cast<size_t>(batch) * heads * splits * (static_cast<size_t>(width) + 1) * 4;
}

// Pages that a request start costs a unit in the balanced plan of the bf16
// H > 32 tensor-core kernel: 512 tokens' worth, the best of 256, 512 and 1024
// on the long-context and multi-token batches.  (A new request costs that
// kernel its query staging behind the last Q.K^T of the previous one and a
// pipeline fill.  The e4m3 kernel stages the query on its idle group and is
// faster with plain page balance.)
int tc_piece_cost(int page_size) { return (512 + page_size - 1) / page_size; }

// Work units for balanced mode: about `resident` thread blocks per head
// group, never more than the workspace's partial budget allows.
int balanced_units(int batch, int splits, int resident_per_group) {
    long long cap = static_cast<long long>(batch) * (splits - 1) + 1;
    long long u = resident_per_group < 1 ? 1 : resident_per_group;
    if (u > mqa::kMaxMergeUnits) u = mqa::kMaxMergeUnits;
    return static_cast<int>(u < cap ? u : cap);
}

// ---- tensor maps (TMA descriptors) for bf16 MLA caches ----------------------

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    const void* base;
    long long rows;
    int cols, box_rows, kind;  // kind: 0 = 3D bf16 rows, 1 = 3D e4m3 rows, 2 = 2D bf16 panels
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && cols == o.cols && box_rows == o.box_rows && kind == o.kind;
    }
};

constexpr int kMapSlots = 32;
std::mutex g_map_mu;
MapKey g_map_keys[kMapSlots];
CUtensorMap g_maps[kMapSlots];
int g_map_used = 0, g_map_next = 0;

bool map_lookup(const MapKey& key, CUtensorMap* out) {
    for (int i = 0; i < g_map_used; ++i)
        if (g_map_keys[i] == key) {
            *out = g_maps[i];
            return true;
        }
    return false;
}

void map_store(const MapKey& key, const CUtensorMap& m) {
    const int slot = g_map_used < kMapSlots ? g_map_used++ : (g_map_next++ % kMapSlots);
    g_map_keys[slot] = key;
    g_maps[slot] = m;
}

// 2D view {cols, rows} of a row-major bf16 matrix with {64, box_rows} boxes and
// the 128-byte swizzle: one copy lands one 64-column panel of box_rows rows in
// the canonical K-major layout of the tensor cores.
bool bf16_panel_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_rows) {
    const MapKey key{base, rows, cols, box_rows, 2};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

// 3D view {64 elements, rows, cols/64 panels} of a row-major bf16 matrix whose
// box is {64, 64 rows, box_panels} with the 128-byte swizzle: one copy lands
// box_panels panels of 64 consecutive rows, panel after panel, which is the
// K-major operand layout of the tensor cores for each panel.  The panel
// dimension has the smaller stride (128 bytes) than the row dimension.
bool bf16_pair_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_panels) {
    const MapKey key{base, rows, cols, box_panels, 3};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
    const cuuint32_t box[3] = {64, 64, static_cast<cuuint32_t>(box_panels)};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

// e4m3 counterparts of the two views above, unswizzled: {64 bytes, rows,
// cols/64 panels} with box {64, 64, box_panels} (one pair, panel after panel,
// 64 bytes per row), and {cols, rows} with box {64, box_rows}.
bool e4m3_pair_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_panels) {
    const MapKey key{base, rows, cols, box_panels, 4};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), 64};
    const cuuint32_t box[3] = {64, 64, static_cast<cuuint32_t>(box_panels)};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

bool e4m3_panel_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_rows) {
    const MapKey key{base, rows, cols, box_rows, 5};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

// 2D view {cols, rows} of the cache with box {32, box_rows}: the 32-column
// rope halves, with the 64-byte swizzle for bf16 (the K-major operand layout
// of 64-byte rows) and unswizzled for e4m3.
bool rope_half_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_rows, bool fp8) {
    const MapKey key{base, rows, cols, box_rows, fp8 ? 7 : 6};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const int elt = fp8 ? 1 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elt};
    const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
           dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
           fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

// 2D view {row_bytes / 8, rows} of the cache as 8-byte elements, unswizzled,
// with a box one row high and box_elems wide, for four-row gathers: a box
// wider than the row is filled with zeros past it (bf16 sparse decode pads
// its staged rows that way).
bool gather_row_map(CUtensorMap* out, const void* base, int row_bytes, long long rows, int box_elems) {
    const MapKey key{base, rows, row_bytes, box_elems, 8};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 8), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_elems), 1};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, const_cast<void*>(base), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

// Encodes (or returns a cached copy of) a 3D view of a row-major MLA cache
// [rows, cols] whose box is `box_rows` whole rows: bf16 rows are viewed as
// {64 elements, cols/64 panels, rows} with the 128-byte swizzle, e4m3 rows as
// {inner, cols/inner, rows} (inner <= 256 bytes) without swizzle.  One copy of
// the box fetches box_rows complete cache rows.
bool mla_tensor_map(CUtensorMap* out, const void* base, int cols, long long rows, int box_rows, bool fp8) {
    const MapKey key{base, rows, cols, box_rows, fp8 ? 1 : 0};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_lookup(key, out)) return true;
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const int inner = fp8 ? (cols % 192 == 0 ? 192 : 160) : 64;  // elements
    const int elt = fp8 ? 1 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(cols / inner),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * elt, static_cast<cuuint64_t>(cols) * elt};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(cols / inner),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (fn(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
           const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
           fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, m);
    *out = m;
    return true;
}

}  // namespace

static mqa_status mla_decode_rows(const void* q, const void* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                      int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                      int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                      void* workspace, size_t workspace_bytes, int* device_status, void* stream,
                      int q_len, int withhold = -1, bool fixed_splits = false, int give_up = -1) {
    // num_heads counts rows here: q_len query tokens x heads, token-major;
    // withhold >= 0 only from the test hook mqa_test_mla_withheld_arrive;
    // fixed_splits: one unit per (request, range) instead of page-balanced units;
    // give_up >= 0 only from the test hook mqa_test_mla_warp_gives_up
    if (!q || !kv_cache || !block_table || !seq_lens || !out) return MQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) || (device_status && !aligned(device_status, 4)))
        return MQA_ERR_INVALID_ARG;
    if (batch < 1 || num_heads < 1 || num_blocks < 1 || max_blocks < 1 || page_size < 1 || num_kv_splits < 1)
        return MQA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !std::isfinite(k_scale)) return MQA_ERR_INVALID_ARG;
    if (!((head_size == 576 && kv_lora_rank == 512) || (head_size == 320 && kv_lora_rank == 256)))
        return MQA_ERR_UNSUPPORTED;
    if (page_size % 16 != 0) return MQA_ERR_UNSUPPORTED;
    if (kv_dtype != MQA_KV_BF16 && kv_dtype != MQA_KV_FP8_E4M3) return MQA_ERR_UNSUPPORTED;
    if (num_heads > 128 || batch > kMaxBatch) return MQA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_blocks) * page_size > INT32_MAX ||
        static_cast<long long>(num_blocks) * page_size > INT32_MAX)
        return MQA_ERR_UNSUPPORTED;

    const size_t need = mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank, num_kv_splits);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MQA_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && !aligned(workspace, 16)) return MQA_ERR_INVALID_ARG;

    // fixed-split mode launches batch * num_kv_splits units (times the head
    // groups on the warp-MMA path)
    if (fixed_splits && static_cast<long long>(batch) * num_kv_splits > (1LL << 24)) return MQA_ERR_UNSUPPORTED;

    const int sms = sm_count_current();
    if (sms < 1) return MQA_ERR_CUDA;
    const bool fp8 = kv_dtype == MQA_KV_FP8_E4M3;
    const int groups = (num_heads + 15) / 16;
    const bool fixed = fixed_splits && num_kv_splits > 1;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t slots_tc = static_cast<size_t>(batch) * num_kv_splits;

    // 33..128 heads (or rows): 2-CTA tensor-core clusters, which read the
    // cache once whatever the head count (the warp-MMA kernel reads it once
    // per 16-head group: 2.3x slower at 64 heads, 5 % faster at 32, measured
    // on the V2-Lite-like batch); an e4m3 cache is widened to
    // f16 in shared memory)
    if (num_heads > 32 && batch <= mqa::kMaxBatchTc) {
        mqa::MlaTcArgs t{};
        // boxes never straddle a page and never exceed a pipeline tile
        // pages of 64 tokens or more hold whole 64-token pairs: one 3D copy per
        // pair and rank; smaller pages take one 2D copy per page and panel
        const int br = (page_size % 64 == 0) ? 64 : (page_size % 32 == 0 ? 32 : 16);
        t.box_rows = br;
        const long long kv_rows = static_cast<long long>(num_blocks) * page_size;
        // each rank holds kv_lora_rank / 128 full 64-column panels and one
        // 32-column half of the rope part
        const int rank_panels = kv_lora_rank / 128;
        auto pair_map = fp8 ? e4m3_pair_map : bf16_pair_map;
        auto panel_map = fp8 ? e4m3_panel_map : bf16_panel_map;
        if (br == 64) {
            if (!pair_map(&t.kv_pair_map[0], kv_cache, head_size, kv_rows, rank_panels))
                return cuda_fail(cudaErrorInvalidValue);
        } else if (!panel_map(&t.kv_map, kv_cache, head_size, kv_rows, br)) {
            return cuda_fail(cudaErrorInvalidValue);
        }
        if (!rope_half_map(&t.kv_rope_map, kv_cache, head_size, kv_rows, br, fp8))
            return cuda_fail(cudaErrorInvalidValue);
        t.q = static_cast<const __nv_bfloat16*>(q);
        t.kv = static_cast<const uint8_t*>(kv_cache);
        t.block_table = block_table;
        t.seq_lens = seq_lens;
        t.out = static_cast<__nv_bfloat16*>(out);
        t.lse = lse;
        t.ws_o = static_cast<float*>(workspace);
        t.ws_lse = need > 0 ? t.ws_o + slots_tc * num_heads * kv_lora_rank : nullptr;
        t.status = device_status;
        // an e4m3 cache holds K / k_scale: k_scale scales the logits and, as
        // V's scale, the output
        t.sl2 = scale * (fp8 ? k_scale : 1.0f) * mqa::kLog2e;
        t.out_scale = fp8 ? k_scale : 1.0f;
        t.H = num_heads;
        t.q_len = q_len;
        t.heads = num_heads / q_len;
        t.withhold = withhold;
        t.give_up = give_up;
        t.num_blocks = num_blocks;
        t.plan.batch = batch;
        t.plan.page = page_size;
        t.plan.max_blocks = max_blocks;
        t.plan.per_seq = num_kv_splits == 1 ? 1 : 0;
        t.plan.fixed_splits = fixed ? num_kv_splits : 0;
        // bf16 cache: balanced units also charge every request start
        t.plan.piece_cost = (t.plan.per_seq || fixed || fp8) ? 0 : tc_piece_cost(page_size);
        t.plan.units = t.plan.per_seq ? batch
                       : fixed        ? batch * num_kv_splits
                                      : balanced_units(batch, num_kv_splits, sms / 2);
        if (cudaError_t e = mqa::mla_tc_stage1(t, head_size, fp8, t.plan.units, st); e != cudaSuccess)
            return cuda_fail(e);
        if (!t.plan.per_seq) {
            mqa::MergeArgs m{};
            m.ws_o = t.ws_o;
            m.ws_lse = t.ws_lse;
            m.seq_lens = seq_lens;
            m.out = t.out;
            m.lse = lse;
            m.status = device_status;
            m.out_scale = 1.0f;
            m.H = num_heads;
            m.R = kv_lora_rank;
            m.plan = t.plan;
            if (cudaError_t e = mqa::lse_merge(m, st); e != cudaSuccess) return cuda_fail(e);
        }
        return MQA_OK;
    }

    mqa::MlaArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const uint8_t*>(kv_cache);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    const size_t slots = static_cast<size_t>(batch) * num_kv_splits;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = need > 0 ? a.ws_o + slots * num_heads * kv_lora_rank : nullptr;
    a.status = device_status;
    const float ks = fp8 ? k_scale : 1.0f;
    a.sl2 = scale * ks * mqa::kLog2e;
    a.out_scale = ks;
    a.H = num_heads;
    a.q_len = q_len;
    a.heads = num_heads / q_len;
    a.withhold = withhold;
    a.num_blocks = num_blocks;
    a.plan.batch = batch;
    a.plan.page = page_size;
    a.plan.max_blocks = max_blocks;
    a.plan.per_seq = num_kv_splits == 1 ? 1 : 0;
    a.plan.fixed_splits = fixed ? num_kv_splits : 0;
    a.plan.units = a.plan.per_seq ? batch
                   : fixed        ? batch * num_kv_splits
                                  : balanced_units(batch, num_kv_splits, sms / groups);

    {
        // tensor boxes never straddle a page: 64 rows when pages are multiples
        // of 64 tokens, else 32 or 16
        const int tile = mqa::mla_mma_tile();
        int br = (page_size % 64 == 0) ? 64 : (page_size % 32 == 0 ? 32 : 16);
        if (br > tile) br = tile;
        a.box_rows = br;
        if (!mla_tensor_map(&a.tmap, kv_cache, head_size, static_cast<long long>(num_blocks) * page_size, br,
                            fp8))
            return cuda_fail(cudaErrorInvalidValue);
    }

    if (cudaError_t e = mqa::mla_mma_stage1(a, head_size, fp8, a.plan.units * groups, st); e != cudaSuccess)
        return cuda_fail(e);
    if (!a.plan.per_seq) {
        mqa::MergeArgs m{};
        m.ws_o = a.ws_o;
        m.ws_lse = a.ws_lse;
        m.seq_lens = seq_lens;
        m.out = a.out;
        m.lse = lse;
        m.status = device_status;
        m.out_scale = 1.0f;  // stage-1 partials already carry k_scale
        m.H = num_heads;
        m.R = kv_lora_rank;
        m.plan = a.plan;
        if (cudaError_t e = mqa::lse_merge(m, st); e != cudaSuccess) return cuda_fail(e);
    }
    return MQA_OK;
}

extern "C" {

int mqa_abi_version(void) { return MQA_ABI_VERSION; }

const char* mqa_status_string(int status) {
    switch (status) {
        case MQA_OK: return "ok";
        case MQA_ERR_INVALID_ARG: return "invalid argument";
        case MQA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case MQA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MQA_ERR_CUDA: return "CUDA error";
        case MQA_ERR_DEVICE_CHECK: return "device check failed (block id or sequence length)";
        case MQA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

int mqa_device_sm_count(void) { return sm_count_current(); }

int mqa_last_cuda_error(void) { return static_cast<int>(g_last_cuda_error); }

const char* mqa_last_cuda_error_string(void) { return cudaGetErrorString(g_last_cuda_error); }

int mqa_num_kv_splits(int max_seq_len, int sm_count, int batch_invariant) {
    if (batch_invariant) return 1;
    long long s = max_seq_len <= 0 ? 1 : (static_cast<long long>(max_seq_len) + 511) / 512;
    const long long cap = 2LL * sm_count;
    if (cap >= 1 && s > cap) s = cap;
    if (s < 1) s = 1;
    return static_cast<int>(s);
}

size_t mla_decode_workspace_bytes(int batch, int num_heads, int kv_lora_rank, int num_kv_splits) {
    return partial_bytes(batch, num_heads, kv_lora_rank, num_kv_splits);
}

size_t gqa_paged_decode_workspace_bytes(int batch, int num_q_heads, int head_size, int num_kv_splits) {
    return partial_bytes(batch, num_q_heads, head_size, num_kv_splits);
}

mqa_status mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                      int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                      int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                      void* workspace, size_t workspace_bytes, int* device_status, void* stream) {
    return mla_decode_rows(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch, num_heads,
                           head_size, kv_lora_rank, num_blocks, page_size, max_blocks, kv_dtype, num_kv_splits,
                           workspace, workspace_bytes, device_status, stream, 1);
}

mqa_status mla_decode_fixed_splits(const void* q, const void* kv_cache, const int32_t* block_table,
                                  const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                  int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                  int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                                  void* workspace, size_t workspace_bytes, int* device_status, void* stream) {
    return mla_decode_rows(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch, num_heads,
                           head_size, kv_lora_rank, num_blocks, page_size, max_blocks, kv_dtype, num_kv_splits,
                           workspace, workspace_bytes, device_status, stream, 1, -1, true);
}

mqa_status mla_decode_multi(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                            int batch, int q_len, int num_heads, int head_size, int kv_lora_rank,
                            int num_blocks, int page_size, int max_blocks, mqa_kv_dtype kv_dtype,
                            int num_kv_splits, void* workspace, size_t workspace_bytes, int* device_status,
                            void* stream) {
    if (q_len < 1 || num_heads < 1) return MQA_ERR_INVALID_ARG;
    if (static_cast<long long>(q_len) * num_heads > 128) return MQA_ERR_UNSUPPORTED;
    return mla_decode_rows(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch,
                           q_len * num_heads, head_size, kv_lora_rank, num_blocks, page_size, max_blocks,
                           kv_dtype, num_kv_splits, workspace, workspace_bytes, device_status, stream, q_len);
}

mqa_status mla_decode_sparse(const void* q, const void* kv_cache, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* indices, float scale, float k_scale,
                             void* out, float* lse, int batch, int num_heads, int head_size,
                             int kv_lora_rank, int num_blocks, int page_size, int max_blocks, int topk,
                             mqa_kv_dtype kv_dtype, int num_kv_splits, void* workspace,
                             size_t workspace_bytes, int* device_status, void* stream) {
    if (!q || !kv_cache || !block_table || !seq_lens || !indices || !out) return MQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(indices, 4) || (lse && !aligned(lse, 4)) ||
        (device_status && !aligned(device_status, 4)))
        return MQA_ERR_INVALID_ARG;
    if (batch < 1 || num_heads < 1 || num_blocks < 1 || max_blocks < 1 || page_size < 1 || num_kv_splits < 1 ||
        topk < 1)
        return MQA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !std::isfinite(k_scale)) return MQA_ERR_INVALID_ARG;
    if (!((head_size == 576 && kv_lora_rank == 512) || (head_size == 320 && kv_lora_rank == 256)))
        return MQA_ERR_UNSUPPORTED;
    // rows are gathered one by one: any page size works
    if (kv_dtype != MQA_KV_BF16 && kv_dtype != MQA_KV_FP8_E4M3) return MQA_ERR_UNSUPPORTED;
    if (num_heads > 128 || batch > kMaxBatch || topk > (1 << 24)) return MQA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_blocks) * page_size > INT32_MAX ||
        static_cast<long long>(num_blocks) * page_size > INT32_MAX)
        return MQA_ERR_UNSUPPORTED;

    const size_t need = mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank, num_kv_splits);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MQA_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && !aligned(workspace, 16)) return MQA_ERR_INVALID_ARG;

    const int sms = sm_count_current();
    if (sms < 1) return MQA_ERR_CUDA;
    const bool fp8 = kv_dtype == MQA_KV_FP8_E4M3;
    const int groups = (num_heads + 15) / 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // The warp-MMA kernel with an index-driven gather: its plan walks the
    // topk entries of every request in "pages" of one pipeline tile (every
    // request has length topk); each 16-head group gathers the rows itself.
    mqa::MlaArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const uint8_t*>(kv_cache);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.indices = indices;
    a.topk = topk;
    a.cache_page = page_size;
    a.bt_stride = max_blocks;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    const size_t slots = static_cast<size_t>(batch) * num_kv_splits;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = need > 0 ? a.ws_o + slots * num_heads * kv_lora_rank : nullptr;
    a.status = device_status;
    const float ks = fp8 ? k_scale : 1.0f;
    a.sl2 = scale * ks * mqa::kLog2e;
    a.out_scale = ks;
    a.H = num_heads;
    a.q_len = 1;
    a.heads = num_heads;
    a.withhold = -1;
    a.num_blocks = num_blocks;
    // four-row gathers of whole rows; bf16 rows get 32 bytes of zero fill
    const int row_bytes = head_size * (fp8 ? 1 : 2);
    if (!gather_row_map(&a.tmap, kv_cache, row_bytes, static_cast<long long>(num_blocks) * page_size,
                        (row_bytes + (fp8 ? 0 : 32)) / 8))
        return MQA_ERR_CUDA;
    const int tile = mqa::mla_mma_sparse_tile(fp8);
    a.plan.batch = batch;
    a.plan.page = tile;
    a.plan.max_blocks = (topk + tile - 1) / tile;
    a.plan.fixed_len = topk;
    a.plan.per_seq = num_kv_splits == 1 ? 1 : 0;
    a.plan.units = a.plan.per_seq ? batch : balanced_units(batch, num_kv_splits, sms / groups);

    if (cudaError_t e = mqa::mla_mma_stage1(a, head_size, fp8, a.plan.units * groups, st); e != cudaSuccess)
        return cuda_fail(e);
    if (!a.plan.per_seq) {
        mqa::MergeArgs m{};
        m.ws_o = a.ws_o;
        m.ws_lse = a.ws_lse;
        m.seq_lens = seq_lens;
        m.out = a.out;
        m.lse = lse;
        m.status = device_status;
        m.out_scale = 1.0f;  // stage-1 partials already carry k_scale
        m.H = num_heads;
        m.R = kv_lora_rank;
        m.plan = a.plan;
        if (cudaError_t e = mqa::lse_merge(m, st); e != cudaSuccess) return cuda_fail(e);
    }
    return MQA_OK;
}

mqa_status mqa_lse_merge(const void* shard_out, const float* shard_lse, void* out, float* lse, int num_shards,
                         long long rows, int head_dim, void* stream) {
    if (!shard_out || !shard_lse || !out) return MQA_ERR_INVALID_ARG;
    if (!aligned(shard_out, 16) || !aligned(shard_lse, 16) || !aligned(out, 16) || (lse && !aligned(lse, 16)))
        return MQA_ERR_INVALID_ARG;
    if (num_shards < 1 || rows < 1 || head_dim < 8 || head_dim > 4096 || head_dim % 8 != 0)
        return MQA_ERR_INVALID_ARG;
    // grid of rows / 4 blocks
    if (rows > 4LL * 0x7fffffffLL) return MQA_ERR_UNSUPPORTED;
    if (cudaError_t e = mqa::shard_merge(static_cast<const __nv_bfloat16*>(shard_out), shard_lse,
                                         static_cast<__nv_bfloat16*>(out), lse, num_shards, rows, head_dim,
                                         static_cast<cudaStream_t>(stream));
        e != cudaSuccess)
        return cuda_fail(e);
    return MQA_OK;
}

mqa_status mqa_dcp_scale_shard(const void* shard_out, const float* gathered_lse, void* scaled, float* lse,
                               int num_ranks, int rank, int batch, int num_heads, int head_dim, int scaled_fp32,
                               void* stream) {
    if (!shard_out || !gathered_lse || !scaled) return MQA_ERR_INVALID_ARG;
    if (!aligned(shard_out, 16) || !aligned(gathered_lse, 16) || !aligned(scaled, 16) || (lse && !aligned(lse, 16)))
        return MQA_ERR_INVALID_ARG;
    if (num_ranks < 1 || rank < 0 || rank >= num_ranks || batch < 1 || num_heads < 1 ||
        num_heads % num_ranks != 0 || head_dim < 8 || head_dim > 4096 || head_dim % 8 != 0)
        return MQA_ERR_INVALID_ARG;
    // grid of batch * num_heads / 4 blocks
    if (static_cast<long long>(batch) * num_heads > 4LL * 0x7fffffffLL) return MQA_ERR_UNSUPPORTED;
    if (cudaError_t e = mqa::dcp_scale(static_cast<const __nv_bfloat16*>(shard_out), gathered_lse, scaled, lse,
                                       num_ranks, rank, batch, num_heads, head_dim, scaled_fp32 != 0,
                                       static_cast<cudaStream_t>(stream));
        e != cudaSuccess)
        return cuda_fail(e);
    return MQA_OK;
}

}  // extern "C"

// gqa_paged_decode; withhold >= 0 (bf16 caches only) is the test hook of the
// bounded waits (see mqa_test_gqa_withheld_arrive).
static mqa_status gqa_decode_impl(const void* q, const void* kv_cache, const int32_t* block_table,
                                  const int32_t* seq_lens, float scale, float k_scale, float v_scale,
                                  void* out, float* lse, int batch, int num_q_heads, int num_kv_heads,
                                  int head_size, int num_blocks, int page_size, int max_blocks,
                                  mqa_kv_dtype kv_dtype, int num_kv_splits, void* workspace,
                                  size_t workspace_bytes, int* device_status, void* stream, int withhold) {
    if (!q || !kv_cache || !block_table || !seq_lens || !out) return MQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) || (device_status && !aligned(device_status, 4)))
        return MQA_ERR_INVALID_ARG;
    if (batch < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_blocks < 1 || max_blocks < 1 ||
        page_size < 1 || num_kv_splits < 1)
        return MQA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return MQA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return MQA_ERR_INVALID_ARG;
    if (head_size != 64 && head_size != 128) return MQA_ERR_UNSUPPORTED;
    if (num_kv_heads > 8 || num_q_heads / num_kv_heads > 16) return MQA_ERR_UNSUPPORTED;
    if (page_size % 16 != 0) return MQA_ERR_UNSUPPORTED;
    if (kv_dtype != MQA_KV_BF16 && kv_dtype != MQA_KV_FP8_E4M3 && kv_dtype != MQA_KV_FP8_E4M3_PER_TOKEN_HEAD &&
        kv_dtype != MQA_KV_INT8_PER_TOKEN_HEAD && kv_dtype != MQA_KV_INT4_PER_TOKEN_HEAD)
        return MQA_ERR_UNSUPPORTED;
    if (kv_dtype == MQA_KV_FP8_E4M3 && (!std::isfinite(k_scale) || !std::isfinite(v_scale)))
        return MQA_ERR_INVALID_ARG;
    if (batch > kMaxBatch) return MQA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_blocks) * page_size > INT32_MAX ||
        static_cast<long long>(num_blocks) * page_size > INT32_MAX)
        return MQA_ERR_UNSUPPORTED;

    const size_t need = gqa_paged_decode_workspace_bytes(batch, num_q_heads, head_size, num_kv_splits);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MQA_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && !aligned(workspace, 16)) return MQA_ERR_INVALID_ARG;

    const int sms = sm_count_current();
    if (sms < 1) return MQA_ERR_CUDA;

    mqa::GqaArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const uint8_t*>(kv_cache);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    const size_t slots = static_cast<size_t>(batch) * num_kv_splits;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = need > 0 ? a.ws_o + slots * num_q_heads * head_size : nullptr;
    a.status = device_status;
    const bool per_tensor_fp8 = kv_dtype == MQA_KV_FP8_E4M3;
    a.sl2 = scale * (per_tensor_fp8 ? k_scale : 1.0f) * mqa::kLog2e;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.num_blocks = num_blocks;
    a.plan.batch = batch;
    a.plan.page = page_size;
    a.plan.max_blocks = max_blocks;
    a.plan.per_seq = num_kv_splits == 1 ? 1 : 0;
    const int resident =
        kv_dtype == MQA_KV_BF16 ? sms : sms * mqa::gqa_q8_ctas_per_sm(num_q_heads / num_kv_heads);
    a.plan.units = a.plan.per_seq ? batch : balanced_units(batch, num_kv_splits, resident);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (withhold >= 0 && kv_dtype != MQA_KV_BF16) return MQA_ERR_UNSUPPORTED;
    if (kv_dtype == MQA_KV_BF16) {
        const cudaError_t e = withhold >= 0
                                  ? mqa::gqa_mma_stage1_withheld(a, head_size, a.plan.units, withhold, st)
                                  : mqa::gqa_mma_stage1(a, head_size, a.plan.units, st);
        if (e != cudaSuccess) return cuda_fail(e);
    } else {
        // 8-bit codes: widened per KV head in shared memory; per-tensor fp8
        // folds k_scale into the softmax scale and v_scale into the output
        const float out_scale = per_tensor_fp8 ? v_scale : 1.0f;
        if (cudaError_t e = mqa::gqa_q8_stage1(a, out_scale, head_size, static_cast<int>(kv_dtype), a.plan.units, st);
            e != cudaSuccess)
            return cuda_fail(e);
    }
    if (!a.plan.per_seq) {
        mqa::MergeArgs m{};
        m.ws_o = a.ws_o;
        m.ws_lse = a.ws_lse;
        m.seq_lens = seq_lens;
        m.out = a.out;
        m.lse = lse;
        m.status = device_status;
        m.out_scale = 1.0f;
        m.H = num_q_heads;
        m.R = head_size;
        m.plan = a.plan;
        if (cudaError_t e = mqa::lse_merge(m, st); e != cudaSuccess) return cuda_fail(e);
    }
    return MQA_OK;
}

extern "C" {

mqa_status gqa_paged_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, float k_scale, float v_scale,
                            void* out, float* lse, int batch, int num_q_heads, int num_kv_heads,
                            int head_size, int num_blocks, int page_size, int max_blocks,
                            mqa_kv_dtype kv_dtype, int num_kv_splits, void* workspace,
                            size_t workspace_bytes, int* device_status, void* stream) {
    return gqa_decode_impl(q, kv_cache, block_table, seq_lens, scale, k_scale, v_scale, out, lse, batch,
                           num_q_heads, num_kv_heads, head_size, num_blocks, page_size, max_blocks, kv_dtype,
                           num_kv_splits, workspace, workspace_bytes, device_status, stream, -1);
}

mqa_status mqa_test_mla_withheld_arrive(const void* q, const void* kv_cache, const int32_t* block_table,
                                        const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                        int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                        int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                                        void* workspace, size_t workspace_bytes, int* device_status, void* stream,
                                        int withhold_unit) {
    if (!test_hooks_enabled()) return MQA_ERR_UNSUPPORTED;
    if (withhold_unit < 0) return MQA_ERR_INVALID_ARG;
    return mla_decode_rows(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch, num_heads,
                           head_size, kv_lora_rank, num_blocks, page_size, max_blocks, kv_dtype, num_kv_splits,
                           workspace, workspace_bytes, device_status, stream, 1, withhold_unit);
}

mqa_status mqa_test_mla_warp_gives_up(const void* q, const void* kv_cache, const int32_t* block_table,
                                      const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                      int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                      int page_size, int max_blocks, int num_kv_splits, void* workspace,
                                      size_t workspace_bytes, int* device_status, void* stream, int unit,
                                      int warp) {
    if (!test_hooks_enabled()) return MQA_ERR_UNSUPPORTED;
    // the tensor-core kernel's softmax warps are warps 2..9 of each CTA
    if (unit < 0 || warp < 2 || warp > 9 || num_heads <= 32) return MQA_ERR_INVALID_ARG;
    return mla_decode_rows(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch, num_heads,
                           head_size, kv_lora_rank, num_blocks, page_size, max_blocks, MQA_KV_FP8_E4M3,
                           num_kv_splits, workspace, workspace_bytes, device_status, stream, 1, -1, false,
                           unit * 16 + warp);
}

mqa_status mqa_test_gqa_withheld_arrive(const void* q, const void* kv_cache, const int32_t* block_table,
                                        const int32_t* seq_lens, float scale, void* out, float* lse, int batch,
                                        int num_q_heads, int num_kv_heads, int head_size, int num_blocks,
                                        int page_size, int max_blocks, int num_kv_splits, void* workspace,
                                        size_t workspace_bytes, int* device_status, void* stream,
                                        int withhold_unit) {
    if (!test_hooks_enabled()) return MQA_ERR_UNSUPPORTED;
    if (withhold_unit < 0) return MQA_ERR_INVALID_ARG;
    return gqa_decode_impl(q, kv_cache, block_table, seq_lens, scale, 1.0f, 1.0f, out, lse, batch, num_q_heads,
                           num_kv_heads, head_size, num_blocks, page_size, max_blocks, MQA_KV_BF16, num_kv_splits,
                           workspace, workspace_bytes, device_status, stream, withhold_unit);
}

}  // extern "C"
