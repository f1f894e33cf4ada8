// Decode context parallelism (DCP): which pages of a request each rank holds
// (host code), and the local step of the merge that all-gathers the shards'
// lse and reduce-scatters their outputs (one kernel).
//
// The pages name the merge of DCP shards (cp_lse_ag_out_rs) and say that it
// rests on the natural-log lse the decode returns ("Triton と MLA" page,
// 設計動機); the merge itself is the LogSumExp combination of partial results
// (tutorial page lshu.cn/news/265860, §12).  Page-aligned placement is this
// library's reading: a rank's share of a request is then an ordinary paged
// sequence, so the decode kernels run on it unchanged.
#include <cstdint>

#include "common.cuh"
#include "dcp.cuh"

namespace {

bool layout_ok(int layout) { return layout == MQA_DCP_ROUND_ROBIN || layout == MQA_DCP_CONTIGUOUS; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

int mqa_dcp_shard_max_blocks(int max_blocks, int num_ranks) {
    if (max_blocks < 1 || num_ranks < 1) return -1;
    return ceil_div(max_blocks, num_ranks);
}

mqa_status mqa_dcp_shard(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                         int page_size, int num_ranks, int rank, mqa_dcp_layout layout,
                         int32_t* shard_block_table, int shard_max_blocks, int32_t* shard_seq_lens) {
    if (!block_table || !seq_lens || !shard_block_table || !shard_seq_lens) return MQA_ERR_INVALID_ARG;
    if (batch < 1 || max_blocks < 1 || page_size < 1 || num_ranks < 1 || rank < 0 || rank >= num_ranks)
        return MQA_ERR_INVALID_ARG;
    if (!layout_ok(layout) || shard_max_blocks < mqa_dcp_shard_max_blocks(max_blocks, num_ranks))
        return MQA_ERR_INVALID_ARG;
    const long long cap = static_cast<long long>(max_blocks) * page_size;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > cap) return MQA_ERR_INVALID_ARG;

    for (int b = 0; b < batch; ++b) {
        const int n = seq_lens[b];
        const int pages = static_cast<int>((static_cast<long long>(n) + page_size - 1) / page_size);
        // the rank's pages of the request: j0, j0 + step, ... below j_end
        int j0, step, j_end;
        if (layout == MQA_DCP_ROUND_ROBIN) {
            j0 = rank;
            step = num_ranks;
            j_end = pages;
        } else {
            const int run = ceil_div(pages, num_ranks);
            j0 = rank * run;
            step = 1;
            j_end = j0 + run < pages ? j0 + run : pages;
        }
        const int32_t* src = block_table + static_cast<long long>(b) * max_blocks;
        int32_t* dst = shard_block_table + static_cast<long long>(b) * shard_max_blocks;
        int k = 0;
        long long tokens = 0;
        for (int j = j0; j < j_end; j += step) {
            dst[k++] = src[j];
            const long long left = n - static_cast<long long>(j) * page_size;
            tokens += left < page_size ? left : page_size;
        }
        for (; k < shard_max_blocks; ++k) dst[k] = -1;
        shard_seq_lens[b] = static_cast<int32_t>(tokens);
    }
    return MQA_OK;
}

mqa_status mqa_dcp_locate(int pos, int seq_len, int page_size, int num_ranks, mqa_dcp_layout layout, int* rank,
                          int* shard_pos) {
    if (!rank || !shard_pos || page_size < 1 || num_ranks < 1 || !layout_ok(layout)) return MQA_ERR_INVALID_ARG;
    if (pos < 0 || pos >= seq_len) return MQA_ERR_INVALID_ARG;
    const int j = pos / page_size, off = pos % page_size;
    if (layout == MQA_DCP_ROUND_ROBIN) {
        *rank = j % num_ranks;
        *shard_pos = (j / num_ranks) * page_size + off;
    } else {
        const int pages = static_cast<int>((static_cast<long long>(seq_len) + page_size - 1) / page_size);
        const int run = ceil_div(pages, num_ranks);
        *rank = j / run;
        *shard_pos = (j - *rank * run) * page_size + off;
    }
    return MQA_OK;
}

}  // extern "C"

namespace mqa {

namespace {

constexpr int kWarps = 4;  // warps per block, one (request, head) row each

// Row (b, h) of this rank's shard output, scaled by its merge weight, into
// chunk h / (H / G) of the reduce-scatter input.  The lanes first take the
// ranks' lse values 32 at a time (max and weight sum by warp reductions), then
// own 8-column groups of the row.
template <bool F32>
__global__ void __launch_bounds__(32 * kWarps)
    dcp_scale_kernel(const __nv_bfloat16* __restrict__ in, const float* __restrict__ lses, void* __restrict__ dst,
                     float* __restrict__ lse, int G, int rank, int B, int H, int D) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(B) * H;
    const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= rows) return;

    float m = -INFINITY;
    for (int g = lane; g < G; g += 32) m = fmaxf(m, __ldg(lses + g * rows + row));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float wsum = 0.f;
    if (m != -INFINITY)
        for (int g = lane; g < G; g += 32) {
            const float l = __ldg(lses + g * rows + row);
            wsum += l == -INFINITY ? 0.f : __expf(l - m);
        }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float own = __ldg(lses + rank * rows + row);
    // weight of this rank's shard; 0 for an empty shard and for a row that no
    // rank holds a token of (whose shard outputs are not read)
    const float w = own == -INFINITY ? 0.f : __expf(own - m) / wsum;

    const int b = static_cast<int>(row / H), h = static_cast<int>(row % H);
    const int hc = H / G, c = h / hc;
    const long long drow = (static_cast<long long>(c) * B + b) * hc + (h - c * hc);
    const __nv_bfloat16* irow = in + row * D;
    for (int col = 8 * lane; col < D; col += 256) {
        const uint4 v = w == 0.f ? make_uint4(0u, 0u, 0u, 0u) : __ldg(reinterpret_cast<const uint4*>(irow + col));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
            f[2 * i] = p.x * w;
            f[2 * i + 1] = p.y * w;
        }
        if constexpr (F32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(dst) + drow * D + col);
            o[0] = make_float4(f[0], f[1], f[2], f[3]);
            o[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + drow * D + col) =
                make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                           pack_bf16x2(f[6], f[7]));
        }
    }
    if (lse && lane == 0) lse[row] = m == -INFINITY ? -INFINITY : m + __logf(wsum);
}

}  // namespace

cudaError_t dcp_scale(const __nv_bfloat16* in, const float* lses, void* dst, float* lse, int G, int rank, int B,
                      int H, int D, bool f32, cudaStream_t stream) {
    const long long rows = static_cast<long long>(B) * H;
    const unsigned blocks = static_cast<unsigned>((rows + kWarps - 1) / kWarps);
    if (f32)
        dcp_scale_kernel<true><<<blocks, 32 * kWarps, 0, stream>>>(in, lses, dst, lse, G, rank, B, H, D);
    else
        dcp_scale_kernel<false><<<blocks, 32 * kWarps, 0, stream>>>(in, lses, dst, lse, G, rank, B, H, D);
    return cudaGetLastError();
}

}  // namespace mqa
