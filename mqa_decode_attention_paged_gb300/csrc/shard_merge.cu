// Merge of sequence-shard results (decode context parallelism).
//
// When a request's KV pages are spread over G ranks, each rank decodes its
// shard and returns a normalised output O_g (bf16) with its natural-log LSE
// lse_g; after the caller has gathered the G results, this kernel merges
// them: with m = max_g lse_g and w_g = e^{lse_g - m},
//   out = sum_g w_g O_g / sum_g w_g,   lse = m + ln sum_g w_g
// (the tutorial page's §12 merge, lshu.cn/news/265860, written for normalised
// partials; the "Triton と MLA" page, 設計動機, names the same merge of DCP
// shards, cp_lse_ag_out_rs).  A shard with lse_g = -inf holds no token: it
// gets weight 0 by selection and its output is never read.
//
// One warp per (request, head) row.  The lanes take the shards' lse values 32
// at a time (max and weight sum by warp reductions), then own 8-column groups
// of the row (16-byte bf16 loads, fp32 sums); the loads of four shards are in
// flight together.  Fixed shard order: reproducible run to run.
#include "common.cuh"
#include "shard_merge.cuh"

namespace mqa {

namespace {

constexpr int kWarps = 4;       // warps per block
constexpr int kInFlight = 4;    // shards whose loads are issued together

__device__ __forceinline__ void add8(float (&acc)[8], uint4 v, float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
        acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
    }
}

__global__ void __launch_bounds__(32 * kWarps) shard_merge_kernel(const __nv_bfloat16* __restrict__ outs,
                                                                  const float* __restrict__ lses,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ lse, int G, long long rows,
                                                                  int R) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= rows) return;

    // m = max_g lse_g, then sum_g e^{lse_g - m}
    float m = -INFINITY;
    for (int g = lane; g < G; g += 32) m = fmaxf(m, __ldg(lses + g * rows + row));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __nv_bfloat16* orow = out + row * R;
    if (m == -INFINITY) {  // no shard holds a token: out = 0, lse = -inf
        for (int c = 8 * lane; c < R; c += 256) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
        if (lse && lane == 0) lse[row] = -INFINITY;
        return;
    }
    float wsum = 0.f;
    for (int g = lane; g < G; g += 32) {
        const float l = __ldg(lses + g * rows + row);
        wsum += l == -INFINITY ? 0.f : __expf(l - m);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = 1.f / wsum;

    for (int c = 8 * lane; c < R; c += 256) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int g0 = 0; g0 < G; g0 += kInFlight) {
            uint4 v[kInFlight];
            float w[kInFlight];
#pragma unroll
            for (int k = 0; k < kInFlight; ++k) {
                const int g = g0 + k;
                const float l = g < G ? __ldg(lses + g * rows + row) : -INFINITY;
                w[k] = l == -INFINITY ? 0.f : __expf(l - m);
                v[k] = l == -INFINITY ? make_uint4(0u, 0u, 0u, 0u)
                                      : __ldg(reinterpret_cast<const uint4*>(outs + (g * rows + row) * R + c));
            }
#pragma unroll
            for (int k = 0; k < kInFlight; ++k)
                if (w[k] != 0.f) add8(acc, v[k], w[k]);
        }
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) ow[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
        *reinterpret_cast<uint4*>(orow + c) = o;
    }
    if (lse && lane == 0) lse[row] = m + __logf(wsum);
}

}  // namespace

cudaError_t shard_merge(const __nv_bfloat16* outs, const float* lses, __nv_bfloat16* out, float* lse, int G,
                        long long rows, int R, cudaStream_t stream) {
    const long long blocks = (rows + kWarps - 1) / kWarps;
    shard_merge_kernel<<<static_cast<unsigned>(blocks), 32 * kWarps, 0, stream>>>(outs, lses, out, lse, G, rows, R);
    return cudaGetLastError();
}

}  // namespace mqa
