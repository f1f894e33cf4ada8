// Stage 2: merge the KV-segment partials of each request by LogSumExp.
//
// Each partial holds O_s normalised by its own softmax sum and its natural-log
// LSE lse_s = m_s + ln l_s.  With m = max_s lse_s and w_s = exp(lse_s - m):
//   out = sum_s w_s O_s / sum_s w_s,   lse = m + ln sum_s w_s,
// which is the tutorial page's §12 merge (m = max m_s, l = sum e^{m_s-m} l_s,
// O = sum e^{m_s-m} O_s / l) rewritten for normalised partials
// (attention-kernel tutorial page, lshu.cn/news/265860).  Segments with
// lse_s = -inf get weight 0.  The merge order is fixed (ascending segment), so
// the result is reproducible run to run.
#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"

namespace mqa {

constexpr int kMergeThreads = 128;
constexpr int kMergeHeads = 4;

__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const MergeArgs a) {
    const int b = blockIdx.x;
    const int hb = blockIdx.y * kMergeHeads;
    const int P = a.plan.page;
    __shared__ int red[2][kMergeThreads / 32];

    // Page offset of request b and total page count, recomputed exactly as the
    // stage-1 kernel's prefix (same clamping).
    int before = 0, total = 0;
    for (int i = threadIdx.x; i < a.plan.batch; i += kMergeThreads) {
        const int n = clamp_len(a.seq_lens[i], a.plan.max_blocks, P, nullptr);
        const int pages = (n + P - 1) / P;
        total += pages;
        if (i < b) before += pages;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = before;
        red[1][threadIdx.x >> 5] = total;
    }
    __syncthreads();
    before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) {
        before += red[0][w];
        total += red[1][w];
    }
    const int n_b = (clamp_len(a.seq_lens[b], a.plan.max_blocks, P, nullptr) + P - 1) / P;
    const int nh = min(kMergeHeads, a.H - hb);
    const int R = a.R;

    if (n_b == 0) {  // empty request: out = 0, lse = -inf
        for (int i = threadIdx.x; i < nh * R; i += kMergeThreads)
            a.out[(static_cast<long long>(b) * a.H + hb) * R + i] = __float2bfloat16(0.f);
        if (a.lse && threadIdx.x < nh) a.lse[static_cast<long long>(b) * a.H + hb + threadIdx.x] = -INFINITY;
        return;
    }
    const int gf = unit_of_page(a.plan.units, total, before);
    const int gl = unit_of_page(a.plan.units, total, before + n_b - 1);
    if (gf == gl) return;  // one unit covered the request and wrote it directly

    // Units between gf and gl overlap request b unless their page range is
    // empty (more units than pages); empty units wrote no partial.
    auto has_pages = [&](int g) {
        return static_cast<long long>(g) * total / a.plan.units <
               static_cast<long long>(g + 1) * total / a.plan.units;
    };
    for (int hh = 0; hh < nh; ++hh) {
        const int h = hb + hh;
        float m = -INFINITY;
        for (int g = gf; g <= gl; ++g)
            if (has_pages(g)) m = fmaxf(m, a.ws_lse[static_cast<long long>(g + b) * a.H + h]);
        float wsum = 0.f;
        for (int g = gf; g <= gl; ++g) {
            if (!has_pages(g)) continue;
            const float l = a.ws_lse[static_cast<long long>(g + b) * a.H + h];
            wsum += l == -INFINITY ? 0.f : __expf(l - m);
        }
        const float inv = wsum > 0.f ? a.out_scale / wsum : 0.f;
        for (int c4 = threadIdx.x; c4 < R / 4; c4 += kMergeThreads) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int g = gf; g <= gl; ++g) {
                if (!has_pages(g)) continue;
                const float l = a.ws_lse[static_cast<long long>(g + b) * a.H + h];
                const float w = l == -INFINITY ? 0.f : __expf(l - m);
                const float4 v = *reinterpret_cast<const float4*>(
                    a.ws_o + (static_cast<long long>(g + b) * a.H + h) * R + 4 * c4);
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
            uint2 packed;
            packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(a.out + (static_cast<long long>(b) * a.H + h) * R + 4 * c4) = packed;
        }
        if (threadIdx.x == 0 && a.lse)
            a.lse[static_cast<long long>(b) * a.H + h] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
    }
}

cudaError_t lse_merge(const MergeArgs& a, cudaStream_t stream) {
    dim3 grid(a.plan.batch, (a.H + kMergeHeads - 1) / kMergeHeads);
    lse_merge_kernel<<<grid, kMergeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace mqa
