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
//
// One thread block per (request, head).  It is launched as a programmatic
// dependent of stage 1: the page prefix (from seq_lens only) is computed
// before waiting for stage 1 to finish, the partials after.
#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"

namespace mqa {

constexpr int kMergeThreads = 128;

__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const MergeArgs a) {
    const int b = blockIdx.x;
    const int h = blockIdx.y;
    const int P = a.plan.page;
    __shared__ int red_i[2][kMergeThreads / 32];
    __shared__ float red_f[kMergeThreads / 32];
    __shared__ float s_w[kMaxMergeUnits];

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
        red_i[0][threadIdx.x >> 5] = before;
        red_i[1][threadIdx.x >> 5] = total;
    }
    __syncthreads();
    before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) {
        before += red_i[0][w];
        total += red_i[1][w];
    }
    const int n_b = (clamp_len(a.seq_lens[b], a.plan.max_blocks, P, nullptr) + P - 1) / P;
    const int R = a.R;
    const long long orow = (static_cast<long long>(b) * a.H + h) * R;

    int gf = 0, gl = 0;
    if (n_b > 0) {
        gf = unit_of_page(a.plan.units, total, before);
        gl = unit_of_page(a.plan.units, total, before + n_b - 1);
        if (gf == gl) return;  // one unit covered the request and wrote it directly
    }
    pdl_wait();  // stage-1 partials (and the outputs' previous readers) are done
    if (n_b == 0) {  // empty request: out = 0, lse = -inf
        for (int i = threadIdx.x; i < R / 2; i += kMergeThreads)
            reinterpret_cast<uint32_t*>(a.out + orow)[i] = 0u;
        if (a.lse && threadIdx.x == 0) a.lse[static_cast<long long>(b) * a.H + h] = -INFINITY;
        return;
    }

    // Units between gf and gl overlap request b unless their page range is
    // empty (more units than pages); empty units wrote no partial.
    const int np = gl - gf + 1;
    float m = -INFINITY;
    for (int i = threadIdx.x; i < np; i += kMergeThreads) {
        const int g = gf + i;
        const bool has = static_cast<long long>(g) * total / a.plan.units <
                         static_cast<long long>(g + 1) * total / a.plan.units;
        const float l = has ? a.ws_lse[static_cast<long long>(g + b) * a.H + h] : -INFINITY;
        s_w[i] = l;
        m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red_f[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red_f[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) m = fmaxf(m, red_f[w]);
    __syncthreads();
    float wsum = 0.f;
    for (int i = threadIdx.x; i < np; i += kMergeThreads) {
        const float l = s_w[i];
        const float w = (l == -INFINITY || m == -INFINITY) ? 0.f : __expf(l - m);
        s_w[i] = w;
        wsum += w;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    if ((threadIdx.x & 31) == 0) red_f[threadIdx.x >> 5] = wsum;
    __syncthreads();
    wsum = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) wsum += red_f[w];
    const float inv = wsum > 0.f ? a.out_scale / wsum : 0.f;

    for (int c4 = threadIdx.x; c4 < R / 4; c4 += kMergeThreads) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* base = a.ws_o + (static_cast<long long>(gf + b) * a.H + h) * R + 4 * c4;
        const long long step = static_cast<long long>(a.H) * R;
        // up to 24 partial rows in flight per thread (one round for most
        // requests); a segment with weight 0 (empty, never written)
        // contributes by selection, not by product
        constexpr int kBatch = 24;
        for (int i0 = 0; i0 < np; i0 += kBatch) {
            float4 v[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                v[k] = i0 + k < np ? __ldcs(reinterpret_cast<const float4*>(base + (i0 + k) * step))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const float w = i0 + k < np ? s_w[i0 + k] : 0.f;
                if (w != 0.f) {
                    acc.x += w * v[k].x;
                    acc.y += w * v[k].y;
                    acc.z += w * v[k].z;
                    acc.w += w * v[k].w;
                }
            }
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(a.out + orow + 4 * c4) = packed;
    }
    if (threadIdx.x == 0 && a.lse)
        a.lse[static_cast<long long>(b) * a.H + h] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

cudaError_t lse_merge(const MergeArgs& a, cudaStream_t stream) {
    cudaError_t e = launch_with_pdl(lse_merge_kernel, dim3(a.plan.batch, a.H), dim3(kMergeThreads), 0,
                                    stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mqa
