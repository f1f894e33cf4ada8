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
// One warp per (request, head) row, or per 128-column quarter of a row when
// the requests are summed from many partials (long sequences over many
// units: the host picks by the mean number of partials per request), four
// warps per block.  The lse maximum and the weight sum are warp reductions
// over the partials; lane l owns the float4 column groups l, l + 32, ... of
// its columns, and the loads of several partials are in flight together.  It
// is launched as a programmatic dependent of stage 1 and kept small (no
// shared memory) so that its blocks fit beside the stage-1 CTAs and wait
// there: the page prefix (from seq_lens only) is computed before waiting for
// stage 1 to finish, the partials after.
#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"

namespace mqa {

constexpr int kMergeWarps = 4;  // warps per block

// G float4 column groups per lane: a warp covers 128 G columns of a row, with
// the loads of 8 (G = 1) or 2 (G = 4) partials in flight together.  The
// row-per-warp form is held to 80 registers so that its blocks fit beside
// the stage-1 CTAs while they wait.
template <int G>
__global__ void __launch_bounds__(32 * kMergeWarps, G == 4 ? 6 : 1) lse_merge_kernel(const MergeArgs a) {
    constexpr int kMergeCols = 128 * G;
    constexpr int kMergeBatch = G == 1 ? 8 : 2;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int nq = (a.R + kMergeCols - 1) / kMergeCols;  // warps per row
    const int item = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int h = item / nq, q = item - h * nq;
    const int P = a.plan.page;
    if (h >= a.H) return;

    // Page offset of request b and total page count, recomputed exactly as the
    // stage-1 kernel's prefix (same clamping).
    int before = 0, total = 0;
    for (int i = lane; i < a.plan.batch; i += 32) {
        const int n = plan_len(a.plan, a.seq_lens, i, nullptr);
        const int pages = (n + P - 1) / P;
        total += pages;
        if (i < b) before += pages;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    const int n_b = (plan_len(a.plan, a.seq_lens, b, nullptr) + P - 1) / P;
    const int R = a.R;
    const long long orow = (static_cast<long long>(b) * a.H + h) * R;
    const int col = q * kMergeCols + 4 * lane;  // first column of the lane's group k: col + 128 k

    // the request's partials: np consecutive slots from slot0
    const int S = a.plan.fixed_splits;
    int gf = 0, np = 0, slot0 = 0;
    if (S > 0) {
        // fixed-split mode: ranges of L pages, range s in slot b S + s; range
        // 0 wrote the output directly when it held the whole request (or the
        // request has no page)
        if (n_b == 0) return;
        const int L = (n_b + S - 1) / S;
        if (L >= n_b) return;
        np = (n_b + L - 1) / L;
        slot0 = b * S;
    } else if (n_b > 0) {
        // balanced mode: a page's position is its page index plus piece_cost
        // per request up to and including its own (0: plain page balance)
        const int c = a.plan.piece_cost;
        total += c * a.plan.batch;
        before += c * (b + 1);
        gf = unit_of_page(a.plan.units, total, before);
        const int gl = unit_of_page(a.plan.units, total, before + n_b - 1);
        if (gf == gl) return;  // one unit covered the request and wrote it directly
        np = gl - gf + 1;
        slot0 = gf + b;
    }
    pdl_wait();  // stage-1 partials (and the outputs' previous readers) are done
    if (n_b == 0) {  // empty request: out = 0, lse = -inf
#pragma unroll
        for (int k = 0; k < G; ++k)
            if (col + 128 * k < R) *reinterpret_cast<uint2*>(a.out + orow + col + 128 * k) = make_uint2(0u, 0u);
        if (a.lse && q == 0 && lane == 0) a.lse[static_cast<long long>(b) * a.H + h] = -INFINITY;
        return;
    }

    // Balanced mode: units between gf and gl overlap request b unless their
    // page range is empty (more units than pages); empty units wrote no
    // partial.  Fixed-split mode: every one of the np ranges holds pages.
    auto unit_lse = [&](int i) {
        const int g = gf + i;
        const bool has = S > 0 || static_cast<long long>(g) * total / a.plan.units <
                                      static_cast<long long>(g + 1) * total / a.plan.units;
        return has ? a.ws_lse[static_cast<long long>(slot0 + i) * a.H + h] : -INFINITY;
    };
    float m = -INFINITY;
    for (int i = lane; i < np; i += 32) m = fmaxf(m, unit_lse(i));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float4 acc[G];
#pragma unroll
    for (int k = 0; k < G; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* base = a.ws_o + (static_cast<long long>(slot0) * a.H + h) * R + col;
    const long long step = static_cast<long long>(a.H) * R;
    float wsum = 0.f;
    for (int j0 = 0; j0 < np; j0 += 32) {
        // weight of unit j0 + lane; a unit with weight 0 (empty, never
        // written) contributes by selection, not by product
        const float l = j0 + lane < np ? unit_lse(j0 + lane) : -INFINITY;
        const float wl = (l == -INFINITY || m == -INFINITY) ? 0.f : __expf(l - m);
        wsum += wl;
        const int nu = min(32, np - j0);
        for (int i0 = 0; i0 < nu; i0 += kMergeBatch) {
            float4 v[kMergeBatch][G];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
                for (int k = 0; k < G; ++k)
                    v[u][k] = (i0 + u < nu && col + 128 * k < R)
                                  ? __ldcs(reinterpret_cast<const float4*>(base + (j0 + i0 + u) * step + 128 * k))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const float w = __shfl_sync(0xffffffffu, wl, (i0 + u) & 31);
                if (i0 + u < nu && w != 0.f) {
#pragma unroll
                    for (int k = 0; k < G; ++k) {
                        acc[k].x += w * v[u][k].x;
                        acc[k].y += w * v[u][k].y;
                        acc[k].z += w * v[u][k].z;
                        acc[k].w += w * v[u][k].w;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? a.out_scale / wsum : 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) {
        if (col + 128 * k >= R) break;
        uint2 packed;
        packed.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
        packed.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
        *reinterpret_cast<uint2*>(a.out + orow + col + 128 * k) = packed;
    }
    if (q == 0 && lane == 0 && a.lse)
        a.lse[static_cast<long long>(b) * a.H + h] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

template <int G>
static cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    const int items = a.H * ((a.R + 128 * G - 1) / (128 * G));  // warps per request
    cudaError_t e = launch_with_pdl(lse_merge_kernel<G>, dim3((items + kMergeWarps - 1) / kMergeWarps, a.plan.batch),
                                    dim3(32 * kMergeWarps), 0, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t lse_merge(const MergeArgs& a, cudaStream_t stream) {
    // a request is summed from about (units + batch) / batch partials: with
    // more than 4 on average, a warp per 128 columns (more warps, fewer
    // loads each) beats a warp per row
    const bool many = a.plan.units > 3 * a.plan.batch;
    return many ? launch_merge<1>(a, stream) : launch_merge<4>(a, stream);
}

}  // namespace mqa
