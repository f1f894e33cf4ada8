// MLA decode, stage 1, warp-level tensor-core path (any head count, 16 heads
// per thread block).
//
// One thread block = 8 consumer warps + 1 producer warp, persistent over a
// work unit (see plan.cuh).  The producer walks the block table and stages
// 64-token tiles of latent rows [kv_c | k_pe] into shared memory with
// per-row bulk copies (TMA engine), zero-filling rows past the sequence end.
// The same staged tile serves as K (all D columns) and V (first R columns),
// the MQA view of MLA ("Triton と MLA" page, vllm-arch-zh
// ja/attention/triton-mla, section データフロー).
//
// Per tile the consumers compute
//   S = Q K^T  (16 heads x 64 tokens; 8 warps = 2 token halves x 4 quarters
//               of the head dimension, partial sums reduced through smem),
//   online softmax per head (tutorial page lshu.cn/news/265860, §7: running
//   max m, running sum l, rescale alpha = 2^(m_old - m_new) in base 2 with
//   log2(e) folded into the scale),
//   O = alpha O + P V (each warp owns R/8 output columns).
// fp8-e4m3 tiles are first widened to bf16 in shared memory (exact); k_scale
// is folded into the logit scale and into the output.
#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"
#include <cuda_fp8.h>

namespace mqa {

template <int D, int R, bool FP8>
struct MlaMmaCfg {
    static constexpr int kHeads = 16;
    static constexpr int kTile = 64;
    static constexpr int kConsumerWarps = 8;
    static constexpr int kConsumers = 32 * kConsumerWarps;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kRowBytes = D * (FP8 ? 1 : 2);      // one cache row in global memory
    static constexpr int kStageStride = kRowBytes + 16;      // padded row stride of a stage
    static constexpr int kOpStride = D * 2 + 16;              // bf16 operand row stride (bytes)
    static constexpr int kStages = (D == 576) ? 2 : (FP8 ? 4 : 3);
    static constexpr int kKSteps = D / 16;
    static constexpr int kKq = kKSteps / 4;                   // k-steps per head-dim quarter
    static constexpr int kColsPerWarp = R / kConsumerWarps;   // output columns per warp
    static constexpr int kNbPV = kColsPerWarp / 8;            // n-blocks per warp in P.V
    static constexpr int kRedStride = kTile + 8;              // floats
    static constexpr int kPStride = kTile + 8;                // bf16 elements

    static constexpr int kStageBytes = kTile * kStageStride;
    static constexpr int kOffStages = 0;
    static constexpr int kOffOp = kOffStages + kStages * kStageBytes;
    static constexpr int kOpBytes = FP8 ? kTile * kOpStride : 0;
    static constexpr int kOffRed = kOffOp + kOpBytes;
    static constexpr int kOffP = kOffRed + 4 * kHeads * kRedStride * 4;
    static constexpr int kOffAlpha = kOffP + kHeads * kPStride * 2;
    static constexpr int kOffMl = kOffAlpha + kHeads * 4;
    static constexpr int kOffMask = kOffMl + kHeads * 8;
    static constexpr int kOffBars = kOffMask + kStages * 8;
    static constexpr int kOffFlags = kOffBars + 2 * kStages * 8;
    static constexpr int kOffCum = kOffFlags + 16;
    static size_t smem_bytes(int batch) { return kOffCum + 4 * (batch + 1); }

    static_assert(D % 64 == 0 && kKSteps % 4 == 0, "head size must split into 4 quarters");
    static_assert(kColsPerWarp % 16 == 0, "P.V columns per warp must be a multiple of 16");
    static_assert(kRowBytes % 16 == 0, "bulk copies need 16-byte rows");
};

template <int D, int R, bool FP8>
__global__ void __launch_bounds__(MlaMmaCfg<D, R, FP8>::kThreads, 1)
    mla_decode_mma_kernel(const MlaArgs a) {
    using C = MlaMmaCfg<D, R, FP8>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem + C::kOffStages;
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + C::kOffP);
    float* alpha_s = reinterpret_cast<float*>(smem + C::kOffAlpha);
    float2* ml_s = reinterpret_cast<float2*>(smem + C::kOffMl);
    uint64_t* mask_s = reinterpret_cast<uint64_t*>(smem + C::kOffMask);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* empty = full + C::kStages;
    int* abort_s = reinterpret_cast<int*>(smem + C::kOffFlags);
    int* cum = reinterpret_cast<int*>(smem + C::kOffCum);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = (a.H + C::kHeads - 1) / C::kHeads;
    const int unit = blockIdx.x / n_groups;
    const int h0 = (blockIdx.x % n_groups) * C::kHeads;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kConsumerWarps);
        }
        *abort_s = 0;
        fence_mbar_init();
    }
    // Zero every staging row once so that rows never written by a copy hold
    // finite values.
    for (int i = threadIdx.x * 16; i < C::kStages * C::kStageBytes; i += C::kThreads * 16)
        *reinterpret_cast<uint4*>(stages + i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    const int T = build_cum(a.plan, a.seq_lens, cum, a.status);  // contains __syncthreads

    const int P = a.plan.page;

    if (warp == C::kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_policy_evict_first();
        PieceIter it;
        it.init(a.plan, cum, T, unit);
        Piece pc;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int issued[C::kStages];
        for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
        while (ok && it.next(cum, pc)) {
            const int len = clamp_len(a.seq_lens[pc.b], a.plan.max_blocks, P, nullptr);
            const int tok0 = pc.j0 * P;
            const int tok_end = min(pc.j1 * P, len);
            const int32_t* bt = a.block_table + static_cast<long long>(pc.b) * a.plan.max_blocks;
            for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
                if (!mbar_wait(&empty[stage], phase ^ 1)) {
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
                uint8_t* dst = stages + stage * C::kStageBytes;
                const uint8_t* src[2];
                bool valid[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int r = lane + 32 * k;
                    const int tok = t0 + r;
                    valid[k] = tok < tok_end;
                    src[k] = nullptr;
                    if (valid[k]) {
                        const int blk = bt[tok / P];
                        if (blk < 0 || blk >= a.num_blocks) {
                            report(a.status, MQA_ERR_DEVICE_CHECK);
                            valid[k] = false;
                        } else {
                            src[k] = a.kv + (static_cast<long long>(blk) * P + tok % P) * C::kRowBytes;
                        }
                    }
                    if (!valid[k]) {
                        uint4* row = reinterpret_cast<uint4*>(dst + r * C::kStageStride);
                        for (int c = 0; c < C::kRowBytes / 16; ++c) row[c] = make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();
                    }
                }
                const uint32_t m0 = __ballot_sync(0xffffffffu, valid[0]);
                const uint32_t m1 = __ballot_sync(0xffffffffu, valid[1]);
                __syncwarp();
                if (lane == 0) {
                    mask_s[stage] = static_cast<uint64_t>(m0) | (static_cast<uint64_t>(m1) << 32);
                    mbar_arrive_expect_tx(&full[stage], (__popc(m0) + __popc(m1)) * C::kRowBytes);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (valid[k])
                        bulk_g2s(dst + (lane + 32 * k) * C::kStageStride, src[k], C::kRowBytes,
                                 &full[stage], pol);
                issued[stage] = static_cast<int>(phase);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // Never leave copies in flight behind: wait (bounded) for the last
        // fill of every stage.
        for (int s = 0; s < C::kStages; ++s)
            if (issued[s] >= 0 && !mbar_wait(&full[s], static_cast<uint32_t>(issued[s])))
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        return;
    }

    // -------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    const int th = warp >> 2, dq = warp & 3;  // QK role: token half, head-dim quarter
    const int t = threadIdx.x;                // softmax role: head sh, tokens 4*sk..4*sk+3
    const int sh = t >> 4, sk = t & 15;

    PieceIter it;
    it.init(a.plan, cum, T, unit);
    Piece pc;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;

    while (!aborted && it.next(cum, pc)) {
        const int len = clamp_len(a.seq_lens[pc.b], a.plan.max_blocks, P, nullptr);
        const int tok0 = pc.j0 * P;
        const int tok_end = min(pc.j1 * P, len);

        // Q fragments of this warp's head-dim quarter (rows beyond H are zero).
        uint32_t qa[C::kKq][4];
        {
            const __nv_bfloat16* qb = a.q + (static_cast<long long>(pc.b) * a.H + h0) * D;
            const bool r0 = h0 + g < a.H, r1 = h0 + g + 8 < a.H;
#pragma unroll
            for (int ks = 0; ks < C::kKq; ++ks) {
                const int k0 = (dq * C::kKq + ks) * 16 + 2 * c;
                qa[ks][0] = r0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + k0) : 0u;
                qa[ks][1] = r1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + k0) : 0u;
                qa[ks][2] = r0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + k0 + 8) : 0u;
                qa[ks][3] = r1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + k0 + 8) : 0u;
            }
        }
        float o[C::kNbPV][4];
#pragma unroll
        for (int i = 0; i < C::kNbPV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;  // softmax role, head sh

        for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
            const bool ok = mbar_wait(&full[stage], phase);
            if (!ok) {
                *abort_s = 1;
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            }
            const uint8_t* stage_buf = stages + stage * C::kStageBytes;
            const uint8_t* op = stage_buf;
            int op_stride = C::kStageStride;
            if constexpr (FP8) {
                // Widen the e4m3 tile to bf16 (exact) in the operand buffer.
                uint8_t* opw = smem + C::kOffOp;
                named_bar_sync(3, C::kConsumers);  // previous tile's P.V is done
                if (ok) {
                    constexpr int kChunks = C::kTile * (D / 16);
                    for (int i = t; i < kChunks; i += C::kConsumers) {
                        const int r = i / (D / 16), cc = i % (D / 16);
                        const uint4 v = *reinterpret_cast<const uint4*>(stage_buf + r * C::kStageStride + cc * 16);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        uint32_t outw[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const __nv_fp8x2_storage_t pr =
                                    static_cast<__nv_fp8x2_storage_t>((w[j] >> (16 * hh)) & 0xffffu);
                                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
                                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
                                outw[2 * j + hh] = pack_bf16x2(f.x, f.y);
                            }
                        }
                        uint4* d = reinterpret_cast<uint4*>(opw + r * C::kOpStride + cc * 32);
                        d[0] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
                        d[1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                named_bar_sync(3, C::kConsumers);
                op = opw;
                op_stride = C::kOpStride;
            }
            const uint64_t vmask = mask_s[stage];

            // ---- S partial = Q[:, quarter] K[tokens of half th, quarter]^T
            float sacc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < C::kKq; ++ks) {
                    const int k0 = (dq * C::kKq + ks) * 16;
#pragma unroll
                    for (int nb2 = 0; nb2 < 2; ++nb2) {
                        const int row = th * 32 + nb2 * 16 + (lane & 7) + ((lane >> 4) << 3);
                        const int col = k0 + ((lane >> 3) & 1) * 8;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(b0, b1, b2, b3, op + row * op_stride + col * 2);
                        mma_bf16_16816(sacc[2 * nb2], qa[ks], b0, b1);
                        mma_bf16_16816(sacc[2 * nb2 + 1], qa[ks], b2, b3);
                    }
                }
            }
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                const int col = th * 32 + nb * 8 + 2 * c;
                *reinterpret_cast<float2*>(&red[(dq * 16 + g) * C::kRedStride + col]) =
                    make_float2(sacc[nb][0], sacc[nb][1]);
                *reinterpret_cast<float2*>(&red[(dq * 16 + g + 8) * C::kRedStride + col]) =
                    make_float2(sacc[nb][2], sacc[nb][3]);
            }
            named_bar_sync(1, C::kConsumers);

            // ---- online softmax for head sh over tokens 4*sk .. 4*sk+3
            {
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 v = *reinterpret_cast<const float4*>(&red[(q4 * 16 + sh) * C::kRedStride + 4 * sk]);
                    x[0] += v.x;
                    x[1] += v.y;
                    x[2] += v.z;
                    x[3] += v.w;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool valid = (vmask >> (4 * sk + i)) & 1ull;
                    x[i] = valid ? x[i] * a.sl2 : -INFINITY;
                    mx = fmaxf(mx, x[i]);
                }
#pragma unroll
                for (int o2 = 8; o2 >= 1; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                const float m_new = fmaxf(m_run, mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = ex2(m_run - m_use);
                float psum = 0.f;
                uint32_t pk[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    // l sums the fp32 probabilities; P.V uses them rounded to bf16
                    const float p0 = ex2(x[2 * i] - m_use), p1 = ex2(x[2 * i + 1] - m_use);
                    psum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
#pragma unroll
                for (int o2 = 8; o2 >= 1; o2 >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o2);
                l_run = l_run * alpha + psum;
                m_run = m_new;
                *reinterpret_cast<uint2*>(&Ps[sh * C::kPStride + 4 * sk]) = make_uint2(pk[0], pk[1]);
                if (sk == 0) alpha_s[sh] = alpha;
            }
            named_bar_sync(2, C::kConsumers);

            // ---- O = alpha O + P V over this warp's output columns
            {
                const float al0 = alpha_s[g], al1 = alpha_s[g + 8];
#pragma unroll
                for (int i = 0; i < C::kNbPV; ++i) {
                    o[i][0] *= al0;
                    o[i][1] *= al0;
                    o[i][2] *= al1;
                    o[i][3] *= al1;
                }
                if (ok) {
#pragma unroll
                    for (int kk = 0; kk < C::kTile / 16; ++kk) {
                        uint32_t pa[4];
                        ldsm_x4(pa[0], pa[1], pa[2], pa[3],
                                &Ps[(lane & 15) * C::kPStride + kk * 16 + (lane >> 4) * 8]);
#pragma unroll
                        for (int nb2 = 0; nb2 < C::kNbPV / 2; ++nb2) {
                            const int tok = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                            const int col = warp * C::kColsPerWarp + nb2 * 16 + (lane >> 4) * 8;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(b0, b1, b2, b3, op + tok * op_stride + col * 2);
                            mma_bf16_16816(o[2 * nb2], pa, b0, b1);
                            mma_bf16_16816(o[2 * nb2 + 1], pa, b2, b3);
                        }
                    }
                }
            }
            if constexpr (!FP8) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
            }
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1;
            }
            if (*abort_s) {
                aborted = true;
                break;
            }
        }
        if (aborted) break;

        // ---- epilogue: normalise and write the piece's result
        if (sk == 0) ml_s[sh] = make_float2(m_run, l_run);
        named_bar_sync(1, C::kConsumers);
        {
            const float l0 = ml_s[g].y, l1 = ml_s[g + 8].y;
            const float i0 = l0 > 0.f ? a.out_scale / l0 : 0.f;
            const float i1 = l1 > 0.f ? a.out_scale / l1 : 0.f;
            const int hr0 = h0 + g, hr1 = h0 + g + 8;
#pragma unroll
            for (int i = 0; i < C::kNbPV; ++i) {
                const int col = warp * C::kColsPerWarp + i * 8 + 2 * c;
                if (pc.whole) {
                    if (hr0 < a.H)
                        *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(pc.b) * a.H + hr0) * R + col) =
                            pack_bf16x2(o[i][0] * i0, o[i][1] * i0);
                    if (hr1 < a.H)
                        *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(pc.b) * a.H + hr1) * R + col) =
                            pack_bf16x2(o[i][2] * i1, o[i][3] * i1);
                } else {
                    if (hr0 < a.H)
                        *reinterpret_cast<float2*>(a.ws_o + (static_cast<long long>(pc.slot) * a.H + hr0) * R + col) =
                            make_float2(o[i][0] * i0, o[i][1] * i0);
                    if (hr1 < a.H)
                        *reinterpret_cast<float2*>(a.ws_o + (static_cast<long long>(pc.slot) * a.H + hr1) * R + col) =
                            make_float2(o[i][2] * i1, o[i][3] * i1);
                }
            }
            if (sk == 0 && h0 + sh < a.H) {
                // natural-log LSE of the scaled logits; k_scale rescales V only
                const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
                if (pc.whole) {
                    if (a.lse) a.lse[static_cast<long long>(pc.b) * a.H + h0 + sh] = lse;
                } else {
                    a.ws_lse[static_cast<long long>(pc.slot) * a.H + h0 + sh] = lse;
                }
            }
        }
        named_bar_sync(1, C::kConsumers);
    }
}

template <int D, int R, bool FP8>
static cudaError_t launch_mla_mma(const MlaArgs& a, int grid, cudaStream_t stream) {
    using C = MlaMmaCfg<D, R, FP8>;
    const size_t smem = C::smem_bytes(a.plan.batch);
    auto kern = mla_decode_mma_kernel<D, R, FP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, C::kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t mla_mma_stage1(const MlaArgs& a, int D, bool fp8, int grid, cudaStream_t stream) {
    if (D == 576) return fp8 ? launch_mla_mma<576, 512, true>(a, grid, stream)
                             : launch_mla_mma<576, 512, false>(a, grid, stream);
    return fp8 ? launch_mla_mma<320, 256, true>(a, grid, stream)
               : launch_mla_mma<320, 256, false>(a, grid, stream);
}

size_t mla_mma_smem_bytes(int D, bool fp8, int batch) {
    if (D == 576) return fp8 ? MlaMmaCfg<576, 512, true>::smem_bytes(batch)
                             : MlaMmaCfg<576, 512, false>::smem_bytes(batch);
    return fp8 ? MlaMmaCfg<320, 256, true>::smem_bytes(batch)
               : MlaMmaCfg<320, 256, false>::smem_bytes(batch);
}

}  // namespace mqa
