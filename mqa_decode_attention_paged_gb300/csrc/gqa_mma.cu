// GQA paged decode, stage 1 (secondary mode).
//
// Cache layout [num_blocks, 2, page, Hkv, D]: plane 0 = K, plane 1 = V
// ("AttentionBackend" page, vllm-arch-zh fr/attention/backend, "Motivation de
// conception").  One thread block = Hkv consumer warps + 1 producer warp,
// persistent over a work unit (plan.cuh).  The producer stages 16-token tiles:
// for each token one bulk copy of its K row (all KV heads, Hkv*D bf16) and
// one of its V row.  Consumer warp g owns KV head g and the query heads
// g*grp .. g*grp+grp-1 (grp = Hq / Hkv <= 16, padded to an m16 tile), and
// runs the whole tile in registers: S = Q K^T, online softmax per query head
// (tutorial page lshu.cn/news/265860, §7), P reused directly as the A operand
// of O += P V.
#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"
#include "gqa_test.cuh"

namespace mqa {

template <int D>
struct GqaCfg {
    static constexpr int kTile = 16;
    static constexpr int kMaxKvHeads = 8;
    static constexpr int kKSteps = D / 16;
    static constexpr int kNb = D / 8;  // n-blocks of the output row
    __host__ __device__ static int row_bytes(int hkv) { return hkv * D * 2; }
    __host__ __device__ static int row_stride(int hkv) { return hkv * D * 2 + 16; }
    __host__ __device__ static int stage_bytes(int hkv) { return 2 * kTile * row_stride(hkv); }
    __host__ __device__ static int stages(int hkv) {
        const int sb = stage_bytes(hkv);
        int n = (200 * 1024) / sb;
        return n < 2 ? 2 : (n > 6 ? 6 : n);
    }
    // layout: stages | masks | full bars | empty bars | flags | cum
    __host__ __device__ static size_t off_masks(int hkv) { return static_cast<size_t>(stages(hkv)) * stage_bytes(hkv); }
    __host__ __device__ static size_t off_bars(int hkv) { return off_masks(hkv) + 8 * stages(hkv); }
    __host__ __device__ static size_t off_flags(int hkv) { return off_bars(hkv) + 16 * stages(hkv); }
    __host__ __device__ static size_t off_cum(int hkv) { return off_flags(hkv) + 16; }
    static size_t smem_bytes(int hkv, int batch) { return off_cum(hkv) + 4 * (2 * batch + 1); }
};

// withhold: test hook for the bounded waits (-1 in every normal call): the
// producer of unit `withhold` fills and announces none of its tiles, so the
// consumers' first wait runs out, they report MQA_ERR_DEVICE_TIMEOUT and
// the block returns; nothing waits without a time limit.
template <int D>
__global__ void __launch_bounds__(32 * (GqaCfg<D>::kMaxKvHeads + 1), 1)
    gqa_decode_mma_kernel(const GqaArgs a, const int withhold) {
    using C = GqaCfg<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int Hkv = a.Hkv;
    const int nstage = C::stages(Hkv);
    const int stride = C::row_stride(Hkv);
    const int rbytes = C::row_bytes(Hkv);
    const int sbytes = C::stage_bytes(Hkv);
    uint8_t* stages = smem;
    uint64_t* mask_s = reinterpret_cast<uint64_t*>(smem + C::off_masks(Hkv));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::off_bars(Hkv));
    uint64_t* empty = full + nstage;
    int* cum = reinterpret_cast<int*>(smem + C::off_cum(Hkv));
    int* lens = cum + a.plan.batch + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x;
    const int grp = a.Hq / Hkv;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstage; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Hkv);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x * 16; i < nstage * sbytes; i += blockDim.x * 16)
        *reinterpret_cast<uint4*>(stages + i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    pdl_wait();
    pdl_launch_dependents();
    const int T = build_cum(a.plan, a.seq_lens, cum, lens, a.status);
    const int P = a.plan.page;

    if (warp == Hkv) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_policy_evict_first();
        TileCursor cur;
        cur.init(a.plan, cum, T, unit, C::kTile);
        int stage = 0;
        uint32_t phase = 0;
        int issued[8];
        for (int s = 0; s < 8; ++s) issued[s] = -1;
        // lane -> (plane, token): lanes 0-15 copy K rows, 16-31 V rows.
        const int plane = lane >> 4, r = lane & 15;
        // block id of this lane's row, fetched one tile ahead of its use
        bool have = cur.next(a.plan, cum, lens, a.block_table);
        int t0 = cur.t0;
        bool val = have && t0 + r < cur.tok_end;
        int blk = val ? cur.bt[(t0 + r) / P] : 0;
        // test hook: the producer of the withheld unit fills and announces
        // nothing at all, so no copy of it is ever in flight and the
        // consumers' first wait runs out
        if (static_cast<int>(blockIdx.x) == withhold) have = false;
        while (have) {
            const bool have_next = cur.next(a.plan, cum, lens, a.block_table);
            const bool nval = have_next && cur.t0 + r < cur.tok_end;
            const int nblk = nval ? cur.bt[(cur.t0 + r) / P] : 0;
            // warp-uniform: the lanes go on or leave together
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                break;
            }
            uint8_t* dst = stages + stage * sbytes + (plane * C::kTile + r) * stride;
            bool valid = val;
            if (valid && (blk < 0 || blk >= a.num_blocks)) {
                report(a.status, MQA_ERR_DEVICE_CHECK);
                valid = false;
            }
            if (!valid) {
                uint4* row = reinterpret_cast<uint4*>(dst);
                for (int c = 0; c < rbytes / 16; ++c) row[c] = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
            }
            const uint32_t m = __ballot_sync(0xffffffffu, valid);
            __syncwarp();
            if (lane == 0) {
                mask_s[stage] = (m & (m >> 16)) & 0xffffu;  // token valid iff both rows are
                mbar_arrive_expect_tx(&full[stage], __popc(m) * rbytes);
            }
            __syncwarp();
            if (valid) {
                const int tok = t0 + r;
                const uint8_t* src = a.kv + ((static_cast<long long>(blk) * 2 + plane) * P + tok % P) *
                                                static_cast<long long>(rbytes);
                bulk_g2s(dst, src, rbytes, &full[stage], pol);
            }
            issued[stage] = static_cast<int>(phase);
            if (++stage == nstage) {
                stage = 0;
                phase ^= 1;
            }
            have = have_next;
            t0 = cur.t0;
            val = nval;
            blk = nblk;
        }
        for (int s = 0; s < nstage; ++s)
            if (issued[s] >= 0 && !mbar_wait(&full[s], static_cast<uint32_t>(issued[s])))
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        return;
    }

    // ------------------------------------------------------------- consumers
    const int gk = warp;  // KV head
    const int g = lane >> 2, c = lane & 3;
    const bool row0 = g < grp, row1 = g + 8 < grp;
    const int koff = gk * D * 2;  // byte offset of this KV head inside a row

    PieceIter it;
    it.init(a.plan, cum, T, unit);
    Piece pc;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;

    while (!aborted && it.next(cum, pc)) {
        const int len = lens[pc.b];
        const int tok0 = pc.j0 * P;
        const int tok_end = min(pc.j1 * P, len);
        const int hq0 = gk * grp;

        uint32_t qa[C::kKSteps][4];
        {
            const __nv_bfloat16* qb = a.q + (static_cast<long long>(pc.b) * a.Hq + hq0) * D;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int k0 = ks * 16 + 2 * c;
                qa[ks][0] = row0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + k0) : 0u;
                qa[ks][1] = row1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + k0) : 0u;
                qa[ks][2] = row0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + k0 + 8) : 0u;
                qa[ks][3] = row1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + k0 + 8) : 0u;
            }
        }
        float o[C::kNb][4];
#pragma unroll
        for (int i = 0; i < C::kNb; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};

        for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
            // warp-uniform: the lanes go on or leave together; a tile that
            // never arrived is not read (its mask and rows were never
            // written), but its stage is still handed back
            if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase))) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                aborted = true;
                break;
            }
            const uint8_t* kbuf = stages + stage * sbytes;
            const uint8_t* vbuf = kbuf + C::kTile * stride;
            const uint64_t vmask = mask_s[stage];

            float s[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int row = (lane & 7) + ((lane >> 4) << 3);
                const int col = ks * 16 + ((lane >> 3) & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, kbuf + row * stride + koff + col * 2);
                mma_bf16_16816(s[0], qa[ks], b0, b1);
                mma_bf16_16816(s[1], qa[ks], b2, b3);
            }
            // online softmax; rows g (values 0,1) and g+8 (values 2,3)
            float x[2][4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = nb * 8 + 2 * c + (j & 1);
                    const bool valid = (vmask >> tok) & 1ull;
                    x[nb][j] = valid ? s[nb][j] * a.sl2 : -INFINITY;
                    mx[j >> 1] = fmaxf(mx[j >> 1], x[nb][j]);
                }
            float alpha[2], m_use[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float m_new = fmaxf(m_run[r], mx[r]);
                m_use[r] = m_new == -INFINITY ? 0.f : m_new;
                alpha[r] = ex2(m_run[r] - m_use[r]);
                m_run[r] = m_new;
                l_part[r] *= alpha[r];
            }
            uint32_t pa[4];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                // l sums the fp32 probabilities; P.V uses them rounded to bf16
                const float p0 = ex2(x[nb][0] - m_use[0]), p1 = ex2(x[nb][1] - m_use[0]);
                const float p2 = ex2(x[nb][2] - m_use[1]), p3 = ex2(x[nb][3] - m_use[1]);
                l_part[0] += p0 + p1;
                l_part[1] += p2 + p3;
                pa[2 * nb] = pack_bf16x2(p0, p1);
                pa[2 * nb + 1] = pack_bf16x2(p2, p3);
            }
#pragma unroll
            for (int i = 0; i < C::kNb; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[0];
                o[i][2] *= alpha[1];
                o[i][3] *= alpha[1];
            }
#pragma unroll
            for (int nb2 = 0; nb2 < C::kNb / 2; ++nb2) {
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int col = nb2 * 16 + (lane >> 4) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3, vbuf + tok * stride + koff + col * 2);
                mma_bf16_16816(o[2 * nb2], pa, b0, b1);
                mma_bf16_16816(o[2 * nb2 + 1], pa, b2, b3);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == nstage) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (aborted) break;

        float l[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[r] = l_part[r];
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
        }
        const float i0 = l[0] > 0.f ? 1.f / l[0] : 0.f, i1 = l[1] > 0.f ? 1.f / l[1] : 0.f;
        const int hr0 = hq0 + g, hr1 = hq0 + g + 8;
#pragma unroll
        for (int i = 0; i < C::kNb; ++i) {
            const int col = i * 8 + 2 * c;
            if (pc.whole) {
                if (row0)
                    *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(pc.b) * a.Hq + hr0) * D + col) =
                        pack_bf16x2(o[i][0] * i0, o[i][1] * i0);
                if (row1)
                    *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(pc.b) * a.Hq + hr1) * D + col) =
                        pack_bf16x2(o[i][2] * i1, o[i][3] * i1);
            } else {
                if (row0)
                    *reinterpret_cast<float2*>(a.ws_o + (static_cast<long long>(pc.slot) * a.Hq + hr0) * D + col) =
                        make_float2(o[i][0] * i0, o[i][1] * i0);
                if (row1)
                    *reinterpret_cast<float2*>(a.ws_o + (static_cast<long long>(pc.slot) * a.Hq + hr1) * D + col) =
                        make_float2(o[i][2] * i1, o[i][3] * i1);
            }
        }
        if (c == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const bool have = r == 0 ? row0 : row1;
                if (!have) continue;
                const int hr = r == 0 ? hr0 : hr1;
                const float lse = l[r] > 0.f ? (m_run[r] + log2f(l[r])) * kLn2 : -INFINITY;
                if (pc.whole) {
                    if (a.lse) a.lse[static_cast<long long>(pc.b) * a.Hq + hr] = lse;
                } else {
                    a.ws_lse[static_cast<long long>(pc.slot) * a.Hq + hr] = lse;
                }
            }
        }
    }
}

template <int D>
static cudaError_t launch_gqa(const GqaArgs& a, int grid, int withhold, cudaStream_t stream) {
    using C = GqaCfg<D>;
    const size_t smem = C::smem_bytes(a.Hkv, a.plan.batch);
    auto kern = gqa_decode_mma_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(grid), dim3(32 * (a.Hkv + 1)), smem, stream, a, withhold);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t gqa_mma_stage1(const GqaArgs& a, int D, int grid, cudaStream_t stream) {
    if (D == 128) return launch_gqa<128>(a, grid, -1, stream);
    return launch_gqa<64>(a, grid, -1, stream);
}

cudaError_t gqa_mma_stage1_withheld(const GqaArgs& a, int D, int grid, int withhold, cudaStream_t stream) {
    if (D == 128) return launch_gqa<128>(a, grid, withhold, stream);
    return launch_gqa<64>(a, grid, withhold, stream);
}

size_t gqa_mma_smem_bytes(int D, int hkv, int batch) {
    if (D == 128) return GqaCfg<128>::smem_bytes(hkv, batch);
    return GqaCfg<64>::smem_bytes(hkv, batch);
}

}  // namespace mqa
