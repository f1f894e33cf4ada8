// GQA paged decode, stage 1, over 8-bit caches.
//
// Formats ("Triton と MLA" page, vllm-arch-zh ja/attention/triton-mla: 役割 and
// 設計動機 list the Triton backend's quantised KV cache dtypes, 主要ファイル
// says the per_token_head modes pad head_dim to hold an inline scale):
//   * e4m3 codes with one k_scale and one v_scale for the whole cache,
//     [num_blocks, 2, page, Hkv, D] bytes;
//   * per-token-head e4m3 or int8 codes, [num_blocks, 2, page, Hkv, D + 4]
//     bytes: each (token, KV head) row holds its D codes followed by its own
//     scale (little-endian fp32); element value = scale * code.
//
// One thread block = Hkv consumer warps + 1 producer warp, persistent over a
// work unit (plan.cuh), as in the bf16 kernel.  The producer stages 16-token
// tiles of the K and V planes of one page (tiles start on a multiple of 16
// tokens and pages hold a multiple of 16, so a tile stays inside its page):
// one bulk copy per token row when a row (all KV heads) is a multiple of 16
// bytes, into rows padded by 16 bytes so that the consumers' reads spread
// over the banks (measured faster than dense tiles even where those would
// collide only 2 ways), else one bulk copy of the 16 dense rows per plane.
// The stage count is set per launch from the shared memory left by the batch.
//
// Consumer warp g owns KV head g and its query heads (an m16 tile).
//   * S = Q K^T by warp MMA with f16 operands.  The reduction order inside
//     each 16-wide step is permuted (lane c takes head dims 4c .. 4c + 3 in
//     both Q and K), so a lane's K operand of one token is one 4-byte read of
//     codes, widened to f16 in registers: no K tile is written back.
//   * the K scale of each token multiplies its logits in fp32; online
//     softmax in base 2 (tutorial page lshu.cn/news/265860, §7) with lazy
//     rescaling: the reference max moves only when a logit exceeds it by more
//     than 8 (P <= 2^8), so O is rescaled rarely.
//   * V codes are widened to f16 into a private 16-row tile (ldmatrix.trans
//     feeds P.V); P is multiplied by the V scale of its token and by 2^-e, e
//     the exponent above the largest V scale of the piece so far, so the f16
//     products stay normal numbers whatever the scales' magnitude; O follows
//     e with exact power-of-two rescales and is multiplied back at the end.
//   * the stage is released as soon as the K reads and the V widening are
//     done, before the softmax.
// Tokens past the sequence end (and whole tiles of a page with an invalid
// block id) are masked out of the softmax, their V rows widened as zeros and
// their V scale taken as 0, so padding never reaches the output.
//
// f16 operands: e4m3 -> f16 is one conversion per code pair and int8 -> f16
// an exact integer trick (1024 + u - 1152), where bf16 needs three more
// steps per pair; the price is the f16 range of the query: its entries must
// stay below 65504 in magnitude.
#include <cuda_fp8.h>

#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"
#include "gqa_q8.cuh"

namespace mqa {

namespace {

constexpr int kFmtE4m3 = MQA_KV_FP8_E4M3;
constexpr int kFmtE4m3Pth = MQA_KV_FP8_E4M3_PER_TOKEN_HEAD;
constexpr int kFmtInt8Pth = MQA_KV_INT8_PER_TOKEN_HEAD;

template <int D, int KIND>
struct GqaQ8Cfg {
    static constexpr bool kPth = KIND != kFmtE4m3;
    static constexpr int kTile = 16;
    static constexpr int kMaxKvHeads = 8;
    static constexpr int kDp = kPth ? D + 4 : D;  // bytes of one (token, KV head) row
    static constexpr int kKSteps = D / 16;
    static constexpr int kNb = D / 8;
    // widened f16 V tile rows: 16 bytes of padding keep ldmatrix conflict-free
    static constexpr int kWStride = 2 * D + 16;
    static constexpr int kWBytes = kTile * kWStride;  // one warp's V tile
    static_assert(kWBytes % 128 == 0, "per-warp tiles stay 128-byte aligned");
    static constexpr int kMaxStages = 8;
    __host__ __device__ static int row_bytes(int hkv) { return hkv * kDp; }  // one token, all heads
    // Rows are copied one by one into rows padded by 16 bytes when a row is a
    // multiple of 16 bytes (the consumers' reads of 8 rows then spread over
    // the banks), else a tile is one copy of 16 dense rows per plane.
    __host__ __device__ static bool per_row(int hkv) { return row_bytes(hkv) % 16 == 0; }
    __host__ __device__ static int row_stride(int hkv) { return row_bytes(hkv) + (per_row(hkv) ? 16 : 0); }
    __host__ __device__ static int plane_bytes(int hkv) { return kTile * row_stride(hkv); }
    __host__ __device__ static int stage_bytes(int hkv) { return 2 * plane_bytes(hkv); }
    // layout: V tiles (per warp) | stages | masks | full bars | empty bars | cum
    __host__ __device__ static size_t off_stages(int hkv) { return static_cast<size_t>(hkv) * kWBytes; }
    __host__ __device__ static size_t off_masks(int hkv, int ns) {
        return off_stages(hkv) + static_cast<size_t>(ns) * stage_bytes(hkv);
    }
    __host__ __device__ static size_t off_bars(int hkv, int ns) { return off_masks(hkv, ns) + 8 * ns; }
    __host__ __device__ static size_t off_cum(int hkv, int ns) { return off_bars(hkv, ns) + 16 * ns; }
    static size_t smem_bytes(int hkv, int ns, int batch) { return off_cum(hkv, ns) + 4 * (2 * batch + 1); }
    // as many stages as fit in `limit` bytes of shared memory (2 .. kMaxStages)
    static int stages_for(int hkv, int batch, size_t limit) {
        int ns = kMaxStages;
        while (ns > 2 && smem_bytes(hkv, ns, batch) > limit) --ns;
        return ns;
    }
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) { return h2_bits(__floats2half2_rn(lo, hi)); }

// A bf16 pair -> the f16 pair of the same values (exact inside the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    return pack_f16x2(f.x, f.y);
}

// Four codes (bytes of w, lowest first) -> four f16 values (exact).
template <int KIND>
__device__ __forceinline__ uint2 widen4(uint32_t w) {
    if constexpr (KIND == kFmtInt8Pth) {
        // u = x + 128 in [0, 255] placed in the mantissa of 1024 (0x6400):
        // the f16 value 1024 + u is exact, minus 1152 gives x
        const uint32_t u = w ^ 0x80808080u;
        const __half2 k = bits_h2(0x64806480u);
        const uint32_t lo = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4140)), k));
        const uint32_t hi = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4342)), k));
        return make_uint2(lo, hi);
    } else {
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
        return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
}

// Widen one KV head's 16 rows of codes (src: the head's first code in the
// plane tile, rows `rbytes` apart) into an f16 tile with row stride kWStride.
// Rows of tokens not in vmask become zeros without reading their bytes.
template <int D, int KIND>
__device__ __forceinline__ void widen_rows(const uint8_t* src, uint8_t* dst, uint64_t vmask, int rbytes,
                                           int lane) {
    using C = GqaQ8Cfg<D, KIND>;
    constexpr int kLanesPerRow = D / 4;
    constexpr int kRowsPer = 32 / kLanesPerRow;
    const int sub = lane / kLanesPerRow, ch = lane % kLanesPerRow;
#pragma unroll
    for (int r0 = 0; r0 < C::kTile; r0 += kRowsPer) {
        const int r = r0 + sub;
        const bool v = (vmask >> r) & 1ull;
        const uint32_t w = v ? *reinterpret_cast<const uint32_t*>(src + r * rbytes + 4 * ch) : 0u;
        *reinterpret_cast<uint2*>(dst + r * C::kWStride + 8 * ch) = widen4<KIND>(w);
    }
}

// Exponent e with vmax < 2^e (vmax > 0, finite): the power of two that P
// times a V scale is divided by.
__device__ __forceinline__ int scale_exponent(float vmax) {
    int e;
    frexpf(vmax, &e);  // vmax = f * 2^e, 0.5 <= f < 1
    return e;
}

template <int D, int KIND>
__global__ void __launch_bounds__(32 * (GqaQ8Cfg<D, KIND>::kMaxKvHeads + 1), 1)
    gqa_decode_q8_kernel(const GqaArgs a, const float out_scale, const int nstage) {
    using C = GqaQ8Cfg<D, KIND>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int Hkv = a.Hkv;
    const int rbytes = C::row_bytes(Hkv);
    const int rstride = C::row_stride(Hkv);
    const int pbytes = C::plane_bytes(Hkv);
    const int sbytes = C::stage_bytes(Hkv);
    uint8_t* stages = smem + C::off_stages(Hkv);
    uint64_t* mask_s = reinterpret_cast<uint64_t*>(smem + C::off_masks(Hkv, nstage));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::off_bars(Hkv, nstage));
    uint64_t* empty = full + nstage;
    int* cum = reinterpret_cast<int*>(smem + C::off_cum(Hkv, nstage));
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
    pdl_wait();
    pdl_launch_dependents();
    const int T = build_cum(a.plan, a.seq_lens, cum, lens, a.status);  // contains __syncthreads
    const int P = a.plan.page;

    if (warp == Hkv) {
        // ------------------------------------------------------------ producer
        const bool rows = C::per_row(Hkv);
        const uint64_t pol = l2_policy_evict_first();
        // per-row mode: lane -> (plane, row): lanes 0-15 copy K rows, 16-31 V rows
        const int plane = lane >> 4, r = lane & 15;
        TileCursor cur;
        cur.init(a.plan, cum, T, unit, C::kTile);
        int stage = 0;
        uint32_t phase = 0;
        int issued[C::kMaxStages];
        for (int s = 0; s < C::kMaxStages; ++s) issued[s] = -1;
        // the tile's block id is read one tile ahead of its use
        bool have = cur.next(a.plan, cum, lens, a.block_table);
        int t0 = have ? cur.t0 : 0, tend = have ? cur.tok_end : 0;
        int blk = have ? __ldg(cur.bt + t0 / P) : 0;
        while (have) {
            const bool have_next = cur.next(a.plan, cum, lens, a.block_table);
            const int nt0 = have_next ? cur.t0 : 0, ntend = have_next ? cur.tok_end : 0;
            const int nblk = have_next ? __ldg(cur.bt + nt0 / P) : 0;
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                break;
            }
            const bool valid = blk >= 0 && blk < a.num_blocks;
            const int nv = min(C::kTile, tend - t0);  // >= 1: the cursor only yields non-empty tiles
            // slot t0 % P of page blk: plane 0 (K), plane 1 (V) P rows later
            const uint8_t* src = a.kv + (static_cast<long long>(blk) * 2 * P + t0 % P) * rbytes;
            uint8_t* dst = stages + stage * sbytes;
            if (lane == 0) {
                if (!valid) report(a.status, MQA_ERR_DEVICE_CHECK);
                mask_s[stage] = valid ? ((1ull << nv) - 1ull) : 0ull;
                // per-row mode copies the nv valid rows of each plane
                const uint32_t bytes = !valid ? 0u : (rows ? 2u * nv * rbytes : 2u * pbytes);
                mbar_arrive_expect_tx(&full[stage], bytes);
            }
            __syncwarp();
            if (valid) {
                if (rows) {
                    if (r < nv)
                        bulk_g2s(dst + plane * pbytes + r * rstride,
                                 src + (static_cast<long long>(plane) * P + r) * rbytes, rbytes, &full[stage], pol);
                } else if (lane == 0) {
                    bulk_g2s(dst, src, pbytes, &full[stage], pol);
                    bulk_g2s(dst + pbytes, src + static_cast<long long>(P) * rbytes, pbytes, &full[stage], pol);
                }
            }
            issued[stage] = static_cast<int>(phase);
            if (++stage == nstage) {
                stage = 0;
                phase ^= 1;
            }
            have = have_next;
            t0 = nt0;
            tend = ntend;
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
    const int hoff = gk * C::kDp;  // byte offset of this KV head inside a token row
    uint8_t* wv = smem + gk * C::kWBytes;

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

        // Q as f16, in the permuted reduction order: step ks, lane c holds
        // head dims 16 ks + 4c .. 4c + 3 of rows g and g + 8 (a0/a2 and a1/a3)
        uint32_t qa[C::kKSteps][4];
        {
            const __nv_bfloat16* qb = a.q + (static_cast<long long>(pc.b) * a.Hq + hq0) * D;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int k0 = ks * 16 + 4 * c;
                const uint2 q0 = row0 ? *reinterpret_cast<const uint2*>(qb + g * D + k0) : make_uint2(0u, 0u);
                const uint2 q1 = row1 ? *reinterpret_cast<const uint2*>(qb + (g + 8) * D + k0) : make_uint2(0u, 0u);
                qa[ks][0] = bf16x2_to_f16x2(q0.x);
                qa[ks][1] = bf16x2_to_f16x2(q1.x);
                qa[ks][2] = bf16x2_to_f16x2(q0.y);
                qa[ks][3] = bf16x2_to_f16x2(q1.y);
            }
        }
        float o[C::kNb][4];
#pragma unroll
        for (int i = 0; i < C::kNb; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
        int e_run = -1000000;  // exponent of the P . V factor 2^-e (per-token-head scales)
        float p_fac = 1.f;     // 2^-e_run

        for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
            const bool ok = mbar_wait(&full[stage], phase);
            if (!ok) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            const uint8_t* kb = stages + stage * sbytes + hoff;
            const uint8_t* vb = kb + pbytes;
            const uint64_t vmask = mask_s[stage];

            // K and V scales of this lane's four token columns (nb * 8 + 2c + e);
            // 0 for masked tokens
            float ksc[4], vsc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = (i >> 1) * 8 + 2 * c + (i & 1);
                const bool v = (vmask >> tok) & 1ull;
                if constexpr (C::kPth) {
                    ksc[i] = v ? *reinterpret_cast<const float*>(kb + tok * rstride + D) : 0.f;
                    vsc[i] = v ? *reinterpret_cast<const float*>(vb + tok * rstride + D) : 0.f;
                } else {
                    ksc[i] = 1.f;
                    vsc[i] = 1.f;
                }
            }
            __syncwarp();  // the previous tile's ldmatrix reads of wv are done
            widen_rows<D, KIND>(vb, wv, vmask, rstride, lane);

            // S = Q K^T: token n = nb * 8 + g, one 4-byte read of its codes
            // per step (masked tokens' columns are discarded below)
            float s[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(kb + (nb * 8 + g) * rstride + ks * 16 + 4 * c);
                    const uint2 kf = widen4<KIND>(w);
                    mma_f16_16816(s[nb], qa[ks], kf.x, kf.y);
                }
            }
            __syncwarp();  // every lane's K reads and V tile writes are done
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == nstage) {
                stage = 0;
                phase ^= 1;
            }
            // P . V factor: grows with the largest |V scale| of the piece
            float o_fix = 1.f;
            if constexpr (C::kPth) {
                float vmax = fmaxf(fmaxf(fabsf(vsc[0]), fabsf(vsc[1])), fmaxf(fabsf(vsc[2]), fabsf(vsc[3])));
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
                if (vmax > 0.f && vmax <= 3.0e38f) {
                    const int e = scale_exponent(vmax);
                    if (e > e_run) {
                        o_fix = e_run == -1000000 ? 1.f : ldexpf(1.f, e_run - e);
                        e_run = e;
                        p_fac = ldexpf(1.f, -e);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) vsc[i] *= p_fac;
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
                    x[nb][j] = valid ? s[nb][j] * ksc[nb * 2 + (j & 1)] * a.sl2 : -INFINITY;
                    mx[j >> 1] = fmaxf(mx[j >> 1], x[nb][j]);
                }
            float alpha[2] = {1.f, 1.f};
            bool grow = false;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                // lazy: move the reference only when P would exceed 2^8
                if (mx[r] > m_run[r] + 8.f) {
                    alpha[r] = ex2(m_run[r] - mx[r]);
                    m_run[r] = mx[r];
                    l_part[r] *= alpha[r];
                    grow = true;
                }
            }
            const float m_use0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
            const float m_use1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
            uint32_t pa[4];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                // l sums the fp32 probabilities; P.V takes them times the V
                // scale of their token and 2^-e_run, rounded to f16
                const float p0 = ex2(x[nb][0] - m_use0), p1 = ex2(x[nb][1] - m_use0);
                const float p2 = ex2(x[nb][2] - m_use1), p3 = ex2(x[nb][3] - m_use1);
                l_part[0] += p0 + p1;
                l_part[1] += p2 + p3;
                pa[2 * nb] = pack_f16x2(p0 * vsc[2 * nb], p1 * vsc[2 * nb + 1]);
                pa[2 * nb + 1] = pack_f16x2(p2 * vsc[2 * nb], p3 * vsc[2 * nb + 1]);
            }
            if (__any_sync(0xffffffffu, grow) || o_fix != 1.f) {
                const float oa0 = alpha[0] * o_fix, oa1 = alpha[1] * o_fix;
#pragma unroll
                for (int i = 0; i < C::kNb; ++i) {
                    o[i][0] *= oa0;
                    o[i][1] *= oa0;
                    o[i][2] *= oa1;
                    o[i][3] *= oa1;
                }
            }
#pragma unroll
            for (int nb2 = 0; nb2 < C::kNb / 2; ++nb2) {
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int col = nb2 * 16 + (lane >> 4) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3, wv + tok * C::kWStride + col * 2);
                mma_f16_16816(o[2 * nb2], pa, b0, b1);
                mma_f16_16816(o[2 * nb2 + 1], pa, b2, b3);
            }
            if (!ok) {
                aborted = true;
                break;
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
        // undo the P . V factor 2^-e_run (per-token-head scales)
        const float osc = (C::kPth && e_run != -1000000) ? ldexpf(out_scale, e_run) : out_scale;
        const float i0 = l[0] > 0.f ? osc / l[0] : 0.f, i1 = l[1] > 0.f ? osc / l[1] : 0.f;
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

// Dynamic shared memory a block may use on sm_103a (227 KB).
constexpr size_t kSmemLimit = 227 * 1024;

template <int D, int KIND>
cudaError_t launch_q8(const GqaArgs& a, float out_scale, int grid, cudaStream_t stream) {
    using C = GqaQ8Cfg<D, KIND>;
    const int ns = C::stages_for(a.Hkv, a.plan.batch, kSmemLimit);
    const size_t smem = C::smem_bytes(a.Hkv, ns, a.plan.batch);
    auto kern = gqa_decode_q8_kernel<D, KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(grid), dim3(32 * (a.Hkv + 1)), smem, stream, a, out_scale, ns);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_q8_kind(const GqaArgs& a, float out_scale, int kind, int grid, cudaStream_t stream) {
    if (kind == kFmtE4m3Pth) return launch_q8<D, kFmtE4m3Pth>(a, out_scale, grid, stream);
    if (kind == kFmtInt8Pth) return launch_q8<D, kFmtInt8Pth>(a, out_scale, grid, stream);
    return launch_q8<D, kFmtE4m3>(a, out_scale, grid, stream);
}

template <int D, int KIND>
size_t smem_of(int hkv, int batch) {
    using C = GqaQ8Cfg<D, KIND>;
    return C::smem_bytes(hkv, C::stages_for(hkv, batch, kSmemLimit), batch);
}

template <int D>
size_t smem_kind(int kind, int hkv, int batch) {
    if (kind == kFmtE4m3Pth) return smem_of<D, kFmtE4m3Pth>(hkv, batch);
    if (kind == kFmtInt8Pth) return smem_of<D, kFmtInt8Pth>(hkv, batch);
    return smem_of<D, kFmtE4m3>(hkv, batch);
}

}  // namespace

cudaError_t gqa_q8_stage1(const GqaArgs& a, float out_scale, int D, int kind, int grid, cudaStream_t stream) {
    if (D == 128) return launch_q8_kind<128>(a, out_scale, kind, grid, stream);
    return launch_q8_kind<64>(a, out_scale, kind, grid, stream);
}

size_t gqa_q8_smem_bytes(int D, int kind, int hkv, int batch) {
    return D == 128 ? smem_kind<128>(kind, hkv, batch) : smem_kind<64>(kind, hkv, batch);
}

}  // namespace mqa
