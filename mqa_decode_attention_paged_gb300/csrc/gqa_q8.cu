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
// tiles with two bulk copies per tile: the 16 consecutive rows of the K plane
// and of the V plane of one page (16 * Hkv * row bytes each; tiles start on a
// multiple of 16 tokens and pages hold a multiple of 16, so every copy is
// 16-byte aligned and stays inside its page).  Consumer warp g owns KV head
// g: it widens its head's 16 K rows and 16 V rows to f16 codes (exact for
// both code types) in a private shared-memory tile, reads the K and V scales
// of its tokens, frees the stage, and then runs the register-resident tile of
// the bf16 kernel with f16 operands (the query is rounded to f16 once per
// piece): S = Q K^T by warp MMA, the K scale applied per token column to S in
// fp32, online softmax in base 2 (tutorial page lshu.cn/news/265860, §7),
// O += P V with P multiplied by the V scale of its token.  So that those
// products stay normal f16 numbers whatever the scales' magnitude, P carries
// a power-of-two factor 2^-e (e: exponent above the largest V scale seen so
// far in the piece); O is rescaled by the same power of two when e grows,
// together with the softmax rescale, and multiplied back at the end.  Tokens
// past the sequence end (and whole tiles of a page with an invalid block id)
// are widened as zeros, masked out of the softmax and get V scale 0, so
// padding never reaches the output.
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
    // widened f16 tile rows: 16 bytes of padding keep ldmatrix conflict-free
    static constexpr int kWStride = 2 * D + 16;
    static constexpr int kWBytes = 2 * kTile * kWStride;  // K and V tiles of one warp
    static_assert(kWBytes % 128 == 0, "per-warp tiles stay 128-byte aligned");
    __host__ __device__ static int row_bytes(int hkv) { return hkv * kDp; }  // one token, all heads
    __host__ __device__ static int plane_bytes(int hkv) { return kTile * row_bytes(hkv); }
    __host__ __device__ static int stage_bytes(int hkv) { return 2 * plane_bytes(hkv); }
    __host__ __device__ static int stages(int hkv) {
        const int n = (200 * 1024 - hkv * kWBytes) / stage_bytes(hkv);
        return n < 2 ? 2 : (n > 8 ? 8 : n);
    }
    // layout: widened tiles (per warp) | stages | masks | full bars | empty bars | cum
    __host__ __device__ static size_t off_stages(int hkv) { return static_cast<size_t>(hkv) * kWBytes; }
    __host__ __device__ static size_t off_masks(int hkv) {
        return off_stages(hkv) + static_cast<size_t>(stages(hkv)) * stage_bytes(hkv);
    }
    __host__ __device__ static size_t off_bars(int hkv) { return off_masks(hkv) + 8 * stages(hkv); }
    __host__ __device__ static size_t off_cum(int hkv) { return off_bars(hkv) + 16 * stages(hkv); }
    static size_t smem_bytes(int hkv, int batch) { return off_cum(hkv) + 4 * (2 * batch + 1); }
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
    gqa_decode_q8_kernel(const GqaArgs a, const float out_scale) {
    using C = GqaQ8Cfg<D, KIND>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int Hkv = a.Hkv;
    const int nstage = C::stages(Hkv);
    const int rbytes = C::row_bytes(Hkv);
    const int pbytes = C::plane_bytes(Hkv);
    const int sbytes = C::stage_bytes(Hkv);
    uint8_t* stages = smem + C::off_stages(Hkv);
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
    pdl_wait();
    pdl_launch_dependents();
    const int T = build_cum(a.plan, a.seq_lens, cum, lens, a.status);  // contains __syncthreads
    const int P = a.plan.page;

    if (warp == Hkv) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = l2_policy_evict_first();
        TileCursor cur;
        cur.init(a.plan, cum, T, unit, C::kTile);
        int stage = 0;
        uint32_t phase = 0;
        int issued[8];
        for (int s = 0; s < 8; ++s) issued[s] = -1;
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
            if (!valid) report(a.status, MQA_ERR_DEVICE_CHECK);
            const int nv = min(C::kTile, tend - t0);  // >= 1: the cursor only yields non-empty tiles
            mask_s[stage] = valid ? ((1ull << nv) - 1ull) : 0ull;
            mbar_arrive_expect_tx(&full[stage], valid ? 2u * pbytes : 0u);
            if (valid) {
                // slot t0 % P of page blk: plane 0 (K) then plane 1 (V), P rows later
                const uint8_t* src = a.kv + (static_cast<long long>(blk) * 2 * P + t0 % P) * rbytes;
                uint8_t* dst = stages + stage * sbytes;
                bulk_g2s(dst, src, pbytes, &full[stage], pol);
                bulk_g2s(dst + pbytes, src + static_cast<long long>(P) * rbytes, pbytes, &full[stage], pol);
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
    uint8_t* wk = smem + gk * C::kWBytes;
    uint8_t* wv = wk + C::kTile * C::kWStride;

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
#pragma unroll
                for (int i = 0; i < 4; ++i) qa[ks][i] = bf16x2_to_f16x2(qa[ks][i]);
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
                    ksc[i] = v ? *reinterpret_cast<const float*>(kb + tok * rbytes + D) : 0.f;
                    vsc[i] = v ? *reinterpret_cast<const float*>(vb + tok * rbytes + D) : 0.f;
                } else {
                    ksc[i] = 1.f;
                    vsc[i] = 1.f;
                }
            }
            __syncwarp();  // the previous tile's ldmatrix reads of wk / wv are done
            widen_rows<D, KIND>(kb, wk, vmask, rbytes, lane);
            widen_rows<D, KIND>(vb, wv, vmask, rbytes, lane);
            __syncwarp();
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

            float s[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int row = (lane & 7) + ((lane >> 4) << 3);
                const int col = ks * 16 + ((lane >> 3) & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, wk + row * C::kWStride + col * 2);
                mma_f16_16816(s[0], qa[ks], b0, b1);
                mma_f16_16816(s[1], qa[ks], b2, b3);
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
                // l sums the fp32 probabilities; P.V takes them times the V
                // scale of their token and 2^-e_run, rounded to f16
                const float p0 = ex2(x[nb][0] - m_use[0]), p1 = ex2(x[nb][1] - m_use[0]);
                const float p2 = ex2(x[nb][2] - m_use[1]), p3 = ex2(x[nb][3] - m_use[1]);
                l_part[0] += p0 + p1;
                l_part[1] += p2 + p3;
                pa[2 * nb] = pack_f16x2(p0 * vsc[2 * nb], p1 * vsc[2 * nb + 1]);
                pa[2 * nb + 1] = pack_f16x2(p2 * vsc[2 * nb], p3 * vsc[2 * nb + 1]);
            }
            const float oa0 = alpha[0] * o_fix, oa1 = alpha[1] * o_fix;
#pragma unroll
            for (int i = 0; i < C::kNb; ++i) {
                o[i][0] *= oa0;
                o[i][1] *= oa0;
                o[i][2] *= oa1;
                o[i][3] *= oa1;
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

template <int D, int KIND>
cudaError_t launch_q8(const GqaArgs& a, float out_scale, int grid, cudaStream_t stream) {
    using C = GqaQ8Cfg<D, KIND>;
    const size_t smem = C::smem_bytes(a.Hkv, a.plan.batch);
    auto kern = gqa_decode_q8_kernel<D, KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(grid), dim3(32 * (a.Hkv + 1)), smem, stream, a, out_scale);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_q8_kind(const GqaArgs& a, float out_scale, int kind, int grid, cudaStream_t stream) {
    if (kind == kFmtE4m3Pth) return launch_q8<D, kFmtE4m3Pth>(a, out_scale, grid, stream);
    if (kind == kFmtInt8Pth) return launch_q8<D, kFmtInt8Pth>(a, out_scale, grid, stream);
    return launch_q8<D, kFmtE4m3>(a, out_scale, grid, stream);
}

template <int D>
size_t smem_kind(int kind, int hkv, int batch) {
    if (kind == kFmtE4m3Pth) return GqaQ8Cfg<D, kFmtE4m3Pth>::smem_bytes(hkv, batch);
    if (kind == kFmtInt8Pth) return GqaQ8Cfg<D, kFmtInt8Pth>::smem_bytes(hkv, batch);
    return GqaQ8Cfg<D, kFmtE4m3>::smem_bytes(hkv, batch);
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
