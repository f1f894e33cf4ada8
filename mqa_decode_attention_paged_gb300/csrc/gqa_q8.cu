// GQA paged decode, stage 1, over 8-bit caches.
//
// Formats ("Triton と MLA" page, vllm-arch-zh ja/attention/triton-mla: 役割 and
// 設計動機 list the Triton backend's quantised KV cache dtypes, 主要ファイル
// says the per_token_head modes pad head_dim to hold an inline scale):
//   * e4m3 codes with one k_scale and one v_scale for the whole cache,
//     [num_blocks, 2, page, Hkv, D] bytes;
//   * per-token-head e4m3 or int8 codes, [num_blocks, 2, page, Hkv, D + 4]
//     bytes, or int4 codes two per byte, [num_blocks, 2, page, Hkv, D/2 + 4]:
//     each (token, KV head) row holds its codes followed by its own scale
//     (little-endian fp32); element value = scale * code.
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
constexpr int kFmtInt4Pth = MQA_KV_INT4_PER_TOKEN_HEAD;

template <int D, int KIND>
struct GqaQ8Cfg {
    static constexpr bool kPth = KIND != kFmtE4m3;
    static constexpr int kTile = 16;
    static constexpr int kMaxKvHeads = 8;
    static constexpr int kCodeBytes = KIND == kFmtInt4Pth ? D / 2 : D;  // codes of one row (int4: 2 per byte)
    static constexpr int kDp = kPth ? kCodeBytes + 4 : D;  // bytes of one (token, KV head) row
    static constexpr int kKSteps = D / 16;
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

// Transpose of an 8x8 matrix of 16-bit values held in the MMA fragment
// layout (lane i: row i / 4, columns 2 (i % 4) and + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) { return h2_bits(__floats2half2_rn(lo, hi)); }

// A bf16 pair -> the f16 pair of the same values (exact inside the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    return pack_f16x2(f.x, f.y);
}

// The eight int4 codes of w (nibble i = element i, two's complement) -> four
// f16 pairs, elements (0, 4), (1, 5), (2, 6), (3, 7), exact.  One
// mask-and-xor per pair (a single LOP3) puts x + 8 = nibble ^ 8 of elements
// i and i + 4 into the mantissas of two f16 1024s (0x6400): a nibble in bits
// 0..3 of a half gives 1024 + (x + 8), so 1032 is subtracted; a nibble in
// bits 4..7 gives 1024 + 16 (x + 8), so the pair is scaled by 1/16 and 72
// subtracted in one fused step (every value is an integer below 2048: no
// rounding).  Elements 2, 3, 6 and 7 take the same two steps after one shift
// by 8.  The callers absorb the element order (the K operand's reduction
// order, V's tile columns).
// Elements (0, 4) and (1, 5) of w.
__device__ __forceinline__ uint2 int4_lo_pairs(uint32_t w) {
    const __half2 k = bits_h2(0x64086408u);
    const __half2 s16 = __float2half2_rn(0.0625f), k72 = __float2half2_rn(-72.f);
    return make_uint2(h2_bits(__hsub2(bits_h2((w & 0x000f000fu) ^ 0x64086408u), k)),
                      h2_bits(__hfma2(bits_h2((w & 0x00f000f0u) ^ 0x64806480u), s16, k72)));
}
// Elements (2, 6) and (3, 7) of w.
__device__ __forceinline__ uint2 int4_hi_pairs(uint32_t w) { return int4_lo_pairs(w >> 8); }
__device__ __forceinline__ uint4 int4x8_to_f16_pairs(uint32_t w) {
    const uint2 lo = int4_lo_pairs(w), hi = int4_hi_pairs(w);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

// Tile column m (0..7) of an 8-column group of widened int4 V holds element
// perm(m) of the group: the order int4x8_to_f16_pairs stores.
__device__ __forceinline__ int int4_col_dim(int m) { return (m >> 1) + 4 * (m & 1); }

// Four 8-bit codes (bytes of w, lowest first) -> four f16 values (exact).
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

// Widen one KV head's 16 rows of codes (src: the head's first code byte in
// the plane tile, rows `rbytes` apart) into an f16 tile with row stride
// kWStride.  e4m3: rows of tokens not in vmask become zeros without reading
// their bytes (a stale or padding byte may be a NaN code).  int8 and int4:
// every byte is a finite code, and a masked token's P and V scale are 0, so
// its row is widened as it stands.
template <int D, int KIND>
__device__ __forceinline__ void widen_rows(const uint8_t* src, uint8_t* dst, uint64_t vmask, int rbytes,
                                           int lane) {
    using C = GqaQ8Cfg<D, KIND>;
    if constexpr (KIND == kFmtInt4Pth) {
        // a lane takes 4 bytes = 8 elements of a row; the tile's 8 columns
        // from 8 ch hold them in the order of int4x8_to_f16_pairs
        constexpr int kLanesPerRow = D / 8;
        constexpr int kRowsPer = 32 / kLanesPerRow;
        const int sub = lane / kLanesPerRow, ch = lane % kLanesPerRow;
#pragma unroll
        for (int r0 = 0; r0 < C::kTile; r0 += kRowsPer) {
            const int r = r0 + sub;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(src + r * rbytes + 4 * ch);
            *reinterpret_cast<uint4*>(dst + r * C::kWStride + 16 * ch) = int4x8_to_f16_pairs(w);
        }
    } else {
        constexpr int kLanesPerRow = D / 4;
        constexpr int kRowsPer = 32 / kLanesPerRow;
        const int sub = lane / kLanesPerRow, ch = lane % kLanesPerRow;
#pragma unroll
        for (int r0 = 0; r0 < C::kTile; r0 += kRowsPer) {
            const int r = r0 + sub;
            const bool v = KIND == kFmtInt8Pth || ((vmask >> r) & 1ull);
            const uint32_t w = v ? *reinterpret_cast<const uint32_t*>(src + r * rbytes + 4 * ch) : 0u;
            *reinterpret_cast<uint2*>(dst + r * C::kWStride + 8 * ch) = widen4<KIND>(w);
        }
    }
}

// Exponent e with vmax < 2^e (vmax > 0, finite): the power of two that P
// times a V scale is divided by.
__device__ __forceinline__ int scale_exponent(float vmax) {
    int e;
    frexpf(vmax, &e);  // vmax = f * 2^e, 0.5 <= f < 1
    return e;
}

// Resident blocks per SM: two when a KV head serves up to 8 query heads (one
// head block: 96 registers a thread suffice), one for up to 16.
__host__ __device__ constexpr int q8_ctas(int nhb) { return nhb == 1 ? 2 : 1; }

// NHB: head blocks of 8 query heads per KV head (1 for up to 8, 2 for up to 16).
template <int D, int KIND, int NHB>
__global__ void __launch_bounds__(32 * (GqaQ8Cfg<D, KIND>::kMaxKvHeads + 1), q8_ctas(NHB))
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
        // Block ids 32 pages at a time: lane l holds the id of page base + l of
        // the current piece, and the next 32 are loaded one chunk ahead, so
        // a tile never waits for a block-table read (with 16-token pages every
        // tile is a new page).
        int cur_b = -1, base = 0, jend = 0, ids = 0, nids = 0;
        auto load_chunk = [&](int j0) {
            return j0 + lane < jend ? __ldg(cur.bt + j0 + lane) : -1;
        };
        while (cur.next(a.plan, cum, lens, a.block_table)) {
            const int t0 = cur.t0, tend = cur.tok_end;
            const int j = t0 / P;
            if (cur.pc.b != cur_b || cur.pc.j1 != jend || j < base) {  // new piece
                cur_b = cur.pc.b;
                jend = cur.pc.j1;
                base = j;
                ids = load_chunk(base);
                nids = load_chunk(base + 32);
            } else if (j >= base + 32) {
                base += 32;
                ids = nids;
                nids = load_chunk(base + 32);
            }
            const int blk = __shfl_sync(0xffffffffu, ids, j - base);
            // warp-uniform decision: the lanes continue or leave together
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                break;
            }
            const bool valid = blk >= 0 && blk < a.num_blocks;
            const int nv = min(C::kTile, tend - t0);  // >= 1: the cursor only yields non-empty tiles
            // slot t0 % P of page blk: plane 0 (K), plane 1 (V) P rows later
            const uint8_t* src = a.kv + (static_cast<long long>(valid ? blk : 0) * 2 * P + t0 % P) * rbytes;
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
        }
        for (int s = 0; s < nstage; ++s)
            if (issued[s] >= 0 && !mbar_wait(&full[s], static_cast<uint32_t>(issued[s])))
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        return;
    }

    // ------------------------------------------------------------- consumers
    // Tokens are the MMA's M dimension: S^T = K Q^T (M = 16 tokens, N = 8
    // query heads per head block, K = head dims) and O^T = V^T P^T (M = 16
    // head dims per block, N = 8 heads, K = 16 tokens).  Lane (g, c) holds
    // tokens g and g + 8 and heads 2c, 2c + 1 of S^T, and head dims
    // 16 mb + g, + 8 of O^T.
    const int gk = warp;  // KV head
    const int g = lane >> 2, c = lane & 3;
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

        // Q^T operand, f16, in the permuted reduction order (step ks, lane c:
        // head dims 16 ks + 4c .. + 3; int4: steps 2j and 2j + 1 take dims
        // 32 j + 8c + (0, 4, 1, 5) and + (2, 6, 3, 7), the order in which
        // int4x8_to_f16_pairs widens one 4-byte word of K codes): query head
        // hb * 8 + g
        uint32_t qb[NHB][C::kKSteps][2];
        {
            const __nv_bfloat16* qrow = a.q + (static_cast<long long>(pc.b) * a.Hq + hq0) * D;
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb) {
                const int h = hb * 8 + g;
                if constexpr (KIND == kFmtInt4Pth) {
#pragma unroll
                    for (int j = 0; j < C::kKSteps / 2; ++j) {
                        const uint4 v = h < grp ? *reinterpret_cast<const uint4*>(qrow + h * D + j * 32 + 8 * c)
                                                : make_uint4(0u, 0u, 0u, 0u);
                        qb[hb][2 * j][0] = bf16x2_to_f16x2(__byte_perm(v.x, v.z, 0x5410));      // dims 0, 4
                        qb[hb][2 * j][1] = bf16x2_to_f16x2(__byte_perm(v.x, v.z, 0x7632));      // 1, 5
                        qb[hb][2 * j + 1][0] = bf16x2_to_f16x2(__byte_perm(v.y, v.w, 0x5410));  // 2, 6
                        qb[hb][2 * j + 1][1] = bf16x2_to_f16x2(__byte_perm(v.y, v.w, 0x7632));  // 3, 7
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < C::kKSteps; ++ks) {
                        const uint2 v = h < grp ? *reinterpret_cast<const uint2*>(qrow + h * D + ks * 16 + 4 * c)
                                                : make_uint2(0u, 0u);
                        qb[hb][ks][0] = bf16x2_to_f16x2(v.x);
                        qb[hb][ks][1] = bf16x2_to_f16x2(v.y);
                    }
                }
            }
        }
        float o[NHB][C::kKSteps][4];  // O^T: head dims 16 mb + g (0, 1) and + 8 (2, 3); heads 2c, 2c + 1
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
            for (int mb = 0; mb < C::kKSteps; ++mb) o[hb][mb][0] = o[hb][mb][1] = o[hb][mb][2] = o[hb][mb][3] = 0.f;
        float m_run[NHB][2], l_part[NHB][2];  // per head 2c + j of each head block
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
            m_run[hb][0] = m_run[hb][1] = -INFINITY;
            l_part[hb][0] = l_part[hb][1] = 0.f;
        }
        int e_run = -1000000;  // exponent of the P . V factor 2^-e (per-token-head scales)
        float p_fac = 1.f;     // 2^-e_run

        for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
            // warp-uniform: the lanes go on or leave together (the MMAs and
            // shuffles below are warp-collective); a tile that never arrived
            // is not read, but its stage is still handed back
            if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase))) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                aborted = true;
                break;
            }
            const uint8_t* kb = stages + stage * sbytes + hoff;
            const uint8_t* vb = kb + pbytes;
            const uint64_t vmask = mask_s[stage];
            const bool v0 = (vmask >> g) & 1ull, v1 = (vmask >> (g + 8)) & 1ull;

            // K and V scales of this lane's tokens g, g + 8 (0 when masked)
            float ks0 = 1.f, ks1 = 1.f, vs0 = 1.f, vs1 = 1.f;
            if constexpr (C::kPth) {
                ks0 = v0 ? *reinterpret_cast<const float*>(kb + g * rstride + C::kCodeBytes) : 0.f;
                ks1 = v1 ? *reinterpret_cast<const float*>(kb + (g + 8) * rstride + C::kCodeBytes) : 0.f;
                vs0 = v0 ? *reinterpret_cast<const float*>(vb + g * rstride + C::kCodeBytes) : 0.f;
                vs1 = v1 ? *reinterpret_cast<const float*>(vb + (g + 8) * rstride + C::kCodeBytes) : 0.f;
            }
            __syncwarp();  // the previous tile's ldmatrix reads of wv are done
            widen_rows<D, KIND>(vb, wv, vmask, rstride, lane);

            // S^T = K Q^T; A = the codes of tokens g and g + 8, one 4-byte read
            // each per step (masked tokens' rows are discarded below); two
            // accumulators per head block halve the dependent MMA chain
            float st[NHB][2][4];
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
                for (int e = 0; e < 2; ++e) st[hb][e][0] = st[hb][e][1] = st[hb][e][2] = st[hb][e][3] = 0.f;
            uint32_t w0 = 0u, w1 = 0u;  // int4: one word of codes per two steps
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                uint2 k0, k1;
                if constexpr (KIND == kFmtInt4Pth) {  // 8 elements = 4 bytes per two steps
                    if ((ks & 1) == 0) {
                        w0 = *reinterpret_cast<const uint32_t*>(kb + g * rstride + ks * 8 + 4 * c);
                        w1 = *reinterpret_cast<const uint32_t*>(kb + (g + 8) * rstride + ks * 8 + 4 * c);
                    }
                    k0 = (ks & 1) ? int4_hi_pairs(w0) : int4_lo_pairs(w0);
                    k1 = (ks & 1) ? int4_hi_pairs(w1) : int4_lo_pairs(w1);
                } else {
                    k0 = widen4<KIND>(*reinterpret_cast<const uint32_t*>(kb + g * rstride + ks * 16 + 4 * c));
                    k1 = widen4<KIND>(*reinterpret_cast<const uint32_t*>(kb + (g + 8) * rstride + ks * 16 + 4 * c));
                }
                const uint32_t af[4] = {k0.x, k1.x, k0.y, k1.y};
#pragma unroll
                for (int hb = 0; hb < NHB; ++hb) mma_f16_16816(st[hb][ks & 1], af, qb[hb][ks][0], qb[hb][ks][1]);
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
                float vmax = fmaxf(fabsf(vs0), fabsf(vs1));
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 4));
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 8));
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 16));
                if (vmax > 0.f && vmax <= 3.0e38f) {
                    const int e = scale_exponent(vmax);
                    if (e > e_run) {
                        o_fix = e_run == -1000000 ? 1.f : ldexpf(1.f, e_run - e);
                        e_run = e;
                        p_fac = ldexpf(1.f, -e);
                    }
                }
                vs0 *= p_fac;
                vs1 *= p_fac;
            }
            const float kx0 = ks0 * a.sl2, kx1 = ks1 * a.sl2;

            // online softmax per head (column of S^T), over the 16 tokens
            uint32_t pb[NHB][2];
            float alpha[NHB][2];
            bool grow = false;
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb) {
                float x[4];
                x[0] = v0 ? (st[hb][0][0] + st[hb][1][0]) * kx0 : -INFINITY;  // token g, head 2c
                x[1] = v0 ? (st[hb][0][1] + st[hb][1][1]) * kx0 : -INFINITY;  // token g, head 2c + 1
                x[2] = v1 ? (st[hb][0][2] + st[hb][1][2]) * kx1 : -INFINITY;  // token g + 8, head 2c
                x[3] = v1 ? (st[hb][0][3] + st[hb][1][3]) * kx1 : -INFINITY;
                float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
                    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
                    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
                    alpha[hb][j] = 1.f;
                    // lazy: move the reference only when P would exceed 2^8
                    if (mx[j] > m_run[hb][j] + 8.f) {
                        alpha[hb][j] = ex2(m_run[hb][j] - mx[j]);
                        m_run[hb][j] = mx[j];
                        l_part[hb][j] *= alpha[hb][j];
                        grow = true;
                    }
                }
                const float mu0 = m_run[hb][0] == -INFINITY ? 0.f : m_run[hb][0];
                const float mu1 = m_run[hb][1] == -INFINITY ? 0.f : m_run[hb][1];
                const float p0 = ex2(x[0] - mu0), p1 = ex2(x[1] - mu1);
                const float p2 = ex2(x[2] - mu0), p3 = ex2(x[3] - mu1);
                // l sums the fp32 probabilities; P.V takes them times the V
                // scale of their token and 2^-e_run, rounded to f16
                l_part[hb][0] += p0 + p2;
                l_part[hb][1] += p1 + p3;
                // P^T rows g and g + 8 -> the B operand (tokens 2c, 2c + 1 and
                // 2c + 8, 2c + 9 of head g) by an 8x8 transpose each
                pb[hb][0] = movmatrix_t(pack_f16x2(p0 * vs0, p1 * vs0));
                pb[hb][1] = movmatrix_t(pack_f16x2(p2 * vs1, p3 * vs1));
            }
            if (__any_sync(0xffffffffu, grow) || o_fix != 1.f) {
#pragma unroll
                for (int hb = 0; hb < NHB; ++hb) {
                    const float f0 = alpha[hb][0] * o_fix, f1 = alpha[hb][1] * o_fix;
#pragma unroll
                    for (int mb = 0; mb < C::kKSteps; ++mb) {
                        o[hb][mb][0] *= f0;
                        o[hb][mb][1] *= f1;
                        o[hb][mb][2] *= f0;
                        o[hb][mb][3] *= f1;
                    }
                }
            }
            // O^T += V^T P^T: A = V^T from the widened tile (16 head dims x 16
            // tokens per ldmatrix.x4.trans), B = P^T
#pragma unroll
            for (int mb = 0; mb < C::kKSteps; ++mb) {
                const int q = lane >> 3;
                const int tok = (lane & 7) + (q >> 1) * 8;
                const int col = mb * 16 + (q & 1) * 8;
                uint32_t av[4];
                ldsm_x4_t(av[0], av[1], av[2], av[3], wv + tok * C::kWStride + col * 2);
#pragma unroll
                for (int hb = 0; hb < NHB; ++hb) mma_f16_16816(o[hb][mb], av, pb[hb][0], pb[hb][1]);
            }
        }
        if (aborted) break;

        // epilogue: head hb * 8 + 2c + j, head dims 16 mb + dg (+ 8); int4 V
        // tiles hold their columns in int4x8_to_f16_pairs order
        const int dg = KIND == kFmtInt4Pth ? int4_col_dim(g) : g;
        const float osc = (C::kPth && e_run != -1000000) ? ldexpf(out_scale, e_run) : out_scale;
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
            float inv[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float l = l_part[hb][j];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                inv[j] = l > 0.f ? osc / l : 0.f;
                const int h = hb * 8 + 2 * c + j;
                if (g == 0 && h < grp) {
                    const float lse = l > 0.f ? (m_run[hb][j] + log2f(l)) * kLn2 : -INFINITY;
                    if (pc.whole) {
                        if (a.lse) a.lse[static_cast<long long>(pc.b) * a.Hq + hq0 + h] = lse;
                    } else {
                        a.ws_lse[static_cast<long long>(pc.slot) * a.Hq + hq0 + h] = lse;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = hb * 8 + 2 * c + j;
                if (h >= grp) continue;
                if (pc.whole) {
                    __nv_bfloat16* orow = a.out + (static_cast<long long>(pc.b) * a.Hq + hq0 + h) * D;
#pragma unroll
                    for (int mb = 0; mb < C::kKSteps; ++mb) {
                        orow[mb * 16 + dg] = __float2bfloat16_rn(o[hb][mb][j] * inv[j]);
                        orow[mb * 16 + dg + 8] = __float2bfloat16_rn(o[hb][mb][2 + j] * inv[j]);
                    }
                } else {
                    float* wrow = a.ws_o + (static_cast<long long>(pc.slot) * a.Hq + hq0 + h) * D;
#pragma unroll
                    for (int mb = 0; mb < C::kKSteps; ++mb) {
                        wrow[mb * 16 + dg] = o[hb][mb][j] * inv[j];
                        wrow[mb * 16 + dg + 8] = o[hb][mb][2 + j] * inv[j];
                    }
                }
            }
        }
    }
}

// Dynamic shared memory a block may use: 227 KB on sm_103a, or its share of
// the SM's 228 KB (less 1 KB reserved per block) with several blocks per SM.
constexpr size_t smem_limit(int ctas) { return ctas == 1 ? 227 * 1024 : (228 * 1024) / ctas - 1024; }

template <int D, int KIND>
cudaError_t launch_q8(const GqaArgs& a, float out_scale, int grid, cudaStream_t stream) {
    using C = GqaQ8Cfg<D, KIND>;
    const int nhb = (a.Hq / a.Hkv) <= 8 ? 1 : 2;
    const int ns = C::stages_for(a.Hkv, a.plan.batch, smem_limit(q8_ctas(nhb)));
    const size_t smem = C::smem_bytes(a.Hkv, ns, a.plan.batch);
    auto kern = nhb == 1 ? gqa_decode_q8_kernel<D, KIND, 1> : gqa_decode_q8_kernel<D, KIND, 2>;
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
    if (kind == kFmtInt4Pth) return launch_q8<D, kFmtInt4Pth>(a, out_scale, grid, stream);
    return launch_q8<D, kFmtE4m3>(a, out_scale, grid, stream);
}

template <int D, int KIND>
size_t smem_of(int hkv, int q_per_kv, int batch) {
    using C = GqaQ8Cfg<D, KIND>;
    const int ctas = q8_ctas(q_per_kv <= 8 ? 1 : 2);
    return C::smem_bytes(hkv, C::stages_for(hkv, batch, smem_limit(ctas)), batch);
}

template <int D>
size_t smem_kind(int kind, int hkv, int q_per_kv, int batch) {
    if (kind == kFmtE4m3Pth) return smem_of<D, kFmtE4m3Pth>(hkv, q_per_kv, batch);
    if (kind == kFmtInt8Pth) return smem_of<D, kFmtInt8Pth>(hkv, q_per_kv, batch);
    if (kind == kFmtInt4Pth) return smem_of<D, kFmtInt4Pth>(hkv, q_per_kv, batch);
    return smem_of<D, kFmtE4m3>(hkv, q_per_kv, batch);
}

}  // namespace

cudaError_t gqa_q8_stage1(const GqaArgs& a, float out_scale, int D, int kind, int grid, cudaStream_t stream) {
    if (D == 128) return launch_q8_kind<128>(a, out_scale, kind, grid, stream);
    return launch_q8_kind<64>(a, out_scale, kind, grid, stream);
}

int gqa_q8_ctas_per_sm(int q_per_kv) { return q8_ctas(q_per_kv <= 8 ? 1 : 2); }

size_t gqa_q8_smem_bytes(int D, int kind, int hkv, int q_per_kv, int batch) {
    return D == 128 ? smem_kind<128>(kind, hkv, q_per_kv, batch) : smem_kind<64>(kind, hkv, q_per_kv, batch);
}

}  // namespace mqa
