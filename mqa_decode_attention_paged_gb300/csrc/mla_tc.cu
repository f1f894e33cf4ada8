// MLA decode, stage 1, fifth-generation tensor-core path for 65..128 heads.
//
// A thread-block cluster of two CTAs owns one work unit (plan.cuh) and splits
// the 576 (or 320) latent columns: rank 0 contracts Q.K^T over the first R/2
// columns and accumulates O[:, 0:R/2]; rank 1 contracts over the remaining
// columns (the rest of kv_c and all of k_pe) and accumulates O[:, R/2:R].  The
// V columns a rank needs are a prefix of the K columns it already loaded (V is
// the first kv_lora_rank columns of the same row: "Triton と MLA" page,
// vllm-arch-zh ja/attention/triton-mla, データフロー), so every cache byte is
// read from HBM once and TMEM holds O[128 x R/2] plus two logit tiles.  The
// two partial logit tiles are exchanged through distributed shared memory and
// summed identically in both CTAs, which then run the same online softmax
// (tutorial page lshu.cn/news/265860, §7).
//
// Per CTA (352 threads), for 32-token tiles grouped in pairs:
//   warp 0      TMA producer: the tile's rows of this CTA's column panels
//               (tensor-map copies, 128-byte swizzle) into a 4-stage ring laid
//               out as two 64-row slots, so that a pair of tiles is one
//               contiguous 64-row operand;
//   warp 1      TMEM owner and single-thread MMA issuer:
//               S[128 x 64] = Q K^T per tile pair (kind::f16, M = 128 heads,
//               N = 64 tokens) into one of two TMEM logit buffers, then per
//               tile O[128 x R/2] += P V (N = R/2, V read MN-major);
//   warps 2..9  two threads per head row (16 tokens of each tile, half of O's
//               columns each): read S from TMEM, send it to the peer
//               with asynchronous remote stores (lane-contiguous, double
//               buffered), add the peer's half, mask, online softmax in base 2
//               with lazy rescaling of O (only when the running max grows by
//               more than 2^8), write P (bf16, swizzled K-major; the two halves
//               of one 64-token tile alternate) and the epilogue;
//   warp 10     Q loader (the query rows of the current request).
// Every wait is bounded; on expiry MQA_ERR_DEVICE_TIMEOUT is recorded and the
// roles wind down.
#include "args.cuh"
#include "common.cuh"
#include "plan.cuh"
#include "tc_ptx.cuh"

namespace mqa {

template <int D, int R>
struct MlaTcCfg {
    static constexpr int kHeads = 128;
    static constexpr int kTile = 32;  // tokens per pipeline stage (a Q.K^T covers two)
    static constexpr int kPanels = D / 64;
    static constexpr int kLoPanels = R / 128;  // rank 0: QK panels = its P.V panels
    static constexpr int kHiPanels = kPanels - kLoPanels;
    static constexpr int kMaxPanels = kHiPanels;
    static constexpr int kOCols = R / 2;  // O columns per CTA
    static constexpr int kPVPanels = kOCols / 64;
    static constexpr int kStages = 4;
    static constexpr int kQPanelBytes = kHeads * 128;
    static constexpr int kKvPanelBytes = 2 * kTile * 128;  // one panel of a 64-row slot
    static constexpr int kQBytes = kMaxPanels * kQPanelBytes;
    static constexpr int kSlotBytes = kMaxPanels * kKvPanelBytes;  // two stages
    static constexpr int kPBytes = kHeads * 128;            // 128 rows x 64 tokens: two tile halves
    static constexpr int kXBytes = kHeads * kTile * 4;      // one fp32 logit tile
    static constexpr int kSoftmaxWarps = 8;  // two threads per head row
    static constexpr int kThreads = 32 * (3 + kSoftmaxWarps);
    static constexpr int kTmemCols = 512;
    static constexpr int kTmemS = 256;  // pair logit buffers at columns 256 and 320

    static constexpr int kOffQ = 0;
    static constexpr int kOffStages = kOffQ + kQBytes;
    static constexpr int kOffP = kOffStages + (kStages / 2) * kSlotBytes;
    static constexpr int kOffX = kOffP + kPBytes;
    static constexpr int kOffBars = kOffX + 2 * kXBytes;
    static constexpr int kNumBars = 32;
    static constexpr int kOffRed = kOffBars + kNumBars * 8;  // row maxima / sums of the two halves
    static constexpr int kRedBytes = 6 * kHeads * 4;
    static constexpr int kOffMask = kOffRed + kRedBytes;
    static constexpr int kOffTmem = kOffMask + kStages * 8;
    static constexpr int kOffCum = kOffTmem + 16;
    static size_t smem_bytes(int batch) { return 1024 + kOffCum + 4 * (2 * batch + 1); }

    static_assert(kOCols <= 256 && kOCols % 64 == 0, "P.V width");
    static_assert(kTmemS >= kOCols && kTmemS + 4 * kTile <= kTmemCols, "TMEM layout");
    static_assert(1024 + kOffCum + 4 * (2 * kMaxBatchTc + 1) <= 227 * 1024, "shared memory budget");
    static_assert(kOffStages % 1024 == 0 && kOffP % 1024 == 0 && kSlotBytes % 1024 == 0,
                  "swizzled operands need 1024-byte alignment");
};

// barrier slots
enum TcBar {
    kKvFull = 0,    // [4] tile landed (producer expect_tx + TMA bytes)
    kKvEmpty = 4,   // [4] P.V of the tile done (tensor-core commit)
    kQFull = 8,     // Q rows landed
    kQEmpty = 9,    // every Q.K^T of the piece done
    kSFull = 10,    // [2] logit tile pair in TMEM
    kSEmpty = 12,   // [2] both tiles of the pair read out by the softmax rows
    kPFull = 14,    // [2] P half written (and O rescaled)
    kPEmpty = 16,   // [2] P.V of that half done
    kXFull = 18,    // [2] the peer's logit tile has arrived
    kXFree = 20,    // [2] the peer has consumed the tile we sent it
    kPair = 22,     // [4] rendezvous of the two softmax warps of a TMEM quadrant
};

template <int D, int R>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MlaTcCfg<D, R>::kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ MlaTcArgs a) {
    using C = MlaTcCfg<D, R>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* q_s = smem + C::kOffQ;
    uint8_t* stages = smem + C::kOffStages;
    uint8_t* p_s = smem + C::kOffP;
    uint8_t* x_s = smem + C::kOffX;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
    uint64_t* mask_s = reinterpret_cast<uint64_t*>(smem + C::kOffMask);
    float* red_s = reinterpret_cast<float*>(smem + C::kOffRed);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);
    int* cum = reinterpret_cast<int*>(smem + C::kOffCum);
    int* lens = cum + a.plan.batch + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int unit = blockIdx.x >> 1;
    const int pbase = rank ? C::kLoPanels : 0;          // first global column panel
    const int np = rank ? C::kHiPanels : C::kLoPanels;  // panels loaded and contracted
    const int P = a.plan.page;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars[kKvFull + s], 1);
            mbar_init(&bars[kKvEmpty + s], 1);
        }
        mbar_init(&bars[kQFull], 1);
        mbar_init(&bars[kQEmpty], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kSFull + i], 1);
            mbar_init(&bars[kSEmpty + i], 2 * 32 * C::kSoftmaxWarps);  // both tiles of a pair
            mbar_init(&bars[kPFull + i], 32 * C::kSoftmaxWarps);
            mbar_init(&bars[kPEmpty + i], 1);
            mbar_init(&bars[kXFull + i], 1);  // own expect_tx; the bytes come from the peer
            mbar_init(&bars[kXFree + i], C::kSoftmaxWarps);  // one arrive per peer softmax warp
        }
        for (int q = 0; q < 4; ++q) mbar_init(&bars[kPair + q], 64);
        fence_mbar_init();
        prefetch_tmap(&a.kv_map);
        prefetch_tmap(&a.q_map);
    }
    if (warp == 1) tmem_alloc(tmem_base_s, C::kTmemCols);
    pdl_wait();
    pdl_launch_dependents();
    const int T = build_cum(a.plan, a.seq_lens, cum, lens, a.status);  // contains __syncthreads
    tc_fence_after();
    cluster_sync();  // the peer's barriers are initialised before any remote operation
    const uint32_t tbase = *tmem_base_s;

    // tiles of a piece: tokens [tok0, tok_end) of request pc.b, rounded up to
    // an even count (a trailing tile past tok_end is fully masked) so that
    // every piece starts on a slot boundary
    auto piece_tiles = [&](const Piece& pc, int& tok0, int& tok_end) {
        tok0 = pc.j0 * P;
        tok_end = min(pc.j1 * P, lens[pc.b]);
        const int n = tok_end > tok0 ? (tok_end - tok0 + C::kTile - 1) / C::kTile : 0;
        return (n + 1) & ~1;
    };
    // byte offset of tile t's rows (of panel 0) in the ring
    auto tile_base = [&](int t) {
        return ((t % C::kStages) >> 1) * C::kSlotBytes + (t & 1) * (C::kTile * 128);
    };

    if (warp == 0) {
        // ------------------------------------------------------ KV producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const int BR = a.box_rows, nbox = C::kTile / BR;
            PieceIter it;
            it.init(a.plan, cum, T, unit);
            Piece pc;
            int t = 0;
            int issued[C::kStages];
            for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
            bool ok = true;
            while (ok && it.next(cum, pc)) {
                int tok0, tok_end;
                const int nt = piece_tiles(pc, tok0, tok_end);
                const int32_t* bt = a.block_table + static_cast<long long>(pc.b) * a.plan.max_blocks;
                for (int j = 0; j < nt; ++j, ++t) {
                    const int t0 = tok0 + j * C::kTile;
                    int blk[2];
                    bool val[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int tok = t0 + k * BR;
                        val[k] = k < nbox && tok < tok_end;
                        blk[k] = val[k] ? bt[tok / P] : 0;
                    }
                    const int st = t % C::kStages;
                    if (!mbar_wait(&bars[kKvEmpty + st], ((t / C::kStages) & 1) ^ 1)) {
                        report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int n_tok = max(tok_end - t0, 0);
                    uint64_t vmask = n_tok >= C::kTile ? 0xFFFFFFFFull : ((1ull << n_tok) - 1);
                    const uint64_t ones = (1ull << BR) - 1;
                    int nvalid = 0;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        if (k >= nbox) break;
                        if (val[k] && (blk[k] < 0 || blk[k] >= a.num_blocks)) {
                            report(a.status, MQA_ERR_DEVICE_CHECK);
                            val[k] = false;
                        }
                        if (val[k])
                            ++nvalid;
                        else
                            vmask &= ~(ones << (k * BR));
                    }
                    mask_s[st] = vmask;
                    mbar_arrive_expect_tx(&bars[kKvFull + st], nvalid * BR * 128 * np);
                    uint8_t* dst = stages + tile_base(t);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        if (k >= nbox || !val[k]) continue;
                        const int row = blk[k] * P + (t0 + k * BR) % P;
                        for (int pn = 0; pn < np; ++pn)
                            tma_load_2d(dst + pn * C::kKvPanelBytes + k * BR * 128, &a.kv_map, (pbase + pn) * 64,
                                        row, &bars[kKvFull + st], pol);
                    }
                    issued[st] = (t / C::kStages) & 1;
                }
            }
            for (int s = 0; s < C::kStages; ++s)
                if (issued[s] >= 0 && !mbar_wait(&bars[kKvFull + s], static_cast<uint32_t>(issued[s])))
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == 2 + C::kSoftmaxWarps) {
        // ------------------------------------------------------ Q loader
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            PieceIter it;
            it.init(a.plan, cum, T, unit);
            Piece pc;
            int qc = 0;
            while (it.next(cum, pc)) {
                int tok0, tok_end;
                if (piece_tiles(pc, tok0, tok_end) == 0) continue;
                if (!mbar_wait(&bars[kQEmpty], (qc & 1) ^ 1)) {
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&bars[kQFull], np * C::kQPanelBytes);
                for (int pn = 0; pn < np; ++pn)
                    tma_load_2d(q_s + pn * C::kQPanelBytes, &a.q_map, (pbase + pn) * 64, pc.b * a.H,
                                &bars[kQFull], pol);
                ++qc;
            }
            if (qc > 0 && !mbar_wait(&bars[kQFull], (qc - 1) & 1)) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdQK = umma_idesc_bf16(128, 2 * C::kTile, 0);
            constexpr uint32_t kIdPV = umma_idesc_bf16(128, C::kOCols, 1);
            const uint32_t q_addr = smem_u32(q_s), st_addr = smem_u32(stages), p_addr = smem_u32(p_s);
            bool ok = true;
            int last_pv = -1;
            // Two independent streams, issued as soon as their inputs are ready:
            //   Q.K^T per tile pair (needs Q, both stages, a free S buffer),
            //   P.V per tile (needs its P half).
            PieceIter qi, vi;
            qi.init(a.plan, cum, T, unit);
            vi.init(a.plan, cum, T, unit);
            Piece qpc, vpc;
            int qt = 0, qj = 0, qnt = 0, qc = 0;  // next pair: global tile qt, piece tile qj
            int vt = 0, vj = 0, vnt = 0;          // next P.V: global tile vt, piece tile vj
            bool q_loaded = false;
            auto next_piece = [&](PieceIter& pi, Piece& pc, int& nt) {
                int tok0, tok_end;
                while (pi.next(cum, pc)) {
                    nt = piece_tiles(pc, tok0, tok_end);
                    if (nt > 0) return true;
                }
                return false;
            };
            bool q_have = next_piece(qi, qpc, qnt);
            bool v_have = next_piece(vi, vpc, vnt);
            unsigned long long idle_since = 0;
            while (q_have || v_have) {
                bool progressed = false;
                if (q_have) {
                    if (!q_loaded && mbar_test(&bars[kQFull], qc & 1)) {
                        q_loaded = true;
                        tc_fence_after();
                    }
                    const int sb = (qt >> 1) & 1;
                    if (q_loaded && mbar_test(&bars[kKvFull + qt % C::kStages], (qt / C::kStages) & 1) &&
                        mbar_test(&bars[kKvFull + (qt + 1) % C::kStages], ((qt + 1) / C::kStages) & 1) &&
                        mbar_test(&bars[kSEmpty + sb], ((qt >> 2) & 1) ^ 1)) {
                        tc_fence_after();
                        const uint32_t kaddr = st_addr + tile_base(qt);
                        for (int ks = 0; ks < np * 4; ++ks)
                            umma_bf16(tbase + C::kTmemS + sb * 2 * C::kTile,
                                      umma_desc(q_addr + (ks >> 2) * C::kQPanelBytes + (ks & 3) * 32, 16, 1024),
                                      umma_desc(kaddr + (ks >> 2) * C::kKvPanelBytes + (ks & 3) * 32, 16, 1024),
                                      kIdQK, ks > 0 ? 1u : 0u);
                        umma_commit(&bars[kSFull + sb]);
                        qt += 2;
                        qj += 2;
                        if (qj >= qnt) {
                            umma_commit(&bars[kQEmpty]);  // Q may be reloaded once these finish
                            ++qc;
                            q_loaded = false;
                            qj = 0;
                            q_have = next_piece(qi, qpc, qnt);
                        }
                        progressed = true;
                    }
                }
                if (v_have && vt < qt && mbar_test(&bars[kPFull + (vt & 1)], (vt >> 1) & 1)) {
                    tc_fence_after();
                    const int pb = vt & 1;
                    const uint32_t v = st_addr + tile_base(vt);
#pragma unroll
                    for (int ks = 0; ks < C::kTile / 16; ++ks)
                        umma_bf16(tbase, umma_desc(p_addr + pb * 64 + ks * 32, 16, 1024),
                                  umma_desc(v + ks * 2048, C::kKvPanelBytes, 1024), kIdPV,
                                  (vj == 0 && ks == 0) ? 0u : 1u);
                    umma_commit(&bars[kPEmpty + pb]);
                    umma_commit(&bars[kKvEmpty + vt % C::kStages]);
                    last_pv = vt;
                    ++vt;
                    if (++vj >= vnt) {
                        vj = 0;
                        v_have = next_piece(vi, vpc, vnt);
                    }
                    progressed = true;
                }
                if (progressed) {
                    idle_since = 0;
                } else {
                    const unsigned long long now = global_timer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            // no tensor-core work may be in flight when the CTA tears down
            if (last_pv >= 0 && !mbar_wait(&bars[kPEmpty + (last_pv & 1)], (last_pv >> 1) & 1))
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp >= 2 && warp < 2 + C::kSoftmaxWarps) {
        // ------------------------------------------------------ softmax rows
        // Two threads per head row: warps w and w + 4 share TMEM lane quadrant
        // w % 4 and split every tile's 32 tokens (and O's columns) in halves.
        const int quad = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int h = quad * 32 + lane;
        const int tc0 = hf * (C::kTile / 2);
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quad * 32) << 16);
        float* mx_s = red_s;                   // [2 tiles][2 halves][128 rows] partial maxima
        float* ls_s = red_s + 4 * C::kHeads;  // [2 halves][128 rows] partial sums
        uint64_t* pair_bar = &bars[kPair + quad];
        uint32_t pair_phase = 0;
        // logit tiles travel lane-contiguously: chunk c (4 floats) of row
        // (quad, lane) sits at ((quad * 8 + c) * 32 + lane) * 16 bytes, so every
        // warp store writes 512 contiguous bytes of the peer's buffer
        const uint32_t x_remote = map_to_rank(x_s, peer) + (quad * 8 * 32 + lane) * 16;
        const uint8_t* x_local = x_s + (quad * 8 * 32 + lane) * 16;
        const uint32_t xfull_remote[2] = {map_to_rank(&bars[kXFull], peer), map_to_rank(&bars[kXFull + 1], peer)};
        const uint32_t xfree_remote[2] = {map_to_rank(&bars[kXFree], peer), map_to_rank(&bars[kXFree + 1], peer)};
        uint8_t* p_row = p_s + h * 128;
        // warp-uniform bounded waits: TMEM accesses are warp-collective, so a
        // lane never leaves the tile loop on its own
        auto wait_all = [&](uint64_t* bar, uint32_t parity, bool cluster_scope) {
            const bool done = cluster_scope ? mbar_wait_cluster(bar, parity) : mbar_wait(bar, parity);
            return __all_sync(0xffffffffu, done);
        };
        // rendezvous of the two warps that own the same rows
        auto pair_sync = [&]() {
            mbar_arrive(pair_bar);
            const bool done = wait_all(pair_bar, pair_phase, false);
            pair_phase ^= 1;
            return done;
        };

        PieceIter it;
        it.init(a.plan, cum, T, unit);
        Piece pc;
        int t = 0;
        bool ok = true;
        while (ok && it.next(cum, pc)) {
            int tok0, tok_end;
            const int nt = piece_tiles(pc, tok0, tok_end);
            const bool live_row = h < a.H;
            const int ocol0 = hf * (C::kOCols / 2);  // this thread's half of O's columns
            if (nt == 0) {  // empty request (per-request mode): out = 0, lse = -inf
                if (live_row && pc.whole) {
                    __nv_bfloat16* o =
                        a.out + (static_cast<long long>(pc.b) * a.H + h) * R + rank * C::kOCols + ocol0;
                    for (int c = 0; c < C::kOCols / 2; c += 8)
                        *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
                    if (rank == 0 && hf == 0 && a.lse) a.lse[static_cast<long long>(pc.b) * a.H + h] = -INFINITY;
                }
                continue;
            }
            float m_run = -INFINITY, l_part = 0.f;
            for (int j = 0; j < nt; ++j, ++t) {
                const int sb = (t >> 1) & 1, xb = t & 1, pb = t & 1, st = t % C::kStages;
                constexpr int kHalfTok = C::kTile / 2;
                float s[kHalfTok];
                if (!wait_all(&bars[kSFull + sb], (t >> 2) & 1, false)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t r[16];
                    tmem_ld16(lane_addr + C::kTmemS + sb * 2 * C::kTile + (t & 1) * C::kTile + tc0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < kHalfTok; ++i) s[i] = __uint_as_float(r[i]);
                }
                tc_fence_before();
                mbar_arrive(&bars[kSEmpty + sb]);

                // send our partial logits, receive and add the peer's
                if (h == 0 && hf == 0) mbar_arrive_expect_tx(&bars[kXFull + xb], C::kXBytes);
                if (t >= 2 && !wait_all(&bars[kXFree + xb], ((t >> 1) & 1) ^ 1, true)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < kHalfTok / 4; ++c)
                    st_async_v4(x_remote + xb * C::kXBytes + (hf * 4 + c) * 512, s[4 * c], s[4 * c + 1],
                                s[4 * c + 2], s[4 * c + 3], xfull_remote[xb]);
                if (!wait_all(&bars[kXFull + xb], (t >> 1) & 1, true)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < kHalfTok / 4; ++c) {
                    const float4 v = *reinterpret_cast<const float4*>(x_local + xb * C::kXBytes + (hf * 4 + c) * 512);
                    s[4 * c] += v.x;
                    s[4 * c + 1] += v.y;
                    s[4 * c + 2] += v.z;
                    s[4 * c + 3] += v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(xfree_remote[xb]);

                // valid tokens of this tile (set by the producer before kv_full)
                if (!wait_all(&bars[kKvFull + st], (t / C::kStages) & 1, false)) {
                    ok = false;
                    break;
                }
                const uint64_t vmask = mask_s[st];
                float lm = -INFINITY;
#pragma unroll
                for (int i = 0; i < kHalfTok; ++i) {
                    s[i] = ((vmask >> (tc0 + i)) & 1ull) ? s[i] * a.sl2 : -INFINITY;
                    lm = fmaxf(lm, s[i]);
                }
                // row maximum of the tile: combine the two halves
                mx_s[((t & 1) * 2 + hf) * C::kHeads + h] = lm;
                if (!pair_sync()) {
                    ok = false;
                    break;
                }
                float mt = fmaxf(lm, mx_s[((t & 1) * 2 + (1 - hf)) * C::kHeads + h]);
                // the half of P this tile writes was last read by P.V(t-2)
                bool half_free = (j == 0) || (t < 2);  // at a piece start the epilogue already waited
                if (j == 0) {
                    m_run = mt;
                } else if (__any_sync(0xffffffffu, mt > m_run + 8.f)) {
                    // the running max grew by more than 2^8 (decided per warp; the
                    // partner warp holds the same rows and decides alike; rows
                    // whose max did not grow rescale by 1): wait for P.V(t-1),
                    // rescale this thread's half of O and its partial sum
                    mt = fmaxf(mt, m_run);
                    const float alpha = ex2(m_run - mt);
                    if (!wait_all(&bars[kPEmpty + ((t - 1) & 1)], ((t - 1) >> 1) & 1, false)) {
                        ok = false;
                        break;
                    }
                    half_free = true;
                    tc_fence_after();
                    for (int c0 = ocol0; c0 < ocol0 + C::kOCols / 2; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(lane_addr + c0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(lane_addr + c0, r);
                    }
                    tmem_wait_st();
                    l_part *= alpha;
                    m_run = mt;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                uint32_t pk[kHalfTok / 2];
                float psum = 0.f;
#pragma unroll
                for (int i = 0; i < kHalfTok / 2; ++i) {
                    const float p0 = ex2(s[2 * i] - m_use), p1 = ex2(s[2 * i + 1] - m_use);
                    psum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                l_part += psum;
                if (!half_free && !wait_all(&bars[kPEmpty + pb], ((t >> 1) & 1) ^ 1, false)) {
                    ok = false;
                    break;
                }
                // rows past the sequence end: zero their V columns in the stage
                if (vmask != 0xFFFFFFFFull) {
                    const int idx = hf * C::kHeads + h;
                    const int r = idx & (C::kTile - 1), pn = idx / C::kTile;
                    if (pn < C::kPVPanels && !((vmask >> r) & 1ull)) {
                        uint8_t* base = stages + tile_base(t) + r * 128 + pn * C::kKvPanelBytes;
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(base + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                // P row h, K-major with the 128-byte swizzle: this tile fills the
                // 16-byte chunks 4 * pb .. 4 * pb + 3 of the row, this thread two
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    *reinterpret_cast<uint4*>(p_row + (((4 * pb + 2 * hf + c) ^ (h & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[kPFull + pb]);
            }
            if (!ok) break;

            // epilogue: O / l for this thread's half of the CTA's columns
            if (!wait_all(&bars[kPEmpty + ((t - 1) & 1)], ((t - 1) >> 1) & 1, false)) {
                ok = false;
                break;
            }
            ls_s[hf * C::kHeads + h] = l_part;
            if (!pair_sync()) {
                ok = false;
                break;
            }
            const float l_run = l_part + ls_s[(1 - hf) * C::kHeads + h];
            tc_fence_after();
            const float inv = l_run > 0.f ? a.out_scale / l_run : 0.f;
            for (int c0 = ocol0; c0 < ocol0 + C::kOCols / 2; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_addr + c0, r);
                tmem_wait_ld();
                if (!live_row) continue;
                const int col = rank * C::kOCols + c0;
                if (pc.whole) {
                    __nv_bfloat16* o = a.out + (static_cast<long long>(pc.b) * a.H + h) * R + col;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(r[i + 4]) * inv, __uint_as_float(r[i + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(r[i + 6]) * inv, __uint_as_float(r[i + 7]) * inv);
                        *reinterpret_cast<uint4*>(o + i) = w;
                    }
                } else {
                    float* o = a.ws_o + (static_cast<long long>(pc.slot) * a.H + h) * R + col;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(o + i) =
                            make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                        __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
                }
            }
            if (live_row && rank == 0 && hf == 0) {
                const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
                if (pc.whole) {
                    if (a.lse) a.lse[static_cast<long long>(pc.b) * a.H + h] = lse;
                } else {
                    a.ws_lse[static_cast<long long>(pc.slot) * a.H + h] = lse;
                }
            }
        }
        if (!ok) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
    }

    // teardown: every role is done with TMEM, shared memory and the peer's
    // shared memory before the allocation is returned and the CTAs exit
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, C::kTmemCols);
    }
}

template <int D, int R>
static cudaError_t launch_mla_tc(const MlaTcArgs& a, int clusters, cudaStream_t stream) {
    using C = MlaTcCfg<D, R>;
    const size_t smem = C::smem_bytes(a.plan.batch);
    auto kern = mla_decode_tc_kernel<D, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(2 * clusters), dim3(C::kThreads), smem, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t mla_tc_stage1(const MlaTcArgs& a, int D, int clusters, cudaStream_t stream) {
    if (D == 576) return launch_mla_tc<576, 512>(a, clusters, stream);
    return launch_mla_tc<320, 256>(a, clusters, stream);
}

int mla_tc_tile() { return MlaTcCfg<576, 512>::kTile; }

}  // namespace mqa
