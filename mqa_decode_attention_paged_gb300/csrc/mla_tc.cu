// MLA decode, stage 1, fifth-generation tensor-core path for 33..128 heads
// (rows past the head count are padding of the M = 128 MMA).
//
// A thread-block cluster of two CTAs owns one work unit (plan.cuh) and splits
// the 576 (or 320) latent columns so that both ranks contract over the same
// number: rank r holds the kv_c panels [r R/128, (r + 1) R/128) (64 columns
// each; they are also its V columns) and the 32-column half r of k_pe, and
// accumulates O[:, r R/2 : (r + 1) R/2].  V is the first kv_lora_rank columns
// of the same cache row ("Triton と MLA" page, vllm-arch-zh
// ja/attention/triton-mla, データフロー), so every cache byte is read from
// HBM once and TMEM holds O[128 x R/2], the logits, P and the rank's Q panels.
// The two partial logit tiles are exchanged through distributed shared memory
// and summed identically in both CTAs, which then run the same online softmax
// (tutorial page lshu.cn/news/265860, §7).
//
// The cache streams in 64-token pairs (masks are kept per 32-token tile).
// Per CTA (352 threads):
//   warp 0      TMA producer: the lanes work out a pair's boxes (page, block
//               id, validity) before its ring slot frees; then one 3D copy of
//               the pair's panels and one of its rope half when pages hold
//               whole pairs (else per-box 2D copies), 128-byte (panels) and
//               64-byte (rope) swizzle; L2 prefetches of the rows and of each
//               piece's query rows;
//   warp 1      TMEM owner and single-thread Q.K^T issuer: S[128 x 64] per
//               pair (kind::f16, M = 128 heads, N = 64 tokens, A = Q from
//               TMEM for the kv_c panels and from shared memory for the rope
//               half);
//   warps 2..9  two softmax groups of four warps (one thread per head row);
//               group g takes the pairs of parity g, so two pairs are in
//               flight: read the 64 partial logits of the row, send them to
//               the peer, add the peer's partial, mask, take the row maximum,
//               continue the running maximum handed over by the other group
//               (lazy rescaling of O only when it grows by more than 2^8),
//               write P into TMEM; the group of a piece's last pair writes the
//               output, and the next piece's Q is loaded by the group that
//               reads the piece's last logits (bf16 cache) or by the other
//               group once those logits are in TMEM (e4m3 cache); with an e4m3 cache, the group owning pair
//               q - 1 first widens pair q to f16 in place;
//   warp 10     single-thread P.V issuer: O += P V per pair in pair order
//               (A = P from TMEM, V read MN-major from the slot).
// Every wait is bounded; on expiry MQA_ERR_DEVICE_TIMEOUT is recorded and the
// roles wind down.
#include "args.cuh"
#include "common.cuh"
#include "plan.cuh"
#include "tc_ptx.cuh"

#include <type_traits>

namespace mqa {

template <int D, int R>
struct MlaTcCfg {
    static constexpr int kHeads = 128;
    static constexpr int kTile = 32;  // tokens per mask word half; a pair (pipeline stage) is two
    static constexpr int kPair = 2 * kTile;
    // Column split between the two ranks: rank r holds the 64-column kv_c
    // panels [r * kFull, (r + 1) * kFull) (its V columns) and the 32-column
    // half r of the 64-column rope part, so both ranks contract over the same
    // number of columns and hold slots of the same size.
    static constexpr int kFull = R / 128;  // full 64-column panels per rank
    static constexpr int kOCols = R / 2;   // O columns per CTA
    static constexpr int kPVPanels = kFull;
    static constexpr int kRopeCols = (D - R) / 2;  // 32
    static constexpr int kKvPanelBytes = kPair * 128;  // one full panel of a slot (128-byte rows, 128-byte swizzle)
    static constexpr int kRopeBytes = kPair * 64;      // the slot's rope half (64-byte rows, 64-byte swizzle)
    static constexpr int kSlotBytes = kFull * kKvPanelBytes + kRopeBytes;
    static constexpr int kQRopeBytes = kHeads * 64;    // Q's rope half in shared memory (64-byte swizzle)
    // TMEM columns: O [0, 256), S [256, 320), P two buffers [320, 384), Q
    // [384, 384 + 32 * kFull) (the rank's kv_c panels as packed 16-bit pairs)
    static constexpr int kTmemCols = 512;
    static constexpr int kTmemS = 256;
    static constexpr int kTmemP = 320;
    static constexpr int kTmemQ = 384;
    static constexpr int kXBytes = kHeads * kPair * 4;  // one fp32 logit pair
    static constexpr int kGroupWarps = 4;
    static constexpr int kGroupThreads = 32 * kGroupWarps;
    static constexpr int kSoftmaxWarps = 2 * kGroupWarps;
    static constexpr int kThreads = 32 * (3 + kSoftmaxWarps);

    static constexpr int kNumBars = 40;
    static constexpr int kRedBytes = 4 * kHeads * 4;  // running maxima [2][128], handed-over sums / maxima
    // everything but the ring: alignment slack, Q rope half, X, barriers,
    // reductions, up to 8 stage masks, the TMEM address, lengths
    static constexpr int kFixedBytes =
        1024 + kQRopeBytes + 2 * kXBytes + kNumBars * 8 + kRedBytes + 8 * 8 + 16 + 4 * (2 * kMaxBatchTc + 1);
    static constexpr int kSlotsFit = (227 * 1024 - kFixedBytes) / kSlotBytes;
    static constexpr int kSlots = kSlotsFit > 6 ? 6 : kSlotsFit;
    static constexpr int kStages = kSlots;  // one pipeline stage per 64-token pair
    static constexpr int kOffQ = 0;
    static constexpr int kOffStages = kOffQ + kQRopeBytes;
    static constexpr int kOffX = kOffStages + kSlots * kSlotBytes;
    static constexpr int kOffBars = kOffX + 2 * kXBytes;
    static constexpr int kOffRed = kOffBars + kNumBars * 8;
    static constexpr int kOffMask = kOffRed + kRedBytes;
    static constexpr int kOffTmem = kOffMask + kStages * 8;
    static constexpr int kOffCum = kOffTmem + 16;
    static size_t smem_bytes(int batch) { return 1024 + kOffCum + 4 * (2 * batch + 1); }

    static_assert(kOCols <= 256 && kOCols % 64 == 0 && kRopeCols == 32, "column split");
    static_assert(kOCols <= kTmemS && kTmemS + kPair <= kTmemP && kTmemP + kPair <= kTmemQ &&
                      kTmemQ + 32 * kFull <= kTmemCols,
                  "TMEM layout");
    static_assert(kSlots >= 2 && kStages <= 8, "pipeline depth");
    static_assert(1024 + kOffCum + 4 * (2 * kMaxBatchTc + 1) <= 227 * 1024, "shared memory budget");
    static_assert(kOffStages % 1024 == 0 && kSlotBytes % 1024 == 0 && (kFull * kKvPanelBytes) % 512 == 0,
                  "swizzled operands need 1024-byte (128-byte swizzle) / 512-byte (64-byte swizzle) alignment");
};

// barrier slots, each range starting where the previous one ends
enum TcBar {
    kKvFull = 0,             // [8] pair landed (producer expect_tx + TMA bytes)
    kKvEmpty = kKvFull + 8,  // [8] P.V of the pair done (tensor-core commit)
    kQTmem = kKvEmpty + 8,   // a softmax group has written the piece's Q (TMEM panels, smem rope half)
    kSFull = kQTmem + 1,     // [2] logit pair of parity i in TMEM
    kSEmpty = kSFull + 2,    // the logit pair read out by its softmax group
    kPFull = kSEmpty + 1,    // [2] P of a pair in TMEM buffer (pair & 1), O rescaled if needed
    kPEmpty = kPFull + 2,    // [2] P.V of that pair done
    kXFull = kPEmpty + 2,    // [2] the peer's logit pair for group g has arrived
    kXFree = kXFull + 2,     // [2] the peer's group g has consumed the pair we sent it
    kMReady = kXFree + 2,    // [2] running maximum after a pair of parity i published
    kLReady = kMReady + 2,   // the group without the piece's last pair handed over its sum
    kOFree = kLReady + 1,    // the piece's output has been read out of TMEM
    kConv = kOFree + 1,      // [4] fp8 cache: pair q (q % 4 = i) was widened to f16 in its slot
    kDrain = kConv + 4,      // every tensor-core operation of the CTA has completed
    kBarCount = kDrain + 1,
};
static_assert(kBarCount <= MlaTcCfg<576, 512>::kNumBars && kBarCount <= MlaTcCfg<320, 256>::kNumBars,
              "barrier slots");

// Q.K^T of one pair into TMEM columns d: NF full panels with Q from TMEM
// (q_tmem) and K from the slot's 128-byte-swizzled panels (kdesc = panel 0),
// then the 32-column rope half with Q from shared memory (qrope) and K from
// the slot (krope), both 64-byte swizzled.  Descriptors advance by constant
// byte offsets >> 4 (the start-address field cannot carry: shared addresses
// stay below 256 KB).
template <int NF, int KvPanelBytes>
__device__ __forceinline__ void issue_qk(uint32_t d, uint32_t q_tmem, uint64_t kdesc, uint64_t qrope, uint64_t krope,
                                         uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < NF * 4; ++ks)
        umma_bf16_ta(d, q_tmem + ks * 8,
                     kdesc + static_cast<uint64_t>(((ks >> 2) * KvPanelBytes + (ks & 3) * 32) >> 4), idesc,
                     ks > 0 ? 1u : 0u);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
        umma_bf16(d, qrope + static_cast<uint64_t>((ks * 32) >> 4), krope + static_cast<uint64_t>((ks * 32) >> 4),
                  idesc, 1u);
}

// MULTI: multi-token decode (per-row key limits); the plain-decode kernels
// are compiled without that code.  MODE: the work plan's iterator, 0 for
// page-balanced units (PieceIter, which per-request mode also takes), 1 for
// the fixed-split mode (one unit per request and range), 2 for units
// balanced on pages plus a cost per request start (CostPieceIter); separate
// instantiations, so that each keeps its own code.
enum TcPlanMode { kModeBalanced = 0, kModeFixed = 1, kModeCost = 2 };
template <int D, int R, bool FP8, bool MULTI, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MlaTcCfg<D, R>::kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ MlaTcArgs a) {
    using C = MlaTcCfg<D, R>;
    using PIter = std::conditional_t<MODE == kModeFixed, FixedPieceIter,
                                     std::conditional_t<MODE == kModeCost, CostPieceIter, PieceIter>>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* q_s = smem + C::kOffQ;
    uint8_t* stages = smem + C::kOffStages;
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
    const int pbase = rank * C::kFull;             // first global 64-column panel of the rank
    const int rope0 = R + rank * C::kRopeCols;     // first column of the rank's rope half
    const int P = a.plan.page;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars[kKvFull + s], 1);
            mbar_init(&bars[kKvEmpty + s], 1);
        }
        mbar_init(&bars[kQTmem], C::kGroupThreads);
        mbar_init(&bars[kSEmpty], C::kGroupThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kSFull + i], 1);
            mbar_init(&bars[kPFull + i], C::kGroupThreads);
            mbar_init(&bars[kPEmpty + i], 1);
            mbar_init(&bars[kXFull + i], 1);                 // own expect_tx; the bytes come from the peer
            mbar_init(&bars[kXFree + i], C::kGroupWarps);    // one arrive per warp of the peer's group
            mbar_init(&bars[kMReady + i], C::kGroupThreads);
        }
        mbar_init(&bars[kLReady], C::kGroupThreads);
        for (int i = 0; i < 4; ++i) mbar_init(&bars[kConv + i], C::kGroupThreads);
        mbar_init(&bars[kOFree], C::kGroupThreads);
        mbar_init(&bars[kDrain], 2);  // one commit from each issuing thread
        fence_mbar_init();
        prefetch_tmap(&a.kv_map);
        prefetch_tmap(&a.kv_pair_map[0]);
        prefetch_tmap(&a.kv_rope_map);
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
    // byte offset of pair p's slot in the ring
    auto slot_base = [&](int p) { return (p % C::kStages) * C::kSlotBytes; };
    // fp8 cache: the pair's e4m3 full panels (64 rows x 64 bytes each) and
    // rope half (64 rows x 32 bytes), unswizzled, land at the end of the slot
    // and are widened in place to f16 in the operand layouts
    constexpr int kF8PanelBytes = C::kPair * 64;
    constexpr int kF8RopeBytes = C::kPair * 32;
    constexpr int kF8Bytes = C::kFull * kF8PanelBytes + kF8RopeBytes;
    constexpr int f8_off = FP8 ? C::kSlotBytes - kF8Bytes : 0;
    constexpr int kRowBytes = FP8 ? 64 : 128;      // bytes per cache row and full panel as copied
    constexpr int kRopeRowBytes = FP8 ? 32 : 64;   // bytes per cache row of the rope half as copied
    // as-copied offsets within the slot of the full panels and of the rope half
    constexpr int kCopyPanelBytes = C::kPair * kRowBytes;
    constexpr int kCopyRopeOff = f8_off + C::kFull * kCopyPanelBytes;

    if (warp == 0) {
        // ------------------------------------------------------ KV producer
        // The whole warp walks the pairs.  Lane l holds the block id of page l
        // of the piece's current 32-page chunk (the next chunk is loaded one
        // chunk ahead, so table reads stay off the issue path); lane k < nbox
        // takes box k of the pair (BR tokens of one page).  Everything for a
        // pair is worked out before its ring slot frees; then lane 0 stores
        // the token mask and arms kv_full, and the lanes issue the copies:
        // one 3D copy of the pair's panels (lane 0) and one of its rope half
        // (lane 1) when pages hold whole pairs, else one 2D copy per panel
        // and one for the rope half per box (lane k).
        const uint64_t pol = l2_policy_evict_first();
        const int BR = a.box_rows, nbox = C::kPair / BR;  // boxes per pair (1, 2 or 4)
        const uint32_t box_bytes = BR * (C::kFull * kRowBytes + kRopeRowBytes);
        const uint64_t box_ones = BR == 64 ? ~0ull : ((1ull << BR) - 1);
        // boxes are whole pages (16- or 32-token pages) or pairs are whole
        // page parts (pages of a multiple of 64 tokens): pages are tracked
        // without division; other page sizes divide
        const bool pages_fit = BR == P || BR == C::kPair;
        const CUtensorMap* pair_map = &a.kv_pair_map[0];
        PIter it;
        it.init(a.plan, cum, T, unit);
        Piece pc;
        int p = 0;
        // test hook: the producer of the withheld unit fills and announces
        // nothing, so its consumers' first waits run out
        bool ok = unit != a.withhold;
        while (ok && it.next(cum, pc)) {
            int tok0, tok_end;
            const int npairs = piece_tiles(pc, tok0, tok_end) >> 1;
            if (npairs == 0) continue;
            // the piece's query rows (this rank's half of the heads) towards
            // L2: a softmax group loads them into TMEM once the pairs before
            // the piece have been read out, several pairs from now
            if (lane == 0) {
                const int hh = (a.H + 1) >> 1, h0 = rank * hh, nh = min(a.H, h0 + hh) - h0;
                if (nh > 0)
                    bulk_prefetch_l2(a.q + (static_cast<long long>(pc.b) * a.H + h0) * D,
                                     static_cast<uint32_t>(nh * D * 2));
            }
            const int32_t* bt = a.block_table + static_cast<long long>(pc.b) * a.plan.max_blocks + pc.j0;
            const int npg = pc.j1 - pc.j0;
            auto load_chunk = [&](int c) {
                const int pg = c * 32 + lane;
                return pg < npg ? __ldg(bt + pg) : -1;
            };
            int chunk = 0;
            int blk_cur = load_chunk(0);
            int blk_nxt = load_chunk(1);
            // page (within the piece) and row offset in it of the pair's first
            // token, advanced without division: pages of less than 64 tokens
            // hold whole boxes (BR = P), larger pages hold whole pairs
            int pg0 = 0, off0 = 0;
            for (int jp = 0; jp < npairs; ++jp, ++p) {
                const int t0 = tok0 + jp * C::kPair;
                // box `lane` of the pair (pages of one pair span at most one
                // chunk boundary: boxes before it read blk_cur, after it blk_nxt)
                const int tok = t0 + lane * BR;
                const bool inbox = lane < nbox && tok < tok_end;
                const int rel = !inbox ? 0 : pages_fit ? pg0 + (BR == P ? lane : 0) : tok / P - pc.j0;
                const int bc = __shfl_sync(0xffffffffu, blk_cur, rel & 31);
                const int bn = __shfl_sync(0xffffffffu, blk_nxt, rel & 31);
                const int blk = (rel >> 5) == chunk ? bc : bn;
                bool v = inbox;
                if (v && (blk < 0 || blk >= a.num_blocks)) {
                    report(a.status, MQA_ERR_DEVICE_CHECK);
                    v = false;
                }
                const int last_rel = __reduce_max_sync(0xffffffffu, rel);
                if ((last_rel >> 5) != chunk) {  // the pair reached the next chunk
                    blk_cur = blk_nxt;
                    ++chunk;
                    blk_nxt = load_chunk(chunk + 1);
                }
                const unsigned vball = __ballot_sync(0xffffffffu, v);
                const int n_tok = max(tok_end - t0, 0);
                uint64_t vmask = n_tok >= C::kPair ? ~0ull : ((1ull << n_tok) - 1);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k < nbox && !((vball >> k) & 1u)) vmask &= ~(box_ones << (k * BR));
                const int row = !v ? 0 : blk * P + (pages_fit ? off0 : tok % P);
                if (BR == P) {
                    pg0 += nbox;
                } else if ((off0 += C::kPair) == P) {
                    off0 = 0;
                    ++pg0;
                }
                const int st = p % C::kStages;
                uint8_t* dst = stages + slot_base(p) + f8_off;
                uint8_t* rope_dst = stages + slot_base(p) + kCopyRopeOff;
                // while the slot is still busy, pull the box's whole cache rows
                // (both ranks' columns) towards L2 so the copies below hit it
                if (rank == 0 && v)
                    bulk_prefetch_l2(a.kv + static_cast<long long>(row) * (D * (FP8 ? 1 : 2)),
                                     static_cast<uint32_t>(BR * D * (FP8 ? 1 : 2)));
                // every issuing lane observes the slot free (P.V of its last pair done)
                if (!__all_sync(0xffffffffu, mbar_wait(&bars[kKvEmpty + st], ((p / C::kStages) & 1) ^ 1))) {
                    if (lane == 0) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mask_s[st] = vmask;
                    mbar_arrive_expect_tx(&bars[kKvFull + st], __popc(vball) * box_bytes);
                }
                if (BR == C::kPair) {
                    const int row0 = __shfl_sync(0xffffffffu, row, 0);
                    if (vball & 1u) {
                        if (lane == 0) tma_load_3d(dst, pair_map, 0, row0, pbase, &bars[kKvFull + st], pol);
                        if (lane == 1) tma_load_2d(rope_dst, &a.kv_rope_map, rope0, row0, &bars[kKvFull + st], pol);
                    }
                } else if (v) {
                    for (int pn = 0; pn < C::kFull; ++pn)
                        tma_load_2d(dst + pn * kCopyPanelBytes + lane * BR * kRowBytes, &a.kv_map, (pbase + pn) * 64,
                                    row, &bars[kKvFull + st], pol);
                    tma_load_2d(rope_dst + lane * BR * kRopeRowBytes, &a.kv_rope_map, rope0, row, &bars[kKvFull + st],
                                pol);
                }
                __syncwarp();
            }
        }
        // every copy issued has landed before the CTA may tear down
        if (lane == 0)
            for (int q = max(p - C::kStages, 0); q < p; ++q)
                if (!mbar_wait(&bars[kKvFull + q % C::kStages], (q / C::kStages) & 1))
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
    } else if (warp == 2 + C::kSoftmaxWarps) {
        // ------------------------------------------------------ P.V issuer
        // One thread issues O += P V per pair, in pair order, as soon as its P
        // is in TMEM (and, for a piece's first pair, the previous piece's
        // output has been read out of O).
        if (lane == 0) {
            constexpr uint32_t kIdPV = FP8 ? umma_idesc_f16(128, C::kOCols, 1) : umma_idesc_bf16(128, C::kOCols, 1);
            const uint64_t vdesc0 = umma_desc(smem_u32(stages), C::kKvPanelBytes, 1024);
            PIter vi;
            vi.init(a.plan, cum, T, unit);
            Piece vpc;
            int vp = 0, vc = 0;  // next pair, pieces with tokens begun
            bool ok = true;
            while (ok && vi.next(cum, vpc)) {
                int tok0, tok_end;
                const int npairs = piece_tiles(vpc, tok0, tok_end) >> 1;
                if (npairs == 0) continue;
                for (int j = 0; j < npairs; ++j, ++vp) {
                    const int pb = vp & 1;
                    if (!mbar_wait(&bars[kPFull + pb], (vp >> 1) & 1) ||
                        (j == 0 && vc > 0 && !mbar_wait(&bars[kOFree], (vc - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t vd = vdesc0 + static_cast<uint64_t>(slot_base(vp) >> 4);
#pragma unroll
                    for (int ks = 0; ks < C::kPair / 16; ++ks)
                        umma_bf16_ta(tbase, tbase + C::kTmemP + pb * (C::kPair / 2) + ks * 8,
                                     vd + static_cast<uint64_t>((ks * 16 * 128) >> 4), kIdPV,
                                     (j == 0 && ks == 0) ? 0u : 1u);
                    umma_commit(&bars[kPEmpty + pb]);
                    umma_commit(&bars[kKvEmpty + vp % C::kStages]);
                }
                ++vc;
            }
            if (!ok) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            // no tensor-core work of this thread may be in flight at teardown
            umma_commit(&bars[kDrain]);
            if (!mbar_wait(&bars[kDrain], 0)) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ Q.K^T issuer
        // One thread issues S = Q K^T per pair, in pair order, once the
        // piece's Q is in TMEM and shared memory, the previous pair's logits
        // were read out and the pair's rows landed (fp8: and were widened).
        if (lane == 0) {
            constexpr uint32_t kIdQK = FP8 ? umma_idesc_f16(128, C::kPair, 0) : umma_idesc_bf16(128, C::kPair, 0);
            const uint64_t kdesc0 = umma_desc(smem_u32(stages), 16, 1024);
            const uint64_t krope0 = umma_desc_sw64(smem_u32(stages) + C::kFull * C::kKvPanelBytes);
            const uint64_t qrope = umma_desc_sw64(smem_u32(q_s));
            PIter qi;
            qi.init(a.plan, cum, T, unit);
            Piece qpc;
            int qp = 0, qc = 0;
            bool ok = true;
            while (ok && qi.next(cum, qpc)) {
                int tok0, tok_end;
                const int npairs = piece_tiles(qpc, tok0, tok_end) >> 1;
                if (npairs == 0) continue;
                if (!mbar_wait(&bars[kQTmem], qc & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < npairs; ++j, ++qp) {
                    // bf16: the pair's rows landed; fp8: they were also widened to f16
                    const bool ready = FP8 ? mbar_wait(&bars[kConv + (qp & 3)], (qp >> 2) & 1)
                                           : mbar_wait(&bars[kKvFull + qp % C::kStages], (qp / C::kStages) & 1);
                    if (!mbar_wait(&bars[kSEmpty], (qp & 1) ^ 1) || !ready) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tbase + C::kTmemS;
                    const uint64_t sb = static_cast<uint64_t>(slot_base(qp) >> 4);
                    issue_qk<C::kFull, C::kKvPanelBytes>(d, tbase + C::kTmemQ, kdesc0 + sb, qrope, krope0 + sb, kIdQK);
                    umma_commit(&bars[kSFull + (qp & 1)]);
                }
                ++qc;
            }
            if (!ok) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            umma_commit(&bars[kDrain]);
            if (!mbar_wait(&bars[kDrain], 0)) report(a.status, MQA_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp >= 2 && warp < 2 + C::kSoftmaxWarps) {
        // ------------------------------------------------------ softmax groups
        // Group g (warps 2 + 4 g .. 5 + 4 g, one of each TMEM lane quadrant)
        // takes the pairs of parity g; thread (quad, lane) owns head row h.
        const int quad = warp & 3;
        const int g = (warp - 2) / C::kGroupWarps;
        const int h = quad * 32 + lane;
        const bool live_row = h < a.H;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quad * 32) << 16);
        float* m_s = red_s;                        // [2][128] running maximum after a pair of parity i
        float* lh_s = red_s + 2 * C::kHeads;      // [128] sum handed to the epilogue group
        float* mh_s = red_s + 3 * C::kHeads;      // [128] maximum that sum is relative to
        // logit pairs travel lane-contiguously: chunk c (4 floats, c < 16) of
        // row (quad, lane) sits at ((quad * 16 + c) * 32 + lane) * 16 bytes, so
        // every warp store writes 512 contiguous bytes of the peer's buffer
        const uint32_t x_off = (quad * 16 * 32 + lane) * 16;
        const uint32_t x_remote = map_to_rank(x_s + g * C::kXBytes, peer) + x_off;
        const uint8_t* x_local = x_s + g * C::kXBytes + x_off;
        const uint32_t xfull_remote = map_to_rank(&bars[kXFull + g], peer);
        const uint32_t xfree_remote = map_to_rank(&bars[kXFree + g], peer);
        // warp-uniform bounded waits: TMEM accesses are warp-collective, so a
        // lane never leaves the loop on its own.  A warp whose wait expires
        // does leave it; in the e4m3 kernel it first makes the rest of its
        // group's widening barrier arrivals (see `widen`), so that no other
        // warp of the group blocks there, and every other wait is bounded.
        // Waits expire only on a broken hand-off or a GPU stalled for
        // seconds, never on caller input: bad block ids and lengths are
        // masked before any wait.
        auto wait_all = [&](uint64_t* bar, uint32_t parity, bool cluster_scope) {
            const bool done = cluster_scope ? mbar_wait_cluster(bar, parity) : mbar_wait(bar, parity);
            return __all_sync(0xffffffffu, done);
        };
        // Q row h of the next piece that holds tokens (after `from`) into
        // TMEM, one 32-bit column per pair of consecutive dims (low half = even)
        auto stage_q = [&](PIter from) {
            Piece nx;
            int tok0, tok_end;
            while (from.next(cum, nx)) {
                if (piece_tiles(nx, tok0, tok_end) == 0) continue;
                const __nv_bfloat16* qrow = a.q + (static_cast<long long>(nx.b) * a.H + (live_row ? h : 0)) * D;
                const uint4* src = reinterpret_cast<const uint4*>(qrow + pbase * 64);
                if constexpr (FP8) {
                    // staged by the group that does not own the piece's last
                    // pair, with no logits live: the rope half's loads go
                    // first, then the loads of four TMEM stores (8 columns, 16
                    // dims, each) are issued before any of them
                    const uint4* rsrc = reinterpret_cast<const uint4*>(qrow + rope0);
                    uint4 rv[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) rv[c] = live_row ? __ldg(rsrc + c) : make_uint4(0, 0, 0, 0);
                    constexpr int kBatch = 4;
                    for (int c0 = 0; c0 < 4 * C::kFull; c0 += kBatch) {
                        uint4 v[2 * kBatch];
#pragma unroll
                        for (int i = 0; i < 2 * kBatch; ++i)
                            v[i] = live_row ? __ldg(src + 2 * c0 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int c = 0; c < kBatch; ++c) {
                            uint32_t r[8] = {v[2 * c].x, v[2 * c].y, v[2 * c].z, v[2 * c].w,
                                             v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
#pragma unroll
                            for (int i = 0; i < 8; ++i) r[i] = bf16x2_to_f16x2(r[i]);
                            tmem_st8(lane_addr + C::kTmemQ + (c0 + c) * 8, r);
                        }
                    }
                    // the rope half: the K-major operand in shared memory with
                    // the 64-byte swizzle
                    uint8_t* row = q_s + h * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(row + ((c ^ ((h >> 1) & 3)) << 4)) =
                            make_uint4(bf16x2_to_f16x2(rv[c].x), bf16x2_to_f16x2(rv[c].y), bf16x2_to_f16x2(rv[c].z),
                                       bf16x2_to_f16x2(rv[c].w));
                    fence_proxy_async_smem();
                } else {
                    // 8 columns (16 dims) per TMEM store; the loads of four
                    // stores are issued before any of them (a TMEM store
                    // orders memory)
                    constexpr int kBatch = 4;
                    for (int c0 = 0; c0 < 4 * C::kFull; c0 += kBatch) {
                        uint4 v[2 * kBatch];
#pragma unroll
                        for (int i = 0; i < 2 * kBatch; ++i)
                            v[i] = live_row ? __ldg(src + 2 * c0 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int c = 0; c < kBatch; ++c) {
                            uint32_t r[8] = {v[2 * c].x, v[2 * c].y, v[2 * c].z, v[2 * c].w,
                                             v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
                            tmem_st8(lane_addr + C::kTmemQ + (c0 + c) * 8, r);
                        }
                    }
                    // the rank's rope half (32 dims = 64 bytes), the K-major
                    // operand in shared memory with the 64-byte swizzle
                    const uint4* rsrc = reinterpret_cast<const uint4*>(qrow + rope0);
                    uint8_t* row = q_s + h * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = live_row ? __ldg(rsrc + c) : make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(row + ((c ^ ((h >> 1) & 3)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kQTmem]);
                return;
            }
        };

        // P.V of this group's own pair p2 (parity g) done.  The group waits on
        // its own barrier once per own pair, in pair order, so every parity
        // wait targets the phase after the last one it saw complete.
        auto wait_own_pv = [&](int p2) { return wait_all(&bars[kPEmpty + g], (p2 >> 1) & 1, false); };

        // fp8 cache: widen pair q's e4m3 panels to f16 in place, then let
        // Q.K^T(q) go.  The group that owns pair q - 1 widens q (group 0 also
        // widens pair 0), one step ahead of its Q.K^T.  Pair q arrives on
        // barrier q % 4: a group starts the step that widens q + 4 only after
        // Q.K^T(q + 1) could run, i.e. after every thread that widened q did,
        // so one barrier's phases never overlap.
        //
        // The reads and writes of the group's threads are separated by named
        // barrier 1 + g, kFull + 1 times per widened pair.  A named barrier
        // has no time limit, so a warp that gives up (an expired wait) first
        // makes the group's remaining arrivals there (`drain_widen`): which
        // pairs a group widens is fixed by the unit's pair count, so every
        // warp of the group then arrives equally often, and the others go on
        // to their own bounded waits instead of blocking.
        auto widen = [&](int q) -> bool {
            // ---- widen the pair's e4m3 panels to f16 in place: thread t
            // takes row t / 2, bytes 32 (t % 2) .. + 31 of each full
            // panel, then bytes 16 (t % 2) .. + 15 of the rope half; all
            // reads of a panel precede its writes (the f16 panel overlaps
            // its own e4m3 source and earlier ones, never a later one)
            if (!wait_all(&bars[kKvFull + q % C::kStages], (q / C::kStages) & 1, false)) return false;
            const int t = quad * 32 + lane, r = t >> 1, hb = t & 1;
            uint8_t* slot = stages + slot_base(q);
            for (int pn = 0; pn < C::kFull; ++pn) {
                const uint8_t* srcp = slot + f8_off + pn * kF8PanelBytes + r * 64 + hb * 32;
                const uint4 w0 = *reinterpret_cast<const uint4*>(srcp);
                const uint4 w1 = *reinterpret_cast<const uint4*>(srcp + 16);
                named_bar_sync(1 + g, C::kGroupThreads);
                const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint8_t* dstp = slot + pn * C::kKvPanelBytes + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        o[2 * i] = e4m3x2_to_f16x2(w[2 * c + i] & 0xffffu);
                        o[2 * i + 1] = e4m3x2_to_f16x2(w[2 * c + i] >> 16);
                    }
                    *reinterpret_cast<uint4*>(dstp + (((hb * 4 + c) ^ (r & 7)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            {
                const uint4 w0 = *reinterpret_cast<const uint4*>(slot + f8_off + C::kFull * kF8PanelBytes +
                                                                  r * 32 + hb * 16);
                named_bar_sync(1 + g, C::kGroupThreads);
                const uint32_t w[4] = {w0.x, w0.y, w0.z, w0.w};
                uint8_t* dstp = slot + C::kFull * C::kKvPanelBytes + r * 64;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        o[2 * i] = e4m3x2_to_f16x2(w[2 * c + i] & 0xffffu);
                        o[2 * i + 1] = e4m3x2_to_f16x2(w[2 * c + i] >> 16);
                    }
                    *reinterpret_cast<uint4*>(dstp + (((hb * 2 + c) ^ ((r >> 1) & 3)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[kConv + (q & 3)]);
            return true;
        };
        // pairs of the whole unit (for the look-ahead widening)
        int total_pairs = 0;
        {
            PIter ti;
            ti.init(a.plan, cum, T, unit);
            Piece tp;
            int t0_, te_;
            while (ti.next(cum, tp)) total_pairs += piece_tiles(tp, t0_, te_) >> 1;
        }

        // Group 0 widens pair 0 and the odd pairs, group 1 the even pairs
        // from 2: the pairs up to pair q (q < total_pairs) that group g widens.
        auto widened_upto = [&](int q) {
            return q < 0 ? 0 : g == 0 ? 1 + (q + 1) / 2 : q / 2;
        };
        // After an expired wait: the widening barrier arrivals this warp still
        // owes its group, when it has widened every pair of its up to pair
        // `done` (computed on the way out, so the fast path keeps no count).
        auto drain_widen = [&](int done) {
            const int last = total_pairs - 1;
            const int owed = (C::kFull + 1) * (widened_upto(last) - widened_upto(done < last ? done : last));
            for (int i = 0; i < owed; ++i) named_bar_sync(1 + g, C::kGroupThreads);
        };
        // set only on the way out after an expired wait (see drain_widen), so
        // that it occupies no register while the pairs go through
        int widened;

        PIter it;
        it.init(a.plan, cum, T, unit);
        Piece pc;
        int gp = 0;      // global index of the current piece's first pair
        int kpiece = 0;  // pieces with tokens so far
        bool ok = true;
        if (g == 0) stage_q(it);
        if (FP8 && g == 0 && total_pairs > 0 && !widen(0)) {
            ok = false;
            widened = -1;
        }
        // test hook: softmax warp give_up % 16 of unit give_up / 16 stops here
        // as if a wait had expired; the rest of its group goes on
        if (ok && a.give_up >= 0 && unit == (a.give_up >> 4) && warp == (a.give_up & 15)) {
            ok = false;
            widened = 0;  // pair 0, if any, was widened (group 0) or is not the group's (group 1)
        }
        while (ok && it.next(cum, pc)) {
            int tok0, tok_end;
            const int nt = piece_tiles(pc, tok0, tok_end);
            const int npairs = nt >> 1;
            if (nt == 0) {  // empty request (per-request mode): out = 0, lse = -inf
                if (g == 0 && live_row && pc.whole) {
                    __nv_bfloat16* o = a.out + (static_cast<long long>(pc.b) * a.H + h) * R + rank * C::kOCols;
                    for (int c = 0; c < C::kOCols; c += 8) *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
                    if (rank == 0 && a.lse) a.lse[static_cast<long long>(pc.b) * a.H + h] = -INFINITY;
                }
                continue;
            }
            // this group's sum of p over its pairs of the piece, relative to m_l
            float l_part = 0.f, m_l = -INFINITY;
            for (int j = ((gp & 1) == g) ? 0 : 1; j < npairs; j += 2) {
                const int p = gp + j, pb = p & 1;
                if (FP8 && p + 1 < total_pairs && !widen(p + 1)) {
                    ok = false;
                    widened = p;  // pair p + 1 was not widened
                    break;
                }
                // ---- logits of the pair: own partial from TMEM
                float s[C::kPair];
                if (!wait_all(&bars[kSFull + pb], (p >> 1) & 1, false)) {
                    ok = false;
                    widened = p + 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + C::kTmemS + half * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[half * 32 + i] = __uint_as_float(r[i]);
                }
                tc_fence_before();
                mbar_arrive(&bars[kSEmpty]);
                // bf16 cache: the piece's last logit pair is in, so every
                // Q.K^T that read the TMEM Q panels has completed: stage the
                // next piece's Q right away (the e4m3 kernel hands this to the
                // other group, see the piece epilogue)
                if (!FP8 && j == npairs - 1) stage_q(it);
                // ---- send the partial to the peer, receive and add the peer's
                if (h == 0) mbar_arrive_expect_tx(&bars[kXFull + g], C::kXBytes);
                if (p >= 2 && !wait_all(&bars[kXFree + g], ((p >> 1) & 1) ^ 1, true)) {
                    ok = false;
                    widened = p + 1;
                    break;
                }
#pragma unroll
                for (int c = 0; c < C::kPair / 4; ++c)
                    st_async_v4(x_remote + c * 512, s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3], xfull_remote);
                // valid tokens of the pair (set by the producer before kv_full)
                if (!wait_all(&bars[kKvFull + p % C::kStages], (p / C::kStages) & 1, false)) {
                    ok = false;
                    widened = p + 1;
                    break;
                }
                const uint64_t vm = mask_s[p % C::kStages];
                // tokens of the pair this row sees: multi-token decode limits
                // row h (token i = h / heads) to tokens below len - q_len + i + 1
                // (tutorial page §10); the V rows past the sequence end are
                // still cleared by vm
                uint64_t vmr = vm;
                if constexpr (MULTI) {
                    const int lim = lens[pc.b] - (a.q_len - 1 - h / a.heads) - (tok0 + j * C::kPair);
                    vmr &= lim >= C::kPair ? ~0ull : lim <= 0 ? 0ull : ((1ull << lim) - 1);
                }
                if (!wait_all(&bars[kXFull + g], (p >> 1) & 1, true)) {
                    ok = false;
                    widened = p + 1;
                    break;
                }
#pragma unroll
                for (int c = 0; c < C::kPair / 4; ++c) {
                    const float4 v = *reinterpret_cast<const float4*>(x_local + c * 512);
                    s[4 * c] += v.x;
                    s[4 * c + 1] += v.y;
                    s[4 * c + 2] += v.z;
                    s[4 * c + 3] += v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(xfree_remote);
                // ---- mask, row maximum in base 2.  With a bf16 cache a pair
                // of valid tokens keeps the raw sums: the base-2 scale k2 =
                // sl2 (> 0) goes into the maximum and into the exponent (P =
                // 2^(s k2 - m), one FMA per logit); otherwise (and always for
                // the e4m3 kernel, whose registers are at their limit) the
                // sums are masked and scaled here and k2 = 1.
                float k2 = FP8 ? 1.f : a.sl2;
                if (FP8 || vmr != ~0ull || !(a.sl2 > 0.f)) {
#pragma unroll
                    for (int i = 0; i < C::kPair; ++i) s[i] = ((vmr >> i) & 1ull) ? s[i] * a.sl2 : -INFINITY;
                    k2 = 1.f;
                }
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    mx[i] = fmaxf(fmaxf(fmaxf(s[i], s[i + 8]), fmaxf(s[i + 16], s[i + 24])),
                                  fmaxf(fmaxf(s[i + 32], s[i + 40]), fmaxf(s[i + 48], s[i + 56])));
                const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * k2;
                // ---- running maximum: continue the one the other group
                // published after pair p - 1 (always waited for, so that its
                // slot is not overwritten before it was read)
                float m_prev = -INFINITY;
                if (p >= 1) {
                    if (!wait_all(&bars[kMReady + ((p - 1) & 1)], ((p - 1) >> 1) & 1, false)) {
                        ok = false;
                        widened = p + 1;
                        break;
                    }
                    m_prev = m_s[((p - 1) & 1) * C::kHeads + h];
                }
                float m_run;
                if (j == 0) {
                    m_run = mt;
                } else if (__any_sync(0xffffffffu, mt > m_prev + 8.f)) {
                    // the running max grew by more than 2^8 (decided per warp;
                    // rows whose max did not grow rescale by 1): wait for
                    // P.V(p - 1), then rescale the row of O
                    m_run = fmaxf(mt, m_prev);
                    const float alpha = ex2(m_prev - m_run);
                    // P.V runs in pair order: with the own P.V(p - 2) seen
                    // complete, the other parity's barrier is at most one
                    // phase short of P.V(p - 1)
                    if ((p >= 2 && !wait_own_pv(p - 2)) ||
                        !wait_all(&bars[kPEmpty + (g ^ 1)], ((p - 1) >> 1) & 1, false)) {
                        ok = false;
                        widened = p + 1;
                        break;
                    }
                    tc_fence_after();
                    for (int c0 = 0; c0 < C::kOCols; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16(lane_addr + c0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st16(lane_addr + c0, r);
                    }
                } else {
                    m_run = m_prev;
                }
                m_s[pb * C::kHeads + h] = m_run;
                mbar_arrive(&bars[kMReady + pb]);
                // ---- P of the pair into TMEM buffer pb (last read by P.V(p - 2))
                if (p >= 2 && !wait_own_pv(p - 2)) {
                    ok = false;
                    widened = p + 1;
                    break;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                float psum = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = ex2(fmaf(s[half * 32 + 2 * i], k2, -m_use));
                        const float p1 = ex2(fmaf(s[half * 32 + 2 * i + 1], k2, -m_use));
                        psum += p0 + p1;
                        pk[i] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                    }
                    tmem_st16(lane_addr + C::kTmemP + pb * (C::kPair / 2) + half * 16, pk);
                }
                if (m_l != m_run) {  // re-express this group's sum relative to the new maximum
                    l_part = m_l == -INFINITY ? 0.f : l_part * ex2(m_l - m_run);
                    m_l = m_run;
                }
                l_part += psum;
                // rows past the sequence end: zero their V columns in the slot
                // (thread h clears row h % 64 of V panels h / 64 + 2 k)
                bool zeroed = false;
                if (vm != ~0ull) {
                    const int r = h & (C::kPair - 1);
                    if (!((vm >> r) & 1ull)) {
                        for (int pn = h / C::kPair; pn < C::kPVPanels; pn += C::kHeads / C::kPair) {
                            uint8_t* base = stages + slot_base(p) + r * 128 + pn * C::kKvPanelBytes;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(base + c * 16) = make_uint4(0, 0, 0, 0);
                        }
                        zeroed = true;
                    }
                }
                if (__any_sync(0xffffffffu, zeroed)) fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[kPFull + pb]);
            }
            if (!ok) break;

            // ---- piece epilogue: the group of the last pair writes the output
            const int plast = gp + npairs - 1;
            if ((plast & 1) != g) {
                // hand this group's sum over (after the previous epilogue read the slot)
                if (kpiece >= 1 && !wait_all(&bars[kOFree], (kpiece - 1) & 1, false)) {
                    ok = false;
                    widened = gp + npairs;
                    break;
                }
                lh_s[h] = l_part;
                mh_s[h] = m_l;
                mbar_arrive(&bars[kLReady]);
                // e4m3 cache: stage the next piece's Q once the piece's last
                // Q.K^T has completed (no Q.K^T reads the TMEM Q panels any
                // more).  The owner of the last pair is the busier group here
                // (it widens as well), so this one takes the staging, with no
                // logits live; in the bf16 kernel the owner staging at once is
                // faster.  The wait cannot alias: the barrier's next phase
                // needs a Q.K^T of the next piece, i.e. this staging.
                if constexpr (FP8) {
                    if (!wait_all(&bars[kSFull + (plast & 1)], (plast >> 1) & 1, false)) {
                        ok = false;
                        widened = gp + npairs;
                        break;
                    }
                    tc_fence_after();
                    stage_q(it);
                }
            } else {
                if (!wait_all(&bars[kLReady], kpiece & 1, false) || !wait_own_pv(plast)) {
                    ok = false;
                    widened = gp + npairs;
                    break;
                }
                const float lo = lh_s[h], mo = mh_s[h];
                const float l_run = l_part + (mo == -INFINITY ? 0.f : lo * ex2(mo - m_l));
                const float m_fin = m_l;
                tc_fence_after();
                const float inv = l_run > 0.f ? a.out_scale / l_run : 0.f;
                for (int c0 = 0; c0 < C::kOCols; c0 += 32) {
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
                if (live_row && rank == 0) {
                    const float lse = l_run > 0.f ? (m_fin + log2f(l_run)) * kLn2 : -INFINITY;
                    if (pc.whole) {
                        if (a.lse) a.lse[static_cast<long long>(pc.b) * a.H + h] = lse;
                    } else {
                        a.ws_lse[static_cast<long long>(pc.slot) * a.H + h] = lse;
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[kOFree]);
            }
            gp += npairs;
            ++kpiece;
        }
        if (!ok) {
            report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            if constexpr (FP8) drain_widen(widened);
        }
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

template <int D, int R, bool FP8>
static cudaError_t launch_mla_tc(const MlaTcArgs& a, int clusters, cudaStream_t stream) {
    using C = MlaTcCfg<D, R>;
    const size_t smem = C::smem_bytes(a.plan.batch);
    // the cost-balanced plan serves the bf16 kernel only (the host sets no
    // piece cost for an e4m3 cache), so no e4m3 kernel is built with it
    constexpr int kCostMode = FP8 ? kModeBalanced : kModeCost;
    const bool cost = a.plan.piece_cost > 0 && !a.plan.per_seq;
    auto kern = a.q_len > 1 ? (cost ? mla_decode_tc_kernel<D, R, FP8, true, kCostMode>
                                    : mla_decode_tc_kernel<D, R, FP8, true, kModeBalanced>)
                : a.plan.fixed_splits ? mla_decode_tc_kernel<D, R, FP8, false, kModeFixed>
                : cost                ? mla_decode_tc_kernel<D, R, FP8, false, kCostMode>
                                      : mla_decode_tc_kernel<D, R, FP8, false, kModeBalanced>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(2 * clusters), dim3(C::kThreads), smem, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t mla_tc_stage1(const MlaTcArgs& a, int D, bool fp8, int clusters, cudaStream_t stream) {
    if (D == 576) return fp8 ? launch_mla_tc<576, 512, true>(a, clusters, stream)
                             : launch_mla_tc<576, 512, false>(a, clusters, stream);
    return fp8 ? launch_mla_tc<320, 256, true>(a, clusters, stream) : launch_mla_tc<320, 256, false>(a, clusters, stream);
}

int mla_tc_tile() { return MlaTcCfg<576, 512>::kTile; }

}  // namespace mqa
