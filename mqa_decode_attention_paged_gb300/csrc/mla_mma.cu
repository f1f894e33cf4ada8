// MLA decode, stage 1, warp-level tensor-core path (any head count, 16 heads
// per thread block).
//
// One thread block = 8 consumer warps + 1 producer warp, persistent over a
// work unit (see plan.cuh).  The producer walks the block table (prefetching
// the next tile's block ids while it waits for a free stage) and stages
// kTile-token tiles of latent rows [kv_c | k_pe] into shared memory: one 3D
// tensor copy per box of whole rows of a page (128-byte swizzle), or, for
// sparse decode, one four-row gather per four selected rows.  Rows past the
// sequence end (or unselected) are masked and their V columns zeroed by the
// consumers.
// The same staged tile serves as K (all D columns) and V (first R columns),
// the MQA view of MLA ("Triton と MLA" page, vllm-arch-zh
// ja/attention/triton-mla, section データフロー).
//
// Per tile the consumers compute
//   S = Q K^T  (16 heads x kTile tokens; 8 warps = 2 token halves x 4
//               quarters of the head dimension, partial sums reduced in smem),
//   online softmax per head (tutorial page lshu.cn/news/265860, §7: running
//   max m, running sum l, rescale alpha = 2^(m_old - m_new) in base 2 with
//   log2(e) folded into the scale),
//   O = alpha O + P V (each warp owns R/8 output columns).
// fp8-e4m3 tiles are first widened to bf16 in shared memory (exact); k_scale
// is folded into the logit scale and into the output.
#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "plan.cuh"
#include "args.cuh"

namespace mqa {

// Four-row gather of a 2D tensor (box one row high) into shared memory: rows
// y0 .. y3, columns x .. x + box - 1 each, landing back to back; completes its
// bytes (four boxes, out-of-range fill included) on `bar`.  x must be a
// multiple of 16 bytes' worth of elements; dst 128-byte aligned.
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared-memory budget: everything but the staging ring is fixed, the ring
// gets as many stages as fit (at most 8).

// SPARSE: the stage is filled by four-row gathers (`tile::gather4` tensor
// copies of whole rows seen as 8-byte elements), one per group of four
// consecutive tile rows.  A group lands its rows back to back at a 128-byte
// aligned place.  bf16 rows are padded to D * 2 + 32 bytes by the copy's own
// out-of-range fill, the data at the start of the row in even groups and 16
// bytes in (the box starts at element -2) in odd ones: the eight rows of two
// groups then start on eight different 16-byte bank groups, so ldmatrix
// reads them in place without conflicts.  e4m3 rows land dense and are
// widened into the swizzled operand tile as for the dense e4m3 path.
template <int D, int R, bool FP8, int TILE, bool SPARSE = false>
struct MlaMmaCfg {
    static constexpr bool kStaged = FP8;                       // operand tile built from the stage
    static constexpr bool kPadRows = SPARSE && !FP8;           // stage rows padded by 32 bytes
    static constexpr int kHeads = 16;
    static constexpr int kTile = TILE;                         // tokens per stage
    static constexpr int kHalf = kTile / 2;                    // tokens per QK warp
    static constexpr int kTokPerThread = kTile / 16;           // softmax tokens per thread
    static constexpr int kConsumerWarps = 8;
    static constexpr int kConsumers = 32 * kConsumerWarps;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kPanels = D / 64;                     // 64-column bf16 panels
    static constexpr int kOpBytes = kPanels * kTile * 128;     // swizzled bf16 operand tile
    static constexpr int kRowStride = kPadRows ? D * 2 + 32 : D * (FP8 ? 1 : 2);  // bytes per staged row
    static constexpr int kGroupBytes = 4 * kRowStride;         // one four-row gather (SPARSE)
    static constexpr int kStageBytes = kTile * kRowStride;     // whole cache rows
    static constexpr int kKSteps = D / 16;
    static constexpr int kKq = kKSteps / 4;                    // k-steps per head-dim quarter
    static constexpr int kColsPerWarp = R / kConsumerWarps;    // output columns per warp
    static constexpr int kNbPV = kColsPerWarp / 8;             // n-blocks per warp in P.V
    static constexpr int kRedStride = kTile + 8;               // floats
    static constexpr int kPStride = kTile + 8;                 // bf16 elements

    static constexpr int kQStride = D * 2 + 16;                // padded smem Q row (bytes)
    static constexpr int kQBytes = 2 * kHeads * kQStride;      // double-buffered Q slot
    static constexpr int kRedBytes = 4 * kHeads * kRedStride * 4;
    static constexpr int kPBytes = kHeads * kPStride * 2;
    static constexpr int kMiscBytes = kHeads * 4 + kHeads * 8 + 8 * 8 + 16 * 8 + 16;
    static constexpr int kFixed = 1024 + (kStaged ? kOpBytes : 0) + kQBytes + kRedBytes + kPBytes + kMiscBytes +
                                  4 * (2 * kMaxBatchSmem + 1) + 1024;
    static constexpr int kStagesFit = (227 * 1024 - kFixed) / kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;

    // Byte offset of bf16 element (row, col) of the tile the consumers read:
    // padded rows of four-row groups for the bf16 gather, else whole rows in
    // the 128-byte swizzled layout of the tensor copies (or of the widened
    // operand tile).
    __device__ __forceinline__ static uint32_t op_addr(int row, int col) {
        if constexpr (kPadRows)
            return static_cast<uint32_t>((row >> 2) * kGroupBytes + (row & 3) * kRowStride + ((row >> 2) & 1) * 16 +
                                         col * 2);
        else
            return swz_rows(row, col, kPanels);
    }

    static constexpr int align1k(int x) { return (x + 1023) & ~1023; }
    static constexpr int kOffStages = 0;
    static constexpr int kOffOp = align1k(kStages * kStageBytes);
    static constexpr int kOffQ = kOffOp + (kStaged ? kOpBytes : 0);
    static constexpr int kOffRed = kOffQ + kQBytes;
    static constexpr int kOffP = kOffRed + kRedBytes;
    static constexpr int kOffAlpha = kOffP + kPBytes;
    static constexpr int kOffMl = kOffAlpha + kHeads * 4;
    static constexpr int kOffMask = kOffMl + kHeads * 8;
    static constexpr int kOffBars = kOffMask + 8 * 8;
    static constexpr int kOffFlags = kOffBars + 16 * 8;
    static constexpr int kOffCum = kOffFlags + 16;
    // +1024: the dynamic window is re-aligned to 1024 bytes in the kernel
    static size_t smem_bytes(int batch) { return 1024 + kOffCum + 4 * (2 * batch + 1); }

    static_assert(kTile == 32 || kTile == 64, "tile of 32 or 64 tokens");
    static_assert(kStages >= 2, "at least two pipeline stages");
    static_assert(D % 64 == 0 && kKSteps % 4 == 0, "head size must split into 4 quarters");
    static_assert(kColsPerWarp % 16 == 0, "P.V columns per warp must be a multiple of 16");
    static_assert(kStageBytes % (SPARSE ? 128 : 1024) == 0, "stages stay aligned for their copies");
    static_assert(!SPARSE || (kGroupBytes % 128 == 0 && kTile % 4 == 0), "gathered groups stay 128-byte aligned");
    static_assert(!kPadRows || (kRowStride % 128 == 32), "padded rows: groups of four fill bank groups 0, 2, 4, 6");
    static_assert(kPanels % 2 == 1, "odd panel count keeps ldmatrix conflict free");
    static_assert(1024 + kOffCum + 4 * (2 * kMaxBatchSmem + 1) <= 227 * 1024, "shared memory budget");
};

// MULTI: multi-token decode (per-row key limits); the plain-decode kernels
// are compiled without that code.  FIXED: fixed-split mode (one unit per
// request and range), separate instantiations.
template <int D, int R, bool FP8, int TILE, bool MULTI, bool SPARSE, bool FIXED>
__global__ void __launch_bounds__(MlaMmaCfg<D, R, FP8, TILE, SPARSE>::kThreads, 1)
    mla_decode_mma_kernel(const __grid_constant__ MlaArgs a) {
    using C = MlaMmaCfg<D, R, FP8, TILE, SPARSE>;
    using PIter = std::conditional_t<FIXED, FixedPieceIter, PieceIter>;
    using Cursor = TileCursorT<PIter>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned window: the 128-byte swizzle pattern is a function of
    // address bits 7..9.
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
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
    int* lens = cum + a.plan.batch + 1;

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
        prefetch_tmap(&a.tmap);
    }
    // Zero the staging ring (and the widened operand tile) once so that rows
    // never written by a copy hold finite values.
    for (int i = threadIdx.x * 16; i < C::kOffRed; i += C::kThreads * 16)
        *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    // Inputs may come from the previous grid in the stream.
    pdl_wait();
    pdl_launch_dependents();
    const int T = build_cum(a.plan, a.seq_lens, cum, lens, a.status);  // contains __syncthreads

    const int P = a.plan.page;

    if (warp == C::kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_policy_evict_first();
        if constexpr (SPARSE) {
            // Sparse decode: a tile is kTile entries of the request's index
            // list; lane l looks up entries l, l + 32 and lane g < kTile / 4
            // gathers rows 4g .. 4g + 3 by one four-row tensor copy into the
            // stage (bf16: padded rows, read in place; e4m3: dense rows,
            // widened by the consumers).  The two dependent lookups of a row (its
            // index entry, then its block id) are spread over the two tiles
            // before its own: in the turn of tile i the producer reads the
            // block ids of tile i + 1 and the entries of tile i + 2, then
            // waits for the stage and copies tile i, so no read waits on
            // another within one turn and both are in flight during the wait.
            // Entries outside [0, seq_len) select nothing; bad block ids are
            // reported.
            static_assert(C::kTile % 32 == 0, "whole warps of rows");
            constexpr int kPer = C::kTile / 32;
            constexpr int kGroups = C::kTile / 4;
            // look-ahead in tiles of the index-entry and block-id reads
            constexpr int kAheadE = 2, kAheadB = 1;
            static_assert(kGroups <= 32, "one four-row group per lane");
            const long long cap = static_cast<long long>(a.bt_stride) * a.cache_page;
            struct Look {
                int b, n;        // request and its length (seq_lens[b])
                int pos[kPer];   // selected position, -1 for none
                int blk[kPer];   // block id of the position's page
                bool val[kPer];  // position selects a row of a mapped page
            };
            // first lookup: the tile's entries and its request's length
            auto read_entries = [&](const Cursor& tc, Look& L) {
                L.b = tc.pc.b;
                L.n = __ldg(a.seq_lens + L.b);
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int e = tc.t0 + lane + 32 * k;
                    L.pos[k] = e < tc.tok_end ? __ldg(a.indices + static_cast<long long>(L.b) * a.topk + e) : -1;
                }
            };
            // second lookup: the block ids of the selected positions
            auto read_blocks = [&](Look& L) {
                if (L.n < 0 && lane == 0) report(a.status, MQA_ERR_DEVICE_CHECK);
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int pos = L.pos[k];
                    bool v = pos >= 0 && pos < L.n;
                    if (v && pos >= cap) {
                        // below the length but beyond what the block table maps
                        report(a.status, MQA_ERR_DEVICE_CHECK);
                        v = false;
                    }
                    L.val[k] = v;
                    L.blk[k] = v ? __ldg(a.block_table + static_cast<long long>(L.b) * a.bt_stride + pos / a.cache_page)
                                 : 0;
                }
            };
            Cursor cur;
            cur.init(a.plan, cum, T, unit, C::kTile);
            int stage = 0;
            uint32_t phase = 0;
            int issued[C::kStages];
            for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
            Look L[kAheadE + 1];
            bool h[kAheadE + 1];
            bool more = unit != a.withhold;  // test hook
#pragma unroll
            for (int j = 0; j < kAheadE; ++j) {
                h[j] = more && cur.next(a.plan, cum, lens, a.block_table);
                more = h[j];
                if (h[j]) read_entries(cur, L[j]);
            }
#pragma unroll
            for (int j = 0; j < kAheadB; ++j)
                if (h[j]) read_blocks(L[j]);
            while (h[0]) {
                if (h[kAheadB]) read_blocks(L[kAheadB]);
                h[kAheadE] = h[kAheadE - 1] && cur.next(a.plan, cum, lens, a.block_table);
                if (h[kAheadE]) read_entries(cur, L[kAheadE]);
                Look& L0 = L[0];
                if (!mbar_wait(&empty[stage], phase ^ 1)) {
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                    break;
                }
                uint8_t* dst = stages + stage * C::kStageBytes;
                int row[kPer];  // the entry's row in the {D * elt / 8, num_blocks * page} view
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    bool v = L0.val[k];
                    if (v && (L0.blk[k] < 0 || L0.blk[k] >= a.num_blocks)) {
                        report(a.status, MQA_ERR_DEVICE_CHECK);
                        v = false;
                    }
                    L0.val[k] = v;
                    row[k] = v ? L0.blk[k] * a.cache_page + L0.pos[k] % a.cache_page : 0;
                }
                uint64_t vmask = 0;
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                    vmask |= static_cast<uint64_t>(__ballot_sync(0xffffffffu, L0.val[k])) << (32 * k);
                // group `lane`: rows 4 lane .. 4 lane + 3, from the lanes
                // holding those entries; an unselected row repeats a selected
                // one of its group (masked by the consumers), and a group with
                // none is not copied
                int y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = (4 * lane + i) & (C::kTile - 1);
                    int r = 0;
#pragma unroll
                    for (int k = 0; k < kPer; ++k) {
                        const int rk = __shfl_sync(0xffffffffu, row[k], e & 31);
                        if ((e >> 5) == k) r = rk;
                    }
                    y[i] = r;
                }
                const uint32_t gbits = lane < kGroups ? static_cast<uint32_t>(vmask >> (4 * lane)) & 0xfu : 0u;
                const int yf = (gbits & 1u) ? y[0] : (gbits & 2u) ? y[1] : (gbits & 4u) ? y[2] : y[3];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (!((gbits >> i) & 1u)) y[i] = yf;
                const uint32_t gm = __ballot_sync(0xffffffffu, gbits != 0u);
                if (lane == 0) {
                    mask_s[stage] = vmask;
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(__popc(gm)) * C::kGroupBytes);
                }
                __syncwarp();
                // bf16: odd groups start their box at element -2, so their
                // rows' data sits 16 bytes in (see MlaMmaCfg)
                if (gbits)
                    tma_gather4(dst + lane * C::kGroupBytes, &a.tmap, (C::kPadRows && (lane & 1)) ? -2 : 0, y[0], y[1],
                                y[2], y[3], &full[stage], pol);
                issued[stage] = static_cast<int>(phase);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1;
                }
#pragma unroll
                for (int j = 0; j < kAheadE; ++j) {
                    L[j] = L[j + 1];
                    h[j] = h[j + 1];
                }
            }
            for (int s = 0; s < C::kStages; ++s)
                if (issued[s] >= 0 && !mbar_wait(&full[s], static_cast<uint32_t>(issued[s])))
                    report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            return;
        }
        Cursor cur;
        cur.init(a.plan, cum, T, unit, C::kTile);
        int stage = 0;
        uint32_t phase = 0;
        int issued[C::kStages];
        for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
        const int BR = a.box_rows;  // rows per tensor box (never straddles a page)
        const int nbox = C::kTile / BR;
        constexpr int kRowBytes = D * (FP8 ? 1 : 2);

        // Block id of box `lane` of the next tile, fetched one tile ahead.
        auto fetch = [&](const Cursor& tc, int& blk, bool& val) {
            const int tok = tc.t0 + lane * BR;
            val = lane < nbox && tok < tc.tok_end;
            blk = val ? tc.bt[tok / P] : 0;
        };
        // test hook: the producer of the withheld unit fills and announces
        // nothing, so its consumers' first wait runs out
        bool have = unit != a.withhold && cur.next(a.plan, cum, lens, a.block_table);
        int blk = 0;
        bool val = false;
        int t0 = cur.t0, tend = cur.tok_end;
        if (have) fetch(cur, blk, val);
        while (have) {
            const bool have_next = cur.next(a.plan, cum, lens, a.block_table);
            int nblk = 0;
            bool nval = false;
            if (have_next) fetch(cur, nblk, nval);

            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
                break;
            }
            uint8_t* dst = stages + stage * C::kStageBytes;
            if (val && (blk < 0 || blk >= a.num_blocks)) {
                report(a.status, MQA_ERR_DEVICE_CHECK);
                val = false;
            }
            // One tensor copy per box of BR whole rows.  Rows of a box past
            // the sequence end arrive too; the consumers mask their logits
            // and zero their V columns.
            const uint32_t bm = __ballot_sync(0xffffffffu, val);
            const int n_tok = tend - t0;
            uint64_t vmask = n_tok >= 64 ? ~0ull : ((1ull << n_tok) - 1);
            const uint64_t box_ones = BR == 64 ? ~0ull : ((1ull << BR) - 1);
            for (int bx = 0; bx < nbox; ++bx)
                if (!((bm >> bx) & 1u)) vmask &= ~(box_ones << (bx * BR));
            if (lane == 0) {
                mask_s[stage] = vmask;
                mbar_arrive_expect_tx(&full[stage], __popc(bm) * BR * kRowBytes);
            }
            __syncwarp();
            if (val) {
                const int row = blk * P + (t0 + lane * BR) % P;
                tma_load_3d(dst + lane * BR * kRowBytes, &a.tmap, 0, 0, row, &full[stage], pol);
            }
            issued[stage] = static_cast<int>(phase);
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1;
            }
            have = have_next;
            t0 = cur.t0;
            tend = cur.tok_end;
            blk = nblk;
            val = nval;
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
    const int t = threadIdx.x;                // softmax role: head sh, tokens sk*kTPT ..
    const int sh = t >> 4, sk = t & 15;
    constexpr int kTPT = C::kTokPerThread;
    constexpr uint64_t kFullMask = C::kTile == 64 ? ~0ull : ((1ull << C::kTile) - 1);

    // Q rows h0 .. h0+15 of request b are staged into one of two padded smem
    // slots with cp.async one piece ahead of their use (rows beyond H are
    // zero-filled); each warp then builds its A fragments with ldmatrix.
    uint8_t* qslot = smem + C::kOffQ;
    auto stage_q = [&](int b, int buf) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.q + (static_cast<long long>(b) * a.H + h0) * D);
        uint8_t* dst = qslot + buf * C::kHeads * C::kQStride;
        for (int i = t; i < C::kHeads * (D / 8); i += C::kConsumers) {
            const int row = i / (D / 8), ch = i % (D / 8);
            const bool live = h0 + row < a.H;
            cp_async_16(dst + row * C::kQStride + ch * 16, live ? src + (row * D + ch * 8) * 2 : src,
                        live ? 16 : 0);
        }
        cp_async_commit();
    };
    auto load_q = [&](int buf, uint32_t (&qf)[C::kKq][4]) {
        const uint8_t* base = qslot + buf * C::kHeads * C::kQStride;
#pragma unroll
        for (int ks = 0; ks < C::kKq; ++ks) {
            const int col = (dq * C::kKq + ks) * 16 + (lane >> 4) * 8;
            ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], base + (lane & 15) * C::kQStride + col * 2);
        }
    };

    PIter it;
    it.init(a.plan, cum, T, unit);
    Piece pc;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;
    bool have = it.next(cum, pc);
    int qbuf = 0;
    if (have) stage_q(pc.b, 0);

    while (!aborted && have) {
        const int len = lens[pc.b];
        // multi-token decode: the softmax row sh (token i = row / heads) sees
        // tokens below len - q_len + i + 1 (tutorial page §10); len otherwise
        const int row_lim = MULTI ? len - (a.q_len - 1 - (h0 + sh) / a.heads) : len;
        const int tok0 = pc.j0 * P;
        const int tok_end = min(pc.j1 * P, len);
        Piece nxt;
        const bool have_next = it.next(cum, nxt);
        uint32_t qa[C::kKq][4];
        cp_async_wait_all();
        named_bar_sync(4, C::kConsumers);  // this piece's Q slot is complete
        load_q(qbuf, qa);
        // the other slot held the previous piece's Q, read before its epilogue
        if (have_next) stage_q(nxt.b, qbuf ^ 1);

        float o[C::kNbPV][4];
#pragma unroll
        for (int i = 0; i < C::kNbPV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;  // softmax role, head sh

        for (int t0 = tok0; t0 < tok_end; t0 += C::kTile) {
            // decided per warp: the MMAs below are warp-collective
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase));
            if (!ok) {
                *abort_s = 1;
                report(a.status, MQA_ERR_DEVICE_TIMEOUT);
            }
            uint8_t* stage_buf = stages + stage * C::kStageBytes;
            uint8_t* op = stage_buf;
            const uint64_t vmask = mask_s[stage];
            bool zeroed = false;
            if constexpr (C::kStaged) {
                // Widen the e4m3 tile to bf16 (exact) into the swizzled
                // operand tile.
                op = smem + C::kOffOp;
                named_bar_sync(3, C::kConsumers);  // previous tile's P.V is done
                if (ok) {
                    constexpr int kChunks = C::kTile * (D / 16);
                    for (int i = t; i < kChunks; i += C::kConsumers) {
                        const int r = i / (D / 16), cc = i % (D / 16);
                        const uint4 v = *reinterpret_cast<const uint4*>(stage_buf + r * D + cc * 16);
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
                        *reinterpret_cast<uint4*>(op + swz_rows(r, 16 * cc, C::kPanels)) =
                            make_uint4(outw[0], outw[1], outw[2], outw[3]);
                        *reinterpret_cast<uint4*>(op + swz_rows(r, 16 * cc + 8, C::kPanels)) =
                            make_uint4(outw[4], outw[5], outw[6], outw[7]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                named_bar_sync(3, C::kConsumers);
            }
            if (vmask != kFullMask) {
                // Rows past the sequence end may hold anything (the tail of a
                // page, or an earlier tile): zero them in the V columns this
                // warp reads, so P = 0 never meets a NaN.  K columns of those
                // rows only reach logits that the mask replaces with -inf.
                constexpr int kChunksPerWarp = C::kColsPerWarp / 8;
                for (int i = lane; i < C::kTile * kChunksPerWarp; i += 32) {
                    const int r = i / kChunksPerWarp;
                    if (!((vmask >> r) & 1ull)) {
                        const int col = warp * C::kColsPerWarp + (i % kChunksPerWarp) * 8;
                        *reinterpret_cast<uint4*>(op + C::op_addr(r, col)) = make_uint4(0, 0, 0, 0);
                    }
                }
                zeroed = true;
                __syncwarp();
            }

            // ---- S partial = Q[:, quarter] K[tokens of half th, quarter]^T
            float sacc[C::kHalf / 8][4];
#pragma unroll
            for (int i = 0; i < C::kHalf / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < C::kKq; ++ks) {
                    const int k0 = (dq * C::kKq + ks) * 16;
#pragma unroll
                    for (int nb2 = 0; nb2 < C::kHalf / 16; ++nb2) {
                        const int row = th * C::kHalf + nb2 * 16 + (lane & 7) + ((lane >> 4) << 3);
                        const int col = k0 + ((lane >> 3) & 1) * 8;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(b0, b1, b2, b3, op + C::op_addr(row, col));
                        mma_bf16_16816(sacc[2 * nb2], qa[ks], b0, b1);
                        mma_bf16_16816(sacc[2 * nb2 + 1], qa[ks], b2, b3);
                    }
                }
            }
#pragma unroll
            for (int nb = 0; nb < C::kHalf / 8; ++nb) {
                const int col = th * C::kHalf + nb * 8 + 2 * c;
                *reinterpret_cast<float2*>(&red[(dq * 16 + g) * C::kRedStride + col]) =
                    make_float2(sacc[nb][0], sacc[nb][1]);
                *reinterpret_cast<float2*>(&red[(dq * 16 + g + 8) * C::kRedStride + col]) =
                    make_float2(sacc[nb][2], sacc[nb][3]);
            }
            named_bar_sync(1, C::kConsumers);

            // ---- online softmax for head sh over tokens sk*kTPT .. +kTPT-1
            {
                float x[kTPT];
#pragma unroll
                for (int i = 0; i < kTPT; ++i) x[i] = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float* src = &red[(q4 * 16 + sh) * C::kRedStride + kTPT * sk];
                    if constexpr (kTPT == 4) {
                        const float4 v = *reinterpret_cast<const float4*>(src);
                        x[0] += v.x;
                        x[1] += v.y;
                        x[2] += v.z;
                        x[3] += v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2*>(src);
                        x[0] += v.x;
                        x[1] += v.y;
                    }
                }
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kTPT; ++i) {
                    const bool valid = ((vmask >> (kTPT * sk + i)) & 1ull) && (!MULTI || t0 + kTPT * sk + i < row_lim);
                    x[i] = valid ? x[i] * a.sl2 : -INFINITY;
                    mx = fmaxf(mx, x[i]);
                }
#pragma unroll
                for (int o2 = 8; o2 >= 1; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                const float m_new = fmaxf(m_run, mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = ex2(m_run - m_use);
                float psum = 0.f;
                uint32_t pk[kTPT / 2];
#pragma unroll
                for (int i = 0; i < kTPT / 2; ++i) {
                    // l sums the fp32 probabilities; P.V uses them rounded to bf16
                    const float p0 = ex2(x[2 * i] - m_use), p1 = ex2(x[2 * i + 1] - m_use);
                    psum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
#pragma unroll
                for (int o2 = 8; o2 >= 1; o2 >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o2);
                l_run = l_run * alpha + psum;
                m_run = m_new;
                if constexpr (kTPT == 4)
                    *reinterpret_cast<uint2*>(&Ps[sh * C::kPStride + kTPT * sk]) = make_uint2(pk[0], pk[1]);
                else
                    *reinterpret_cast<uint32_t*>(&Ps[sh * C::kPStride + kTPT * sk]) = pk[0];
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
                            ldsm_x4_t(b0, b1, b2, b3, op + C::op_addr(tok, col));
                            mma_bf16_16816(o[2 * nb2], pa, b0, b1);
                            mma_bf16_16816(o[2 * nb2 + 1], pa, b2, b3);
                        }
                    }
                }
            }
            if constexpr (!C::kStaged) {
                // the stage goes back to the tensor copies (async proxy)
                if (zeroed) fence_proxy_async_smem();
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
        pc = nxt;
        have = have_next;
        qbuf ^= 1;
    }
    cp_async_wait_all();
}

// Tile size (tokens per pipeline stage; 32 or 64).  The number of stages is
// the largest that fits the staging budget.
#ifndef MQA_MLA_TILE
#define MQA_MLA_TILE 64
#endif
template <int D, bool FP8, bool SPARSE = false>
struct MlaTile {
    // dense, e4m3 and gathered tiles alike (a gathered bf16 tile is read in
    // place from its padded rows, so two 64-row stages fit)
    static constexpr int value = MQA_MLA_TILE;
};

template <int D, int R, bool FP8, bool MULTI, bool SPARSE, bool FIXED = false>
static cudaError_t launch_form(const MlaArgs& a, int grid, cudaStream_t stream) {
    constexpr int kTile = MlaTile<D, FP8, SPARSE>::value;
    using C = MlaMmaCfg<D, R, FP8, kTile, SPARSE>;
    const size_t smem = C::smem_bytes(a.plan.batch);
    auto kern = mla_decode_mma_kernel<D, R, FP8, kTile, MULTI, SPARSE, FIXED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(kern, dim3(grid), dim3(C::kThreads), smem, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, int R, bool FP8>
static cudaError_t launch_mla_mma(const MlaArgs& a, int grid, cudaStream_t stream) {
    if (a.indices) return launch_form<D, R, FP8, false, true>(a, grid, stream);
    if (a.q_len > 1) return launch_form<D, R, FP8, true, false>(a, grid, stream);
    if (a.plan.fixed_splits) return launch_form<D, R, FP8, false, false, true>(a, grid, stream);
    return launch_form<D, R, FP8, false, false>(a, grid, stream);
}

cudaError_t mla_mma_stage1(const MlaArgs& a, int D, bool fp8, int grid, cudaStream_t stream) {
    if (D == 576) return fp8 ? launch_mla_mma<576, 512, true>(a, grid, stream)
                             : launch_mla_mma<576, 512, false>(a, grid, stream);
    return fp8 ? launch_mla_mma<320, 256, true>(a, grid, stream)
               : launch_mla_mma<320, 256, false>(a, grid, stream);
}

int mla_mma_tile() { return MQA_MLA_TILE; }

int mla_mma_sparse_tile(bool fp8) {
    return fp8 ? MlaTile<576, true, true>::value : MlaTile<576, false, true>::value;
}

size_t mla_mma_smem_bytes(int D, bool fp8, int batch) {
    if (D == 576) return fp8 ? MlaMmaCfg<576, 512, true, MQA_MLA_TILE>::smem_bytes(batch)
                             : MlaMmaCfg<576, 512, false, MQA_MLA_TILE>::smem_bytes(batch);
    return fp8 ? MlaMmaCfg<320, 256, true, MQA_MLA_TILE>::smem_bytes(batch)
               : MlaMmaCfg<320, 256, false, MQA_MLA_TILE>::smem_bytes(batch);
}

}  // namespace mqa
