// Work decomposition shared by the stage-1 kernels and the stage-2 merge.
//
// The KV pages of all requests are laid end to end: request b owns the
// global page range [cum[b], cum[b+1]), cum[b+1] - cum[b] = ceil(len_b / page).
//
//  * per-request mode (num_kv_splits == 1): work unit g is request g.  One
//    thread block walks the whole request in order and writes the final
//    output; the result does not depend on the other requests
//    (batch-invariant, bitwise reproducible).
//  * balanced mode (num_kv_splits >= 2): the T pages are cut into `units`
//    contiguous ranges of (almost) equal length, unit g owning pages
//    [floor(g*T/units), floor((g+1)*T/units)).  A unit that covers a whole
//    request writes its final output directly; otherwise each (unit, request)
//    overlap produces one partial (O normalised, lse) in workspace slot
//    g + b, and the stage-2 merge combines the partials of each request by
//    LogSumExp (attention-kernel tutorial page, lshu.cn/news/265860, §12).
//    Along the staircase of overlaps g + b strictly increases, so slots are
//    unique and lie below units + B - 1 <= B * num_kv_splits when
//    units <= B * (num_kv_splits - 1) + 1 (the host enforces this).
//  * fixed-split mode (fixed_splits = S >= 2, its own kernel instantiations
//    through FixedPieceIter): every request is cut into S page ranges of
//    L = ceil(pages / S) pages, the split of the Triton MLA backend (one
//    program per request and split: "Triton と MLA" page, 主要ファイル /
//    データフロー; tutorial page §12), and unit g takes range g % S of
//    request g / S, writing its partial to slot g.  A request's reduction
//    order then depends on nothing but its own length and S: the result is
//    batch-invariant at any S.  Range 0 of a request that fits one range (or
//    has no page) writes the final output directly.
#pragma once

#include "common.cuh"

namespace mqa {

struct Plan {
    int batch;
    int page;
    int max_blocks;
    int units;
    int per_seq;
    int fixed_len;     // > 0: every request has this length (sparse decode: its index list)
    int fixed_splits;  // >= 2: fixed-split mode with this many ranges per request, else 0
    int piece_cost;    // balanced mode through CostPieceIter: pages charged per request start
};

// The length the plan gives request b: fixed_len, or its clamped seq_len.
__device__ __forceinline__ int clamp_len(int n, int max_blocks, int page, int* status);
__device__ __forceinline__ int plan_len(const Plan& p, const int32_t* seq_lens, int b, int* status) {
    return p.fixed_len > 0 ? p.fixed_len : clamp_len(seq_lens[b], p.max_blocks, p.page, status);
}

// Clamp a request length to [0, max_blocks * page]; report out-of-range values.
__device__ __forceinline__ int clamp_len(int n, int max_blocks, int page, int* status) {
    const long long cap = static_cast<long long>(max_blocks) * page;
    if (n < 0) {
        report(status, MQA_ERR_DEVICE_CHECK);
        return 0;
    }
    if (n > cap) {
        report(status, MQA_ERR_DEVICE_CHECK);
        return static_cast<int>(cap);
    }
    return n;
}

// Fill cum[0..B] (shared memory) with the exclusive page prefix and lens[b]
// with the clamped request lengths; every thread of the block must call this.
// Returns T = cum[B].
__device__ __forceinline__ int build_cum(const Plan& p, const int32_t* __restrict__ seq_lens,
                                         int* cum, int* lens, int* status) {
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
        const int n = plan_len(p, seq_lens, i, status);
        lens[i] = n;
        cum[i + 1] = (n + p.page - 1) / p.page;
    }
    if (threadIdx.x == 0) cum[0] = 0;
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int running = 0;
        for (int base = 0; base < p.batch; base += 32) {
            const int i = base + lane;
            int v = i < p.batch ? cum[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (i < p.batch) cum[i + 1] = running + v;
            running += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
    return cum[p.batch];
}

// Largest b in [0, B) with cum[b] <= pg: the request that owns global page pg
// (empty requests share their cum value with the next one and are skipped).
__device__ __forceinline__ int seq_of_page(const int* cum, int B, int pg) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= pg)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Balanced mode: the unit whose page range holds global page pg (T > 0).
__device__ __forceinline__ int unit_of_page(int units, int T, int pg) {
    return static_cast<int>(((static_cast<long long>(pg) + 1) * units - 1) / T);
}

__device__ __forceinline__ void unit_range(const Plan& p, const int* cum, int T, int g, int& p0,
                                           int& p1) {
    if (p.per_seq) {
        p0 = cum[g];
        p1 = cum[g + 1];
    } else {
        p0 = static_cast<int>(static_cast<long long>(g) * T / p.units);
        p1 = static_cast<int>(static_cast<long long>(g + 1) * T / p.units);
    }
}

// One (unit, request) overlap: local pages [j0, j1) of request b.
struct Piece {
    int b, j0, j1;
    int whole;  // the unit covers the request entirely: write the final output
    int slot;   // workspace partial slot (balanced mode)
};

// Iterates over the pieces of unit g in page order.  Per-request mode yields
// exactly one piece (possibly with no pages) so that empty requests still get
// their output written.
struct PieceIter {
    int g, B, p, p1, b, first_done;
    int per_seq;

    __device__ __forceinline__ void init(const Plan& plan, const int* cum, int T, int unit) {
        g = unit;
        B = plan.batch;
        per_seq = plan.per_seq;
        int p0;
        unit_range(plan, cum, T, unit, p0, p1);
        p = p0;
        b = per_seq ? unit : (p0 < p1 ? seq_of_page(cum, B, p0) : 0);
        first_done = 0;
    }

    __device__ __forceinline__ bool next(const int* cum, Piece& pc) {
        if (per_seq) {
            if (first_done) return false;
            first_done = 1;
            pc.b = b;
            pc.j0 = 0;
            pc.j1 = cum[b + 1] - cum[b];
            pc.whole = 1;
            pc.slot = 0;
            return true;
        }
        if (p >= p1) return false;
        while (cum[b + 1] <= p) ++b;  // skip empty requests
        const int end = min(p1, cum[b + 1]);
        pc.b = b;
        pc.j0 = p - cum[b];
        pc.j1 = end - cum[b];
        pc.whole = (pc.j0 == 0 && end == cum[b + 1]) ? 1 : 0;
        pc.slot = g + b;
        p = end;
        return true;
    }
};

// Balanced mode in which every request also costs c = piece_cost pages for
// its start (a new request costs its units a query staging and a pipeline
// fill): request b spans the positions [cum[b] + c b, cum[b + 1] + c (b + 1)),
// its pages the last cum[b + 1] - cum[b] of them, and unit g takes the
// positions [g CT / units, (g + 1) CT / units), CT = T + c B.  A unit then
// holds fewer pages the more requests it starts.  Pieces, whole-request flags
// and slots (g + b along the same staircase) are as in PieceIter, which this
// is with c = 0; the merge maps pages to units by the same positions.
struct CostPieceIter {
    int g, B, c, x0, x1, b;

    __device__ __forceinline__ void init(const Plan& plan, const int* cum, int T, int unit) {
        g = unit;
        B = plan.batch;
        c = plan.piece_cost;
        const long long CT = T + static_cast<long long>(c) * B;
        x0 = static_cast<int>(static_cast<long long>(unit) * CT / plan.units);
        x1 = static_cast<int>(static_cast<long long>(unit + 1) * CT / plan.units);
        int lo = 0, hi = B - 1;  // the last request starting at or before x0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] + c * mid <= x0)
                lo = mid;
            else
                hi = mid - 1;
        }
        b = lo;
    }

    __device__ __forceinline__ bool next(const int* cum, Piece& pc) {
        while (b < B && cum[b] + c * b < x1) {
            const int first = cum[b] + c * (b + 1);  // position of the request's page 0
            const int np = cum[b + 1] - cum[b];
            const int j0 = max(x0 - first, 0);
            const int j1 = min(x1 - first, np);
            const int bb = b++;
            if (j1 > j0) {
                pc.b = bb;
                pc.j0 = j0;
                pc.j1 = j1;
                pc.whole = (j0 == 0 && j1 == np) ? 1 : 0;
                pc.slot = g + bb;
                return true;
            }
        }
        return false;
    }
};

// Fixed-split mode's iterator: unit g yields one piece, range g % S of
// request g / S (possibly without pages), with the interface of PieceIter.
struct FixedPieceIter {
    int g, b, j0, j1, whole, done;

    __device__ __forceinline__ void init(const Plan& plan, const int* cum, int, int unit) {
        const int S = plan.fixed_splits;
        g = unit;
        b = unit / S;
        const int s = unit - b * S;
        const int np = cum[b + 1] - cum[b];
        const int L = (np + S - 1) / S;
        j0 = min(s * L, np);
        j1 = min(j0 + L, np);
        whole = (s == 0 && j1 == np) ? 1 : 0;
        done = 0;
    }

    __device__ __forceinline__ bool next(const int*, Piece& pc) {
        if (done) return false;
        done = 1;
        pc.b = b;
        pc.j0 = j0;
        pc.j1 = j1;
        pc.whole = whole;
        pc.slot = g;
        return true;
    }
};

// Producer-side flat walk over the tiles of a unit: `tile` tokens at a time,
// skipping pieces that hold no token.  After next() returns true, tokens
// [t0, min(t0 + tile, tok_end)) of request pc.b are the current tile and `bt`
// points at that request's block-table row.
template <class Iter>
struct TileCursorT {
    Iter it;
    Piece pc;
    int t0, tok_end, tile;
    const int32_t* bt;

    __device__ __forceinline__ void init(const Plan& plan, const int* cum, int T, int unit,
                                         int tile_tokens) {
        it.init(plan, cum, T, unit);
        t0 = 0;
        tok_end = 0;
        tile = tile_tokens;
        bt = nullptr;
    }

    __device__ __forceinline__ bool next(const Plan& plan, const int* cum, const int* lens,
                                         const int32_t* __restrict__ block_table) {
        t0 += tile;
        while (t0 >= tok_end) {
            if (!it.next(cum, pc)) return false;
            t0 = pc.j0 * plan.page;
            tok_end = min(pc.j1 * plan.page, lens[pc.b]);
            bt = block_table + static_cast<long long>(pc.b) * plan.max_blocks;
        }
        return true;
    }
};
using TileCursor = TileCursorT<PieceIter>;

}  // namespace mqa
