/*
 * CPU fp64 oracle for single-query paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark load this file.  The library's product
 * path never links, loads or calls it, and it shares no code, header, table or
 * helper with the CUDA kernels.
 *
 * What it computes (plain definitions, no blocking or fusion):
 *
 *   MLA-as-MQA decode.  The cache row of a token is one latent vector
 *   [kv_c (kv_lora_rank) | k_pe (rope)] of head_size D.  It is the key of every
 *   query head, and its first R = kv_lora_rank columns are the value.
 *     Sources: "Triton と MLA" page (vllm-arch-zh, ja/attention/triton-mla),
 *     sections 役割 / 設計動機 (single KV channel, head_size 320 or 576) and
 *     データフロー (the cache passed as a single-head K cache, V = its first
 *     kv_lora_rank columns, k_scale passed as both scales).
 *
 *   Paged address translation: logical block = pos / page, physical block from
 *   the request's block table, slot = physical block * page + pos % page.
 *     Source: attention-kernel tutorial page (lshu.cn/news/265860), §11
 *     "Paged KV Cache 如何参与计算".
 *
 *   Decode has no mask: the single query sits after every cached key.
 *     Source: tutorial page §9.
 *
 *   Online softmax (running max m, sum l, accumulator acc, rescale factor
 *   alpha = exp(m_old - m_new)).  Source: tutorial page §7.
 *
 *   Split-KV segments merged by m = max m_s, l = sum_s exp(m_s - m) l_s,
 *   O = sum_s exp(m_s - m) O_s / l.  Source: tutorial page §12.
 *
 *   Number of KV splits: ceil(max_seq_len / 512) capped at 2 * sm_count, and 1
 *   in batch-invariant mode.  Source: "Triton と MLA" page, 主要ファイル
 *   (_compute_num_kv_splits) and データフロー (VLLM_BATCH_INVARIANT branch).
 *
 *   Multi-token decode (several new positions of a request verified in one
 *   call): query i of q_len sits at absolute position
 *   context_length + i, context_length = kv_length - q_len, and sees the keys
 *   at positions <= its own: a full rectangle over the history plus a
 *   q_len x q_len lower triangle.  Source: tutorial page §10
 *   ("多 Token 验证时的 Attention 结构": query_abs_position =
 *   context_length + query_local_position, mask = key_position <=
 *   query_abs_position).
 *
 *   Sparse (top-k) decode: each query attends only the key positions its
 *   request's index list selects (e.g. the top 2048), each translated to a
 *   physical slot through the request's block table.  Source: tutorial page
 *   §13 (Dense / Sparse Attention: "每个 Query 只与选中的 2048 个 Key 计算相关性",
 *   and the request's top-k logical positions converted to physical KV
 *   slots through its block table).
 *
 *   Merging the results of sequence shards (decode context parallelism): each
 *   shard g of a request's KV cache gives its normalised output O_g and its
 *   lse_g; with m = max_g lse_g the merged result is
 *   O = sum_g e^{lse_g - m} O_g / sum_g e^{lse_g - m}, lse = m + ln sum_g
 *   e^{lse_g - m}.  Source: tutorial page §12 (the split-KV merge written for
 *   normalised partials) and the "Triton と MLA" page, 設計動機 (lse is
 *   returned so that DCP shards can be merged by cp_lse_ag_out_rs).
 *
 *   The same merge taken apart for an exchange that all-gathers the lse and
 *   sums the outputs across ranks: shard g's share of the merged output is
 *   its weight times its output, e^{lse_g - lse} O_g with lse the merged lse,
 *   and the shares of all shards add up to O.  Source: the merge above; the
 *   name cp_lse_ag_out_rs (lse all-gather, output reduce-scatter) on the
 *   "Triton と MLA" page, 設計動機.
 *
 *   GQA paged decode over a [num_blocks, 2, page, num_kv_heads, head_size]
 *   cache.  Source: "AttentionBackend" page (vllm-arch-zh, fr/attention/backend),
 *   section "Motivation de conception" (FlashAttention cache layout).
 *
 *   Per-token-head quantised GQA cache (fp8_per_token_head /
 *   int8_per_token_head): every (token, KV head) vector is stored as 8-bit
 *   codes with its own scale kept inline, the head dimension padded to make
 *   room for it.  Source: "Triton と MLA" page, 役割 and 設計動機
 *   (supported_kv_cache_dtypes) and 主要ファイル (get_kv_cache_shape pads
 *   head_dim for the inline scale in per_token_head modes).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - lse is the natural log of sum_t exp(s_t) of the SCALED logits s_t.
 *   - bf16 caches ignore k_scale (the page's "is_fp8 check is a no-op").
 *   - fp8 caches are OCP e4m3fn; value = k_scale * e4m3(code) for K and V.
 *   - a sequence of length 0 gives out = 0 and lse = -inf.
 *   - sparse decode: index entries outside [0, seq_lens[b]) (e.g. -1 padding)
 *     select nothing; the others are used as listed (an index listed twice
 *     counts twice: callers pass distinct positions); none selected gives
 *     out = 0 and lse = -inf.
 *   - multi-token decode: seq_lens[b] is kv_length (history plus the q_len
 *     new tokens, whose keys are already in the cache); a query that sees no
 *     key (kv_length < q_len - i) gives out = 0 and lse = -inf.
 *   - GQA query head h reads KV head h / (Hq / Hkv).
 *   - per-token-head caches: a (token, KV head) row is its codes followed by
 *     the row's scale as a little-endian IEEE binary32; element value =
 *     scale * code, with the code read as OCP e4m3fn or as a two's-complement
 *     int8 (D bytes of codes), or as a two's-complement 4-bit code, two per
 *     byte, element 2i in the low nibble of byte i (D / 2 bytes).  K and V
 *     rows carry separate scales.
 *   - split s of a sequence with n tokens covers the page-aligned token range
 *     [s*L, min((s+1)*L, n)), L = ceil(ceil(n/page)/S) * page.
 *
 * Every public function returns 0 on success and -1 if a block-table entry that
 * a valid token needs is outside [0, num_blocks) (nothing is read then).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8_E4M3 = 1 };

/* ---- element decoders --------------------------------------------------- */

/* bf16 is the upper 16 bits of an IEEE-754 binary32; the value is exact. */
double oracle_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn": no infinities): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits.  Exponent field 0 is subnormal
 * (m * 2^-9); exponent 15 with mantissa 7 is NaN; the largest finite value is
 * 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

void oracle_bf16_values(const uint16_t* bits, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_value(bits[i]);
}

void oracle_e4m3_values(const uint8_t* codes, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]);
}

/* ---- host-side helpers named on the pages ------------------------------- */

int oracle_num_kv_splits(int max_seq_len, int sm_count, int batch_invariant) {
    if (batch_invariant) return 1;
    long s = max_seq_len <= 0 ? 1 : ((long)max_seq_len + 511) / 512;
    long cap = 2L * (long)sm_count;
    if (cap >= 1 && s > cap) s = cap;
    if (s < 1) s = 1;
    return (int)s;
}

/* Slot of logical position pos of request req (tutorial page, §11). */
int64_t oracle_physical_slot(const int32_t* block_table, int max_blocks, int req,
                             int64_t pos, int page_size) {
    int64_t logical_block = pos / page_size;
    int64_t physical_block = block_table[(int64_t)req * max_blocks + logical_block];
    return physical_block * page_size + pos % page_size;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- token access --------------------------------------------------------- */

/* Describes where token t of request b keeps its key and value vectors. */
typedef struct {
    const void* kv;
    int kv_dtype;
    const int32_t* block_table;
    int max_blocks, page, num_blocks;
    /* element offsets of (physical slot 0, plane) and per-slot stride */
    int64_t slot_stride;   /* elements between consecutive slots of one plane */
    int64_t block_stride;  /* elements between consecutive physical blocks */
    int64_t k_offset;      /* element offset of the key inside a slot */
    int64_t v_offset;      /* element offset of the value inside a slot */
    int dk, dv;            /* key and value lengths */
    double k_mult, v_mult; /* dequantisation multipliers (1 for bf16) */
} token_view;

static double elem(const token_view* tv, int64_t idx) {
    if (tv->kv_dtype == ORACLE_KV_BF16)
        return oracle_bf16_value(((const uint16_t*)tv->kv)[idx]);
    return oracle_e4m3_value(((const uint8_t*)tv->kv)[idx]);
}

/* Base element index of token t of request b, or -1 for a bad block id. */
static int64_t token_base(const token_view* tv, int b, int64_t t) {
    int64_t logical_block = t / tv->page;
    int32_t blk = tv->block_table[(int64_t)b * tv->max_blocks + logical_block];
    if (blk < 0 || blk >= tv->num_blocks) return -1;
    return (int64_t)blk * tv->block_stride + (t % tv->page) * tv->slot_stride;
}

static int check_table(const token_view* tv, int b, int n) {
    if (((int64_t)n + tv->page - 1) / tv->page > tv->max_blocks) return -1;
    for (int64_t t = 0; t < n; t += tv->page)
        if (token_base(tv, b, t) < 0) return -1;
    return 0;
}

/* Scaled logit s_t = scale * sum_d q[d] * K_t[d]. */
static double logit(const token_view* tv, const double* qd, int64_t base, double scale) {
    double acc = 0.0;
    for (int d = 0; d < tv->dk; ++d)
        acc += qd[d] * (tv->k_mult * elem(tv, base + tv->k_offset + d));
    return scale * acc;
}

/* ---- the three formulations ---------------------------------------------- */

/* Direct definition: lse = log sum_t exp(s_t) (evaluated as m + log sum
 * exp(s_t - m)), out = sum_t exp(s_t - lse) V_t. */
static int attend_direct(const token_view* tv, int b, int n, const double* qd, double scale,
                         double* out, double* lse) {
    int dv = tv->dv;
    for (int r = 0; r < dv; ++r) out[r] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return 0;
    }
    if (check_table(tv, b, n)) return -1;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        s[t] = logit(tv, qd, token_base(tv, b, t), scale);
        if (s[t] > m) m = s[t];
    }
    double sum = 0.0;
    for (int t = 0; t < n; ++t) sum += exp(s[t] - m);
    double L = m + log(sum);
    for (int t = 0; t < n; ++t) {
        double w = exp(s[t] - L);
        int64_t base = token_base(tv, b, t);
        for (int r = 0; r < dv; ++r) out[r] += w * (tv->v_mult * elem(tv, base + tv->v_offset + r));
    }
    *lse = L;
    free(s);
    return 0;
}

/* Online softmax over consecutive tiles of `tile` tokens (tutorial page §7):
 * m_new = max(m_old, rowmax S_tile); alpha = exp(m_old - m_new);
 * l_new = alpha l_old + sum exp(S_tile - m_new);
 * acc_new = alpha acc_old + exp(S_tile - m_new) V_tile;  out = acc / l. */
static int attend_streaming(const token_view* tv, int b, int n, const double* qd, double scale,
                            int tile, double* out, double* lse) {
    int dv = tv->dv;
    double* acc = (double*)calloc((size_t)dv, sizeof(double));
    double* s = (double*)malloc(sizeof(double) * (size_t)(tile > 0 ? tile : 1));
    double m = -INFINITY, l = 0.0;
    if (n > 0 && check_table(tv, b, n)) {
        free(acc);
        free(s);
        return -1;
    }
    for (int t0 = 0; t0 < n; t0 += tile) {
        int t1 = t0 + tile < n ? t0 + tile : n;
        double tile_max = -INFINITY;
        for (int t = t0; t < t1; ++t) {
            s[t - t0] = logit(tv, qd, token_base(tv, b, t), scale);
            if (s[t - t0] > tile_max) tile_max = s[t - t0];
        }
        double m_new = m > tile_max ? m : tile_max;
        double alpha = exp(m - m_new);
        double psum = 0.0;
        for (int r = 0; r < dv; ++r) acc[r] *= alpha;
        for (int t = t0; t < t1; ++t) {
            double p = exp(s[t - t0] - m_new);
            int64_t base = token_base(tv, b, t);
            psum += p;
            for (int r = 0; r < dv; ++r) acc[r] += p * (tv->v_mult * elem(tv, base + tv->v_offset + r));
        }
        l = alpha * l + psum;
        m = m_new;
    }
    for (int r = 0; r < dv; ++r) out[r] = l > 0.0 ? acc[r] / l : 0.0;
    *lse = l > 0.0 ? m + log(l) : -INFINITY;
    free(acc);
    free(s);
    return 0;
}

/* Split-KV: each segment keeps (m_s, l_s, O_s unnormalised); the segments are
 * then merged with the tutorial page's §12 formulas.  Segment s covers the
 * page-aligned token range [s*L, min((s+1)*L, n)) with
 * L = ceil(ceil(n / page) / S) * page; segments past the end are empty
 * (m_s = -inf, l_s = 0, O_s = 0) and get weight 0. */
static int attend_split(const token_view* tv, int b, int n, const double* qd, double scale,
                        int num_splits, double* out, double* lse) {
    int dv = tv->dv, S = num_splits < 1 ? 1 : num_splits;
    if (n > 0 && check_table(tv, b, n)) return -1;
    double* ms = (double*)malloc(sizeof(double) * (size_t)S);
    double* ls = (double*)malloc(sizeof(double) * (size_t)S);
    double* Os = (double*)calloc((size_t)S * (size_t)dv, sizeof(double));
    int64_t pages = ((int64_t)n + tv->page - 1) / tv->page;
    int64_t L = ((pages + S - 1) / S) * tv->page;
    for (int sp = 0; sp < S; ++sp) {
        int64_t t0 = (int64_t)sp * L, t1 = t0 + L < n ? t0 + L : n;
        double m = -INFINITY;
        for (int64_t t = t0; t < t1; ++t) {
            double st = logit(tv, qd, token_base(tv, b, t), scale);
            if (st > m) m = st;
        }
        double l = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            int64_t base = token_base(tv, b, t);
            double p = exp(logit(tv, qd, base, scale) - m);
            l += p;
            for (int r = 0; r < dv; ++r)
                Os[(size_t)sp * dv + r] += p * (tv->v_mult * elem(tv, base + tv->v_offset + r));
        }
        ms[sp] = m;
        ls[sp] = l;
    }
    double M = -INFINITY;
    for (int sp = 0; sp < S; ++sp)
        if (ms[sp] > M) M = ms[sp];
    double Lsum = 0.0;
    for (int r = 0; r < dv; ++r) out[r] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
    } else {
        for (int sp = 0; sp < S; ++sp) {
            if (ls[sp] == 0.0) continue; /* empty segment: weight 0 */
            double w = exp(ms[sp] - M);
            Lsum += w * ls[sp];
            for (int r = 0; r < dv; ++r) out[r] += w * Os[(size_t)sp * dv + r];
        }
        for (int r = 0; r < dv; ++r) out[r] /= Lsum;
        *lse = M + log(Lsum);
    }
    free(ms);
    free(ls);
    free(Os);
    return 0;
}

/* ---- MLA and GQA drivers --------------------------------------------------- */

enum { FORM_DIRECT = 0, FORM_STREAMING = 1, FORM_SPLIT = 2 };

static int run_heads(const token_view* tv, const uint16_t* q, const int32_t* seq_lens,
                     double scale, int B, int Hq, int group, int dq, double* out, double* lse,
                     int form, int param) {
    int failed = 0;
    int64_t pairs = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        (void)group;
        double* qd = (double*)malloc(sizeof(double) * (size_t)dq);
        for (int d = 0; d < dq; ++d) qd[d] = oracle_bf16_value(q[bh * dq + d]);
        int n = seq_lens[b];
        /* GQA: query head h reads KV head h / group (the view's k/v offsets
         * are those of KV head 0; add the head's offset). */
        token_view v = *tv;
        int g = h / group;
        v.k_offset += (int64_t)g * tv->dk;
        v.v_offset += (int64_t)g * tv->dv;
        double* o = out + bh * tv->dv;
        int rc;
        if (form == FORM_STREAMING)
            rc = attend_streaming(&v, b, n, qd, scale, param, o, lse + bh);
        else if (form == FORM_SPLIT)
            rc = attend_split(&v, b, n, qd, scale, param, o, lse + bh);
        else
            rc = attend_direct(&v, b, n, qd, scale, o, lse + bh);
        failed |= (rc != 0);
        free(qd);
    }
    return failed ? -1 : 0;
}

static token_view mla_view(const void* kv, int kv_dtype, const int32_t* block_table, double k_scale,
                           int D, int R, int num_blocks, int P, int max_blocks) {
    token_view tv;
    tv.kv = kv;
    tv.kv_dtype = kv_dtype;
    tv.block_table = block_table;
    tv.max_blocks = max_blocks;
    tv.page = P;
    tv.num_blocks = num_blocks;
    tv.slot_stride = D;
    tv.block_stride = (int64_t)P * D;
    tv.k_offset = 0;
    tv.v_offset = 0; /* V is the first R columns of the same row */
    tv.dk = D;
    tv.dv = R;
    tv.k_mult = kv_dtype == ORACLE_KV_FP8_E4M3 ? k_scale : 1.0;
    tv.v_mult = tv.k_mult; /* v_scale = k_scale for MLA */
    return tv;
}

/* q: bf16 bits [B, H, D]; kv: [num_blocks, P, D] bf16 bits or e4m3 codes;
 * out: [B, H, R]; lse: [B, H]. */
int oracle_mla_decode(const uint16_t* q, const void* kv, int kv_dtype, const int32_t* block_table,
                      const int32_t* seq_lens, double scale, double k_scale, double* out,
                      double* lse, int B, int H, int D, int R, int num_blocks, int P,
                      int max_blocks) {
    token_view tv = mla_view(kv, kv_dtype, block_table, k_scale, D, R, num_blocks, P, max_blocks);
    tv.dk = D; /* the whole latent row is the key */
    return run_heads(&tv, q, seq_lens, scale, B, H, H /* one KV head */, D, out, lse,
                     FORM_DIRECT, 0);
}

int oracle_mla_decode_streaming(const uint16_t* q, const void* kv, int kv_dtype,
                                const int32_t* block_table, const int32_t* seq_lens, double scale,
                                double k_scale, double* out, double* lse, int B, int H, int D,
                                int R, int num_blocks, int P, int max_blocks, int tile) {
    token_view tv = mla_view(kv, kv_dtype, block_table, k_scale, D, R, num_blocks, P, max_blocks);
    return run_heads(&tv, q, seq_lens, scale, B, H, H, D, out, lse, FORM_STREAMING,
                     tile < 1 ? 1 : tile);
}

int oracle_mla_decode_split(const uint16_t* q, const void* kv, int kv_dtype,
                            const int32_t* block_table, const int32_t* seq_lens, double scale,
                            double k_scale, double* out, double* lse, int B, int H, int D, int R,
                            int num_blocks, int P, int max_blocks, int num_splits) {
    token_view tv = mla_view(kv, kv_dtype, block_table, k_scale, D, R, num_blocks, P, max_blocks);
    return run_heads(&tv, q, seq_lens, scale, B, H, H, D, out, lse, FORM_SPLIT, num_splits);
}

/* Sparse MLA decode.  q: bf16 bits [B, H, D]; indices: [B, topk] token
 * positions; out: [B, H, R]; lse: [B, H].  softmax(s) V over the selected
 * tokens, written out directly (lse = m + log sum exp(s - m)). */
int oracle_mla_decode_sparse(const uint16_t* q, const void* kv, int kv_dtype, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* indices, int topk, double scale,
                             double k_scale, double* out, double* lse, int B, int H, int D, int R,
                             int num_blocks, int P, int max_blocks) {
    token_view tv = mla_view(kv, kv_dtype, block_table, k_scale, D, R, num_blocks, P, max_blocks);
    int failed = 0;
    int64_t pairs = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / H);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* s = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
        int64_t* base = (int64_t*)malloc(sizeof(int64_t) * (size_t)(topk > 0 ? topk : 1));
        for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[bh * D + d]);
        double* o = out + bh * R;
        for (int r = 0; r < R; ++r) o[r] = 0.0;
        int n = 0;
        double m = -INFINITY;
        for (int e = 0; e < topk; ++e) {
            int pos = indices[(int64_t)b * topk + e];
            if (pos < 0 || pos >= seq_lens[b]) continue;
            if (pos / P >= max_blocks) { failed = 1; continue; }
            int64_t bs = token_base(&tv, b, pos);
            if (bs < 0) { failed = 1; continue; }
            base[n] = bs;
            s[n] = logit(&tv, qd, bs, scale);
            if (s[n] > m) m = s[n];
            ++n;
        }
        if (n == 0) {
            lse[bh] = -INFINITY;
        } else {
            double sum = 0.0;
            for (int t = 0; t < n; ++t) sum += exp(s[t] - m);
            double L = m + log(sum);
            for (int t = 0; t < n; ++t) {
                double w = exp(s[t] - L);
                for (int r = 0; r < R; ++r) o[r] += w * (tv.v_mult * elem(&tv, base[t] + tv.v_offset + r));
            }
            lse[bh] = L;
        }
        free(qd);
        free(s);
        free(base);
    }
    return failed ? -1 : 0;
}

/* Multi-token MLA decode.  q: bf16 bits [B, q_len, H, D]; out: [B, q_len, H, R];
 * lse: [B, q_len, H].  Query i of request b attends the first
 * seq_lens[b] - q_len + i + 1 tokens (the direct definition over them). */
int oracle_mla_decode_multi(const uint16_t* q, const void* kv, int kv_dtype, const int32_t* block_table,
                            const int32_t* seq_lens, double scale, double k_scale, double* out,
                            double* lse, int B, int q_len, int H, int D, int R, int num_blocks, int P,
                            int max_blocks) {
    if (q_len < 1) return -1;
    token_view tv = mla_view(kv, kv_dtype, block_table, k_scale, D, R, num_blocks, P, max_blocks);
    int failed = 0;
    int64_t rows = (int64_t)B * q_len * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t row = 0; row < rows; ++row) {
        int b = (int)(row / ((int64_t)q_len * H));
        int i = (int)((row / H) % q_len);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[row * D + d]);
        int n = seq_lens[b] - q_len + i + 1; /* keys at positions <= context_length + i */
        if (n > seq_lens[b]) n = seq_lens[b];
        if (n < 0) n = 0;
        failed |= attend_direct(&tv, b, n, qd, scale, out + row * R, lse + row) != 0;
        free(qd);
    }
    return failed ? -1 : 0;
}

/* q: bf16 bits [B, Hq, D]; kv: [num_blocks, 2, P, Hkv, D] (plane 0 = K,
 * plane 1 = V); out: [B, Hq, D]; lse: [B, Hq]. */
int oracle_gqa_paged_decode(const uint16_t* q, const void* kv, int kv_dtype,
                            const int32_t* block_table, const int32_t* seq_lens, double scale,
                            double k_scale, double v_scale, double* out, double* lse, int B,
                            int Hq, int Hkv, int D, int num_blocks, int P, int max_blocks) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    token_view tv;
    tv.kv = kv;
    tv.kv_dtype = kv_dtype;
    tv.block_table = block_table;
    tv.max_blocks = max_blocks;
    tv.page = P;
    tv.num_blocks = num_blocks;
    tv.slot_stride = (int64_t)Hkv * D;
    tv.block_stride = 2LL * P * Hkv * D;
    tv.k_offset = 0;
    tv.v_offset = (int64_t)P * Hkv * D; /* plane 1 */
    tv.dk = D;
    tv.dv = D;
    tv.k_mult = kv_dtype == ORACLE_KV_FP8_E4M3 ? k_scale : 1.0;
    tv.v_mult = kv_dtype == ORACLE_KV_FP8_E4M3 ? v_scale : 1.0;
    return run_heads(&tv, q, seq_lens, scale, B, Hq, Hq / Hkv, D, out, lse, FORM_DIRECT, 0);
}

/* ---- per-token-head quantised GQA --------------------------------------- */

enum { ORACLE_PTH_E4M3 = 0, ORACLE_PTH_INT8 = 1, ORACLE_PTH_INT4 = 2 };

/* Bytes of codes in one row of D elements: one per element, or two 4-bit
 * codes per byte for int4. */
static int pth_code_bytes(int D, int kind) { return kind == ORACLE_PTH_INT4 ? D / 2 : D; }

/* Two's-complement nibble: 0..7 -> 0..7, 8..15 -> -8..-1. */
static double int4_code_value(unsigned nib) { return nib < 8 ? (double)nib : (double)nib - 16.0; }

/* Two's-complement byte, without relying on the signedness of char. */
static double int8_code_value(uint8_t c) { return c < 128 ? (double)c : (double)c - 256.0; }

/* The inline scale of a row: the 4 bytes after its D codes, little-endian
 * binary32. */
static double pth_row_scale(const uint8_t* row, int D) {
    uint32_t u = (uint32_t)row[D] | ((uint32_t)row[D + 1] << 8) | ((uint32_t)row[D + 2] << 16) |
                 ((uint32_t)row[D + 3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Dequantised row: out[d] = scale * value(code of element d); int4 rows hold
 * element 2i in the low nibble and element 2i + 1 in the high nibble of byte
 * i; the scale follows the code bytes. */
static void pth_row_values(const uint8_t* row, int D, int kind, double* out) {
    double sc = pth_row_scale(row, pth_code_bytes(D, kind));
    for (int d = 0; d < D; ++d) {
        double v;
        if (kind == ORACLE_PTH_INT4)
            v = int4_code_value((d & 1) ? (unsigned)(row[d / 2] >> 4) : (unsigned)(row[d / 2] & 15u));
        else if (kind == ORACLE_PTH_INT8)
            v = int8_code_value(row[d]);
        else
            v = oracle_e4m3_value(row[d]);
        out[d] = sc * v;
    }
}

/* Values of packed int4 rows: n bytes -> 2n elements (low nibble first). */
void oracle_int4_values(const uint8_t* bytes, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        out[2 * i] = int4_code_value(bytes[i] & 15u);
        out[2 * i + 1] = int4_code_value(bytes[i] >> 4);
    }
}

void oracle_int8_values(const uint8_t* codes, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = int8_code_value(codes[i]);
}

/* q: bf16 bits [B, Hq, D]; kv: bytes [num_blocks, 2, P, Hkv, C + 4] (plane 0 =
 * K, plane 1 = V, each row C code bytes + its scale, C = D, or D / 2 for
 * int4); out: [B, Hq, D]; lse:
 * [B, Hq].  The direct definition: K_t, V_t dequantised row by row,
 * s_t = scale * <q, K_t>, lse = m + log sum exp(s_t - m),
 * out = sum_t exp(s_t - lse) V_t. */
int oracle_gqa_paged_decode_pth(const uint16_t* q, const uint8_t* kv, int kind,
                                const int32_t* block_table, const int32_t* seq_lens, double scale,
                                double* out, double* lse, int B, int Hq, int Hkv, int D,
                                int num_blocks, int P, int max_blocks) {
    if (Hkv <= 0 || Hq % Hkv != 0 ||
        (kind != ORACLE_PTH_E4M3 && kind != ORACLE_PTH_INT8 && kind != ORACLE_PTH_INT4) ||
        (kind == ORACLE_PTH_INT4 && D % 2 != 0))
        return -1;
    const int group = Hq / Hkv;
    const int64_t Dp = (int64_t)pth_code_bytes(D, kind) + 4;
    int failed = 0;
    int64_t pairs = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq), g = h / group;
        int n = seq_lens[b];
        double* o = out + bh * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n <= 0) {
            lse[bh] = -INFINITY;
            continue;
        }
        if (((int64_t)n + P - 1) / P > max_blocks) {
            failed = 1;
            continue;
        }
        int bad = 0;
        for (int64_t t = 0; t < n; t += P) {
            int32_t blk = block_table[(int64_t)b * max_blocks + t / P];
            if (blk < 0 || blk >= num_blocks) bad = 1;
        }
        if (bad) {
            failed = 1;
            continue;
        }
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* kd = (double*)malloc(sizeof(double) * (size_t)D);
        double* s = (double*)malloc(sizeof(double) * (size_t)n);
        for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_value(q[bh * D + d]);
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            int64_t blk = block_table[(int64_t)b * max_blocks + t / P];
            const uint8_t* krow = kv + (((blk * 2 + 0) * P + t % P) * Hkv + g) * Dp;
            pth_row_values(krow, D, kind, kd);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * kd[d];
            s[t] = scale * acc;
            if (s[t] > m) m = s[t];
        }
        double sum = 0.0;
        for (int t = 0; t < n; ++t) sum += exp(s[t] - m);
        double L = m + log(sum);
        for (int t = 0; t < n; ++t) {
            int64_t blk = block_table[(int64_t)b * max_blocks + t / P];
            const uint8_t* vrow = kv + (((blk * 2 + 1) * P + t % P) * Hkv + g) * Dp;
            pth_row_values(vrow, D, kind, kd);
            double w = exp(s[t] - L);
            for (int d = 0; d < D; ++d) o[d] += w * kd[d];
        }
        lse[bh] = L;
        free(qd);
        free(kd);
        free(s);
    }
    return failed ? -1 : 0;
}

/* ---- merge of shard results ---------------------------------------------- */

/* outs: [G, B, H, R] normalised shard outputs; lses: [G, B, H] natural-log
 * LSEs (-inf for a shard with no token); out: [B, H, R]; lse: [B, H].  A shard
 * whose lse is -inf has weight 0 and its output is not read. */
void oracle_lse_merge(const double* outs, const double* lses, double* out, double* lse, int G, int B,
                      int H, int R) {
    int64_t rows = (int64_t)B * H;
    for (int64_t row = 0; row < rows; ++row) {
        double m = -INFINITY;
        for (int g = 0; g < G; ++g)
            if (lses[(int64_t)g * rows + row] > m) m = lses[(int64_t)g * rows + row];
        double* o = out + row * R;
        for (int r = 0; r < R; ++r) o[r] = 0.0;
        if (m == -INFINITY) {
            lse[row] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int g = 0; g < G; ++g) {
            double lg = lses[(int64_t)g * rows + row];
            if (lg == -INFINITY) continue;
            double w = exp(lg - m);
            wsum += w;
            const double* og = outs + ((int64_t)g * rows + row) * R;
            for (int r = 0; r < R; ++r) o[r] += w * og[r];
        }
        for (int r = 0; r < R; ++r) o[r] /= wsum;
        lse[row] = m + log(wsum);
    }
}

/* Shard g's share of the merged output: lses [G, B, H] natural-log shard
 * LSEs (-inf for a shard with no token), out_g [B, H, R] shard g's normalised
 * output; share [B, H, R] = e^{lse_g - lse} out_g (0 when lse_g = -inf, and
 * out_g is then not read) with lse = ln sum_g' e^{lse_g'} (-inf when every
 * shard is empty), written to lse [B, H]. */
void oracle_lse_share(const double* out_g, const double* lses, int g, double* share, double* lse, int G, int B,
                      int H, int R) {
    int64_t rows = (int64_t)B * H;
    for (int64_t row = 0; row < rows; ++row) {
        double m = -INFINITY;
        for (int k = 0; k < G; ++k)
            if (lses[(int64_t)k * rows + row] > m) m = lses[(int64_t)k * rows + row];
        double total = -INFINITY;
        if (m != -INFINITY) {
            double wsum = 0.0;
            for (int k = 0; k < G; ++k)
                if (lses[(int64_t)k * rows + row] != -INFINITY) wsum += exp(lses[(int64_t)k * rows + row] - m);
            total = m + log(wsum);
        }
        lse[row] = total;
        double lg = lses[(int64_t)g * rows + row];
        double w = lg == -INFINITY ? 0.0 : exp(lg - total);
        for (int r = 0; r < R; ++r) share[row * R + r] = w == 0.0 ? 0.0 : w * out_g[row * R + r];
    }
}
