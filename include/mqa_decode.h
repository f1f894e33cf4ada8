/*
 * mqa_decode.h — C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * One query token per request attends to that request's paged KV cache.  Two
 * cache formats are served:
 *
 *   MLA (primary).  The cache row of a token is one latent vector
 *   [kv_c (kv_lora_rank) | k_pe (64 rope dims)], head_size 576 or 320.  That
 *   row is the key of EVERY query head, and its first kv_lora_rank columns are
 *   the value ("Triton と MLA" page, vllm-arch-zh ja/attention/triton-mla:
 *   sections 設計動機 and データフロー, where forward_mqa hands the cache to the
 *   decode kernel as a single-head K cache and its first kv_lora_rank columns
 *   as V).
 *
 *   GQA (secondary).  Standard paged attention over a
 *   [num_blocks, 2, page, num_kv_heads, head_size] cache ("AttentionBackend"
 *   page, vllm-arch-zh fr/attention/backend: section "Motivation de
 *   conception", the FlashAttention layout).
 *
 * For request b and query head h the library returns
 *   s_t      = scale * <q[b,h,:], K_t>                  for t < seq_lens[b]
 *   lse[b,h] = ln sum_t exp(s_t)                        (natural log, fp32)
 *   out[b,h] = sum_t exp(s_t - lse[b,h]) * V_t          (bf16)
 * where token t lives in physical block block_table[b][t / page] at slot
 * t % page (attention-kernel tutorial page, lshu.cn/news/265860, §11), there is
 * no mask inside [0, seq_lens[b]) (same page, §9), and a sequence of length 0
 * yields out = 0, lse = -inf.
 *
 * The work on one sequence may be cut into KV segments that run on separate
 * thread blocks; their partial results are merged by LogSumExp
 * (m = max_s m_s, l = sum_s e^{m_s-m} l_s, O = sum_s e^{m_s-m} O_s / l; same
 * page, §12).  num_kv_splits bounds how many segment partials per request the
 * caller's workspace holds, exactly as the workspace shape
 * [B, H, num_kv_splits, kv_lora_rank + 1] fp32 of the Triton MLA backend does
 * ("Triton と MLA" page, データフロー).  num_kv_splits == 1 processes every
 * request in one thread block in a fixed order: the result is bitwise
 * reproducible and independent of the other requests in the batch
 * (batch-invariant mode, same section).
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers to caller-owned, contiguous,
 *     row-major memory on the current CUDA device, 16-byte aligned.
 *   - The library allocates nothing, never synchronises the stream and keeps
 *     no per-call state: a call only enqueues kernels on `stream`
 *     (a cudaStream_t; NULL = legacy default stream).
 *   - Argument errors are returned before anything is enqueued.  A launch
 *     failure returns MQA_ERR_CUDA.  Conditions found on the device (a block
 *     id outside [0, num_blocks), seq_len < 0 or > max_blocks * page, a wait
 *     that exceeded its time limit) are written into *device_status (an int in
 *     device memory that the caller zeroes; the kernels only raise it to the
 *     matching mqa_status code) and the offending page is treated as empty.
 */
#ifndef MQA_DECODE_H
#define MQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MQA_ABI_VERSION 1

typedef enum mqa_status {
    MQA_OK = 0,
    MQA_ERR_INVALID_ARG = 1,         /* null/unaligned pointer, bad size or count */
    MQA_ERR_UNSUPPORTED = 2,         /* shape or dtype the library does not serve */
    MQA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the *_workspace_bytes value */
    MQA_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
    MQA_ERR_DEVICE_CHECK = 5,        /* device-side: bad block id or sequence length */
    MQA_ERR_DEVICE_TIMEOUT = 6       /* device-side: a bounded wait expired */
} mqa_status;

typedef enum mqa_kv_dtype {
    MQA_KV_BF16 = 0,     /* bfloat16 cache; k_scale / v_scale are ignored */
    MQA_KV_FP8_E4M3 = 1, /* OCP e4m3fn cache; element value = scale * e4m3(code) */
    /* Per-token-head quantised GQA caches (gqa_paged_decode only): each
     * (token, KV head) row of the K and V planes carries its own scale
     * inline, after its codes; see gqa_paged_decode. */
    MQA_KV_FP8_E4M3_PER_TOKEN_HEAD = 2,
    MQA_KV_INT8_PER_TOKEN_HEAD = 3,
    MQA_KV_INT4_PER_TOKEN_HEAD = 4
} mqa_kv_dtype;

/* ABI version of the loaded library (MQA_ABI_VERSION at build time). */
int mqa_abi_version(void);

/* Static, NUL-terminated description of a status code. */
const char* mqa_status_string(int status);

/* Number of streaming multiprocessors of the current device, or -1. */
int mqa_device_sm_count(void);

/* The cudaError_t code (and its text) of the last CUDA runtime call that made
 * an entry point of this library return MQA_ERR_CUDA on the calling thread;
 * 0 / "no error" if none did.  Diagnostic only. */
int mqa_last_cuda_error(void);
const char* mqa_last_cuda_error_string(void);

/* Split-count heuristic of the Triton MLA backend ("Triton と MLA" page,
 * 主要ファイル: _compute_num_kv_splits, and データフロー: the
 * VLLM_BATCH_INVARIANT branch): ceil(max_seq_len / 512), at least 1, at most
 * 2 * sm_count; 1 when batch_invariant is non-zero.  Host-only, pure. */
int mqa_num_kv_splits(int max_seq_len, int sm_count, int batch_invariant);

/* Workspace bytes mla_decode needs: batch * num_heads * num_kv_splits *
 * (kv_lora_rank + 1) * 4, i.e. the fp32 [B, H, S, R + 1] partial buffer of the
 * Triton MLA backend ("Triton と MLA" page, データフロー).  0 when
 * num_kv_splits == 1 (no partials are kept).  0 on invalid arguments. */
size_t mla_decode_workspace_bytes(int batch, int num_heads, int kv_lora_rank, int num_kv_splits);

/* Workspace bytes gqa_paged_decode needs: batch * num_q_heads * num_kv_splits *
 * (head_size + 1) * 4; 0 when num_kv_splits == 1. */
size_t gqa_paged_decode_workspace_bytes(int batch, int num_q_heads, int head_size,
                                        int num_kv_splits);

/* MLA decode (the MQA view of MLA: forward_mqa, "Triton と MLA" page,
 * データフロー).
 *
 *   q            bf16 [batch, num_heads, head_size]: the absorbed query
 *                (q_nope absorbed ‖ q_pe) already concatenated.
 *   kv_cache     [num_blocks, page_size, head_size], bf16 or e4m3 codes
 *                (kv_dtype).  Row layout [kv_c (kv_lora_rank) | k_pe].
 *   block_table  int32 [batch, max_blocks]: physical block of each logical
 *                block.  Only entries below ceil(seq_lens[b] / page_size) are
 *                read.
 *   seq_lens     int32 [batch]: KV length of each request.
 *   scale        softmax scale applied to q.K.
 *   k_scale      fp8 dequantisation scale (used for K and V); ignored for bf16.
 *   out          bf16 [batch, num_heads, kv_lora_rank], fully written.
 *   lse          fp32 [batch, num_heads] natural-log LSE of the scaled logits,
 *                or NULL.  (fp32 rather than the query dtype: a bf16 lse cannot
 *                carry the 1e-3 accuracy the merge across shards needs.)
 *   With kv_dtype = MQA_KV_FP8_E4M3 and more than 32 query rows (num_heads
 *   here, q_len * num_heads in mla_decode_multi) the tensor cores take the
 *   query in f16 (the e4m3 codes widen to f16 exactly): every q entry must
 *   lie within +-65504 (an entry beyond makes that row's out and lse
 *   undefined, typically NaN; the other rows are unaffected), and entries
 *   below 2^-14 in magnitude keep an absolute precision of 2^-24 only.  With a
 *   bf16 cache, or 32 rows or fewer, the query is used in bf16 as given.
 *   Valid tokens of an e4m3 cache hold finite codes (0x7F / 0xFF are NaN).
 *   head_size / kv_lora_rank must be 576/512 or 320/256 ("Triton と MLA" page,
 *   境界と失敗: head sizes 320 and 576 only).  page_size must be a multiple of
 *   16 ("AttentionBackend" page, "Limites et échecs": MultipleOf(16)).
 *   num_heads in [1, 128]; batch >= 1; max_blocks >= 1; num_blocks >= 1.
 *   num_kv_splits >= 1: the per-request partial budget (see the file header);
 *   workspace / workspace_bytes: caller scratch of at least
 *   mla_decode_workspace_bytes(...) bytes (may be NULL when that is 0).
 *   device_status: device int or NULL (see the file header).
 */
mqa_status mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                      int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                      int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                      void* workspace, size_t workspace_bytes, int* device_status, void* stream);

/* mla_decode with the split of the Triton MLA backend taken literally: each
 * request is cut into num_kv_splits page ranges of ceil(pages /
 * num_kv_splits) pages and one work unit (thread block, or 2-CTA cluster
 * with more than 32 heads) decodes each (request, range), whereas mla_decode
 * treats num_kv_splits as a partial budget and cuts the batch's pages into
 * units of equal size ("Triton と MLA" page, 主要ファイル / データフロー:
 * one program per request and split; tutorial page lshu.cn/news/265860,
 * §12).  A request's reduction order depends only on its own length and
 * num_kv_splits, so the result is bitwise reproducible and independent of
 * the rest of the batch at ANY num_kv_splits (mla_decode: only at 1).  Slower
 * when the lengths are uneven.  Arguments, workspace, results and errors as
 * for mla_decode; batch * num_kv_splits <= 2^24 (else MQA_ERR_UNSUPPORTED). */
mqa_status mla_decode_fixed_splits(const void* q, const void* kv_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                   int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                   int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                                   void* workspace, size_t workspace_bytes, int* device_status, void* stream);

/* Multi-token MLA decode: q_len new positions of each request verified in
 * one call (speculative decoding).  The tutorial page (lshu.cn/news/265860)
 * §10 gives the structure: query i of q_len sits at absolute position
 * context_length + i and sees the keys at positions <= its own, i.e. the
 * whole history plus a q_len x q_len lower triangle over the new tokens.
 *
 *   q        bf16 [batch, q_len, num_heads, head_size] (contiguous).
 *   seq_lens int32 [batch]: kv_length, the history plus the q_len new tokens,
 *            whose cache rows are already written; query i attends the first
 *            seq_lens[b] - q_len + i + 1 tokens (none when that is <= 0:
 *            out = 0, lse = -inf).
 *   out      bf16 [batch, q_len, num_heads, kv_lora_rank], fully written.
 *   lse      fp32 [batch, q_len, num_heads] or NULL.
 *   q_len >= 1 and q_len * num_heads <= 128 (else MQA_ERR_UNSUPPORTED);
 *   workspace: mla_decode_workspace_bytes(batch, q_len * num_heads,
 *   kv_lora_rank, num_kv_splits) bytes.  The rows q_len * num_heads share the
 *   cache exactly as query heads do; q_len = 1 is mla_decode.  Other
 *   arguments, results and errors are those of mla_decode. */
mqa_status mla_decode_multi(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                            int batch, int q_len, int num_heads, int head_size, int kv_lora_rank,
                            int num_blocks, int page_size, int max_blocks, mqa_kv_dtype kv_dtype,
                            int num_kv_splits, void* workspace, size_t workspace_bytes, int* device_status,
                            void* stream);

/* Sparse (top-k) MLA decode.  The tutorial page (lshu.cn/news/265860) §13
 * describes it: an indexer picks, per request, topk key positions (2048 in
 * its example, at head size 576), and the query attends those positions
 * only, each found in the paged cache through the block table, so one query
 * row's logits are [1, 576] x [576, topk] instead of a walk over the whole
 * context.
 *
 *   indices  int32 [batch, topk] (row-major, 4-byte aligned): logical token
 *            positions of request b.  An entry selects position p when
 *            0 <= p < seq_lens[b]; anything else (the usual -1 padding, or a
 *            position at or past the end) selects nothing.  The order of
 *            entries does not matter; a position listed twice counts twice.
 *            A request that selects nothing gets out = 0, lse = -inf.
 *   topk     entries per request, 1 .. 2^24.
 *   seq_lens int32 [batch]: cached tokens per request (bounds the valid
 *            positions; the work done is topk entries per request whatever
 *            the length).
 *   num_heads 1 .. 128 (query heads of the request, all sharing the cache).
 *   workspace: mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank,
 *   num_kv_splits) bytes; splits divide the topk entries (mqa_num_kv_splits
 *   with max_seq_len = topk is a good choice).
 *   A selected position whose page has no valid block id (outside
 *   [0, num_blocks)), or that lies at or past max_blocks * page_size while
 *   below seq_lens[b], is skipped and MQA_ERR_DEVICE_CHECK is written to
 *   *device_status.  Other arguments, results and errors are those of
 *   mla_decode (q, out, lse, dtypes, scale, k_scale, head sizes). */
mqa_status mla_decode_sparse(const void* q, const void* kv_cache, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* indices, float scale, float k_scale,
                             void* out, float* lse, int batch, int num_heads, int head_size,
                             int kv_lora_rank, int num_blocks, int page_size, int max_blocks, int topk,
                             mqa_kv_dtype kv_dtype, int num_kv_splits, void* workspace,
                             size_t workspace_bytes, int* device_status, void* stream);

/* Merge of sequence-shard results, the local step of decode context
 * parallelism (DCP): a request's KV pages are spread over num_shards ranks,
 * each rank decodes its shard (mla_decode / gqa_paged_decode on its pages,
 * returning the shard's normalised output and natural-log lse), the caller
 * gathers the shards' results (that exchange is the caller's), and this call
 * merges them by LogSumExp: with m = max_g lse_g and w_g = e^{lse_g - m},
 *   out = sum_g w_g out_g / sum_g w_g,   lse = m + ln sum_g w_g
 * (tutorial page lshu.cn/news/265860, §12; the "Triton と MLA" page,
 * 設計動機: lse is returned so that DCP shards can be merged,
 * cp_lse_ag_out_rs).  A shard with lse_g = -inf (no token) has weight 0 and
 * its output is not read; when every shard is empty, out = 0, lse = -inf.
 *
 *   shard_out  bf16 [num_shards, rows, head_dim], rows = batch * num_heads.
 *   shard_lse  fp32 [num_shards, rows].
 *   out        bf16 [rows, head_dim], fully written.
 *   lse        fp32 [rows] or NULL.
 *   num_shards >= 1, rows >= 1, head_dim a multiple of 8 in [8, 4096];
 *   every pointer 16-byte aligned.  Fixed shard order: reproducible.
 *   Allocates nothing; enqueues one kernel on `stream`. */
mqa_status mqa_lse_merge(const void* shard_out, const float* shard_lse, void* out, float* lse, int num_shards,
                         long long rows, int head_dim, void* stream);

/* ---- Decode context parallelism: page placement and the exchange ---------
 *
 * The pages say that DCP shards of a sequence are merged by LogSumExp, which
 * is why the decode returns a natural-log lse, and they name the merge
 * cp_lse_ag_out_rs ("Triton と MLA" page, 設計動機; "AttentionBackend" page,
 * Motivation de conception, on the lse base).  Where the pages stop, the
 * library reads it as follows: every rank holds whole pages of a request
 * (page-aligned shards, so each shard is an ordinary paged sequence that
 * mla_decode / gqa_paged_decode take as is), the lse of every shard is
 * all-gathered, and each rank scales its own shard output by its weight so
 * that a sum reduce-scatter over the ranks yields the merged output, split by
 * heads.  The alternative, all-gathering the outputs and calling
 * mqa_lse_merge, is served as well.  Positions play no part in a q_len = 1
 * decode, so a shard's decode is exact; the placement does not serve
 * multi-token or index-sparse decode.  The collectives are the caller's. */

typedef enum mqa_dcp_layout {
    /* page j of a request lives on rank j % num_ranks: a page never moves as
     * its sequence grows (the placement a serving system keeps) */
    MQA_DCP_ROUND_ROBIN = 0,
    /* rank g holds pages [g L, min((g + 1) L, n_pages)) with
     * L = ceil(n_pages / num_ranks): contiguous runs, for a fixed sequence */
    MQA_DCP_CONTIGUOUS = 1
} mqa_dcp_layout;

/* Columns of a rank's block table under either layout:
 * ceil(max_blocks / num_ranks), or -1 if max_blocks < 1 or num_ranks < 1. */
int mqa_dcp_shard_max_blocks(int max_blocks, int num_ranks);

/* The pages rank `rank` of `num_ranks` holds, as a block table and lengths
 * that the decode entry points take directly.  HOST pointers (the one
 * exception to the device-pointer convention): no GPU is touched and nothing
 * is enqueued.
 *
 *   block_table       int32 [batch, max_blocks]: the whole sequences' pages.
 *   seq_lens          int32 [batch], 0 <= seq_lens[b] <= max_blocks * page_size.
 *   shard_block_table int32 [batch, shard_max_blocks] out: the rank's pages of
 *                     request b in sequence order, then -1.
 *   shard_seq_lens    int32 [batch] out: tokens in those pages (every page
 *                     full except the sequence's last one, which is always
 *                     the last page of the rank that holds it).
 *   shard_max_blocks  >= mqa_dcp_shard_max_blocks(max_blocks, num_ranks).
 * Over the ranks the shards cover each sequence's tokens exactly once.
 * Errors: MQA_ERR_INVALID_ARG for a null pointer, a bad size, rank outside
 * [0, num_ranks), an unknown layout or a sequence length out of range
 * (nothing is written then). */
mqa_status mqa_dcp_shard(const int32_t* block_table, const int32_t* seq_lens, int batch, int max_blocks,
                         int page_size, int num_ranks, int rank, mqa_dcp_layout layout,
                         int32_t* shard_block_table, int shard_max_blocks, int32_t* shard_seq_lens);

/* Where token `pos` of a sequence of seq_len tokens lives: the rank and its
 * position in that rank's shard (the slot a cache writer fills).  Host only;
 * pos in [0, seq_len), else MQA_ERR_INVALID_ARG. */
mqa_status mqa_dcp_locate(int pos, int seq_len, int page_size, int num_ranks, mqa_dcp_layout layout, int* rank,
                          int* shard_pos);

/* The local step of the all-gather-lse / reduce-scatter-output merge: with
 * every rank's shard lse gathered, rank `rank` scales its normalised shard
 * output by its weight in the merge,
 *   lse = m + ln sum_g e^{lse_g - m},  m = max_g lse_g,
 *   scaled = e^{lse_rank - lse} * shard_out     (0 where lse_rank = -inf),
 * so that the sum over the ranks of `scaled` is the merged output of
 * mqa_lse_merge.  `scaled` is written in the order a sum reduce-scatter over
 * the ranks wants (NCCL's reduce-scatter splits its input into num_ranks
 * consecutive chunks): chunk c holds heads [c H / num_ranks, (c + 1) H /
 * num_ranks) of every request, so after it rank c holds its heads' merged
 * output.
 *
 *   shard_out     bf16 [batch, num_heads, head_dim]: this rank's shard result.
 *   gathered_lse  fp32 [num_ranks, batch, num_heads]: every rank's shard lse.
 *   scaled        [num_ranks, batch, num_heads / num_ranks, head_dim], fp32
 *                 if scaled_fp32, else bf16 (half the exchange bytes, one
 *                 more rounding per term).
 *   lse           fp32 [batch, num_heads] or NULL: the merged lse (-inf where
 *                 no rank holds a token; scaled is 0 there).
 *   num_heads a multiple of num_ranks; head_dim a multiple of 8 in [8, 4096];
 *   0 <= rank < num_ranks; device pointers, 16-byte aligned.  Allocates
 *   nothing; enqueues one kernel on `stream`. */
mqa_status mqa_dcp_scale_shard(const void* shard_out, const float* gathered_lse, void* scaled, float* lse,
                               int num_ranks, int rank, int batch, int num_heads, int head_dim, int scaled_fp32,
                               void* stream);

/* Size of the library-owned scratch array used by mla_decode_noalloc. */
#define MQA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* mla_decode without a caller workspace (the pages have no counterpart to this
 * entry point; it exists for callers of this library that cannot allocate
 * device memory).
 *
 * Who needs it: a plugin running inside a host program whose memory pool owns
 * all device memory, a plain C caller without a caching allocator whose hot
 * loop cannot pay for the device-wide synchronisation cudaMalloc/cudaFree may
 * cause, or code with a fixed memory plan.  Such callers still pass q, the
 * cache, the block table, the lengths, out and lse exactly as for mla_decode;
 * only the split partials move into a fixed device array of
 * MQA_NOALLOC_SCRATCH_BYTES (64 MiB) that this library declares at file scope.
 * Every GPU that loads the library holds that array until the process exits.
 *
 *   - Calls needing more than the array returns MQA_ERR_WORKSPACE_TOO_SMALL
 *     before anything is enqueued: the requirement is
 *     mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank, num_kv_splits)
 *     <= MQA_NOALLOC_SCRATCH_BYTES (lower num_kv_splits to fit; e.g. B=64,
 *     H=16, R=512 fits up to 31 splits, B=4, H=128 up to 63).
 *   - Every call looks up the array's device address for the current device
 *     (cudaGetSymbolAddress, a host-side query; so a device reset never
 *     leaves a stale address behind).  The first call on a device also loads
 *     the library's device code there: make that first call before any
 *     stream capture.  The function allocates nothing and never calls
 *     cudaMalloc or cudaFree.
 *   - All calls share the one array, which keeps the previous call's contents
 *     (nothing in it needs to start at zero).  Calls whose kernels may overlap
 *     on the GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller.
 *   Other arguments, results and errors are those of mla_decode. */
mqa_status mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                              const int32_t* seq_lens, float scale, float k_scale, void* out,
                              float* lse, int batch, int num_heads, int head_size,
                              int kv_lora_rank, int num_blocks, int page_size, int max_blocks,
                              mqa_kv_dtype kv_dtype, int num_kv_splits, int* device_status,
                              void* stream);

/* GQA paged decode (TritonAttentionImpl.forward's paged_attention path,
 * "Triton と MLA" page, 主要ファイル; cache layout from the "AttentionBackend"
 * page, "Motivation de conception").
 *
 *   q            bf16 [batch, num_q_heads, head_size]
 *   kv_cache     [num_blocks, 2, page_size, num_kv_heads, row]; plane 0
 *                holds K, plane 1 holds V.  By kv_dtype:
 *                  MQA_KV_BF16      row = head_size bf16 values;
 *                  MQA_KV_FP8_E4M3  row = head_size e4m3 codes, K value =
 *                                   k_scale * code, V value = v_scale * code;
 *                  MQA_KV_FP8_E4M3_PER_TOKEN_HEAD / MQA_KV_INT8_PER_TOKEN_HEAD
 *                                   row = head_size + 4 bytes: head_size e4m3
 *                                   or int8 (two's complement) codes, then
 *                                   the row's scale as a little-endian IEEE
 *                                   binary32; value = that scale * code
 *                                   (k_scale / v_scale are ignored).
 *                  MQA_KV_INT4_PER_TOKEN_HEAD
 *                                   row = head_size / 2 + 4 bytes: 4-bit two's
 *                                   complement codes, two per byte (element
 *                                   2i in the low nibble of byte i), then the
 *                                   scale as above.
 *                                   These are the Triton backend's
 *                                   fp8 / int8 / int4_per_token_head caches
 *                                   ("Triton と MLA" page, 設計動機 and
 *                                   主要ファイル: the head dimension is padded
 *                                   to hold the inline scale; the packing,
 *                                   the 4-byte padding and the scale's
 *                                   position are this library's reading).
 *   k_scale, v_scale  finite; used by MQA_KV_FP8_E4M3 only.
 *   With an 8-bit (or 4-bit) cache the tensor cores take the query as f16
 *   (the codes widen to f16 exactly): q entries must lie within +-65504.
 *   Per-token-head scales must be zero or normal fp32 numbers (magnitude at
 *   least 2^-126).
 *   out          bf16 [batch, num_q_heads, head_size]; lse fp32 [batch,
 *                num_q_heads] or NULL.
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   head_size in {64, 128}; num_kv_heads in [1, 8]; num_q_heads a multiple of
 *   num_kv_heads with at most 16 query heads per KV head; page_size a multiple
 *   of 16.  Tokens past seq_lens[b] in a request's last page are never used,
 *   whatever their bytes (NaN codes or scales included).  Other arguments as
 *   for mla_decode.
 */
mqa_status gqa_paged_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, float k_scale, float v_scale,
                            void* out, float* lse, int batch, int num_q_heads, int num_kv_heads,
                            int head_size, int num_blocks, int page_size, int max_blocks,
                            mqa_kv_dtype kv_dtype, int num_kv_splits, void* workspace,
                            size_t workspace_bytes, int* device_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MQA_DECODE_H */
