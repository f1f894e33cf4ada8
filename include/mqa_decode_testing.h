/*
 * mqa_decode_testing.h — test-only entry points of the GB300 paged
 * decode-attention library (not part of the product interface in
 * mqa_decode.h).  The pages have no counterpart to them.
 *
 * They exist so that the library's bounded waits can be tested on a GPU
 * without faulting or hanging it: each runs a normal decode in which one
 * role of one work unit deliberately never delivers what another role waits
 * for.  The waiting role gives up after its time limit (2 s of the GPU's
 * global timer), MQA_ERR_DEVICE_TIMEOUT is written to *device_status, every
 * thread block returns, and the context stays usable; the outputs of the
 * affected requests are undefined.
 *
 * Gate: every hook returns MQA_ERR_UNSUPPORTED, before anything is enqueued,
 * unless the environment variable MQA_ENABLE_TEST_HOOKS is "1" at the time
 * of the call, so that no product caller can start a deliberately stalled
 * kernel by accident.  Argument validation runs after the gate, exactly as
 * for the product entry point each hook mirrors.
 */
#ifndef MQA_DECODE_TESTING_H
#define MQA_DECODE_TESTING_H

#include "mqa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* A bf16-cache gqa_paged_decode in which the producer of work unit
 * `withhold_unit` fills and announces none of its tiles: its consumers' first
 * wait runs out.  Arguments as for gqa_paged_decode (k_scale = v_scale = 1);
 * withhold_unit >= 0 (with num_kv_splits == 1, unit b is request b). */
mqa_status mqa_test_gqa_withheld_arrive(const void* q, const void* kv_cache, const int32_t* block_table,
                                        const int32_t* seq_lens, float scale, void* out, float* lse, int batch,
                                        int num_q_heads, int num_kv_heads, int head_size, int num_blocks,
                                        int page_size, int max_blocks, int num_kv_splits, void* workspace,
                                        size_t workspace_bytes, int* device_status, void* stream,
                                        int withhold_unit);

/* An mla_decode in which the producer of work unit `withhold_unit` fills and
 * announces none of its tiles: with more than 32 heads the 2-CTA tensor-core
 * cluster of that unit, else every 16-head block of that unit, waits in vain.
 * Arguments as for mla_decode; withhold_unit >= 0 (with num_kv_splits == 1,
 * unit b is request b). */
mqa_status mqa_test_mla_withheld_arrive(const void* q, const void* kv_cache, const int32_t* block_table,
                                        const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                        int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                        int page_size, int max_blocks, mqa_kv_dtype kv_dtype, int num_kv_splits,
                                        void* workspace, size_t workspace_bytes, int* device_status, void* stream,
                                        int withhold_unit);

/* An e4m3-cache mla_decode with more than 32 heads (the 2-CTA tensor-core
 * kernel) in which softmax warp `warp` (2..9) of both CTAs of work unit
 * `unit` gives up before its first pair as if one of its waits had expired,
 * while the other warps of its group go on: nothing may block on the warp
 * that left (every wait for it is a bounded mbarrier wait), every wait that
 * then misses that warp's arrivals runs out, and the call reports
 * MQA_ERR_DEVICE_TIMEOUT.  Arguments as for mla_decode with
 * kv_dtype = MQA_KV_FP8_E4M3; MQA_ERR_INVALID_ARG for unit < 0, a warp
 * outside 2..9 or num_heads <= 32. */
mqa_status mqa_test_mla_warp_gives_up(const void* q, const void* kv_cache, const int32_t* block_table,
                                      const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                      int batch, int num_heads, int head_size, int kv_lora_rank, int num_blocks,
                                      int page_size, int max_blocks, int num_kv_splits, void* workspace,
                                      size_t workspace_bytes, int* device_status, void* stream, int unit,
                                      int warp);

#ifdef __cplusplus
}
#endif

#endif /* MQA_DECODE_TESTING_H */
