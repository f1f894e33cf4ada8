// mla_decode_noalloc: MLA decode whose scratch lives in a fixed device array
// owned by this library, for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plugin running inside a host
// program whose memory pool owns every device byte (allocating behind the
// pool's back breaks its accounting or fails outright), a plain C caller with
// no caching allocator whose hot loop cannot afford the device-wide
// synchronisation that cudaMalloc/cudaFree may trigger, or code with a fixed,
// pre-planned memory budget.  Such callers still pass q, the cache, the block
// table, the lengths and the outputs; the split partials go to the array
// below instead of a caller workspace.
//
// The array is file-scope device memory of kNoallocScratchBytes bytes: every
// GPU that loads this library holds it until the process exits.  Host code may
// not use the array's name as an address (on the host it is only a stand-in
// symbol), so every call looks the device address up with
// cudaGetSymbolAddress for the current device.  The lookup is a host-side
// query that allocates nothing; it is made on every call rather than cached,
// so a call after a device reset (a new primary context, a new array) never
// uses the old address.  The first call on a device also loads the library's
// device code there; make that first call before any stream capture begins.
// Every call shares the array and it keeps the previous call's contents; the
// kernels write every partial slot before reading it, so nothing needs to
// start at zero.  Calls whose kernels may overlap on the GPU (different
// streams, or several host threads) race on the array: serialise them.
#include "common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = MQA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device.
mqa_status scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MQA_ERR_CUDA;
    *out = p;
    return MQA_OK;
}

}  // namespace

extern "C" mqa_status mla_decode_noalloc(const void* q, const void* kv_cache,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         float scale, float k_scale, void* out, float* lse,
                                         int batch, int num_heads, int head_size, int kv_lora_rank,
                                         int num_blocks, int page_size, int max_blocks,
                                         mqa_kv_dtype kv_dtype, int num_kv_splits,
                                         int* device_status, void* stream) {
    const size_t need = mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank, num_kv_splits);
    if (need > kNoallocScratchBytes) return MQA_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    const mqa_status st = scratch_address(&scratch);
    if (st != MQA_OK) return st;
    return mla_decode(q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, batch, num_heads,
                      head_size, kv_lora_rank, num_blocks, page_size, max_blocks, kv_dtype,
                      num_kv_splits, scratch, kNoallocScratchBytes, device_status, stream);
}
