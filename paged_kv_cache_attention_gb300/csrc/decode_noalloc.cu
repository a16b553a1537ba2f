// decode_noalloc.cu -- paged_decode for callers that cannot allocate device
// memory (a plug-in whose host framework owns all device memory, a serving
// loop that must not allocate once running).  The split-KV scratch is a
// fixed device array owned by the library instead of a caller workspace.
#include <mutex>

#include "pkv_internal.h"

namespace {

// The scratch every call of pkv_paged_decode_noalloc uses.  Each GPU that
// loads the library holds it until the process exits.  In host code this name
// is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_DECODE_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current.
pkv_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr)
            return PKV_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache, pkv_cache_desc cache,
    const int32_t *block_table, int max_blocks_per_seq, const int32_t *cache_seqlens,
    int max_seqlen, const float *sink, int batch, int num_qo_heads, int window_left,
    float sm_scale, int partition_size, float *lse_out, int32_t *dev_error, void *stream) {
    if (batch == 0) return PKV_OK;  // nothing to do: no device lookup either
    const size_t need = pkv_paged_decode_workspace_size(batch, num_qo_heads, cache.head_dim,
                                                        max_seqlen, partition_size, window_left);
    if (need > PKV_NOALLOC_DECODE_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    const pkv_status st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    return pkv_paged_decode(out, q, k_cache, v_cache, cache, block_table, max_blocks_per_seq,
                            cache_seqlens, max_seqlen, sink, /*alibi_slopes=*/nullptr, batch,
                            num_qo_heads, window_left,
                            sm_scale, partition_size, lse_out, scratch,
                            PKV_NOALLOC_DECODE_SCRATCH_BYTES, dev_error, stream);
}
