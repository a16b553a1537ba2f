// cache_write.cu -- the reshape_and_cache scatter.
//
// vLLM attention.py, PagedAttention.forward: after the prompt attention and
// before decode, the new tokens' keys and values are stored into the paged
// cache at the flat slots slot_mapping names.  With the NHD page layout a
// token's row (num_kv_heads * head_dim elements) is contiguous both in the
// input and in the pool, so the scatter is a row copy: 16-byte vector loads
// and stores, K and V rows interleaved over one flat index space.  With the
// HND layout the same vectors go to one page row per kv head.  The copy is
// bit-exact (integers, no arithmetic on the values).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;  // 16-byte vectors each thread moves

// Flat index space: [2 (K, V)][num_tokens][vecs_per_row].  Each thread moves
// kVecPerThread vectors spaced one grid apart, loads first, then stores.
// HND pools: vector c of a token's row belongs to kv head c / vecs_per_head
// and goes to that head's page, row slot % block_size.
template <bool HND>
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                         int64_t vecs_per_row, int64_t capacity, int block_size,
                         int64_t vecs_per_head, int32_t *dev_error) {
    pdl_trigger();  // the next call's kernel may begin launching
    pdl_wait();     // the previous kernel on the stream has finished
    const int64_t per_tensor = num_tokens * vecs_per_row;
    const int64_t total = 2 * per_tensor;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; idx < total; idx += stride * kVecPerThread) {
        uint4 v[kVecPerThread];
        int64_t dst[kVecPerThread];
        bool is_v[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t i = idx + u * stride;
            dst[u] = -1;
            if (i >= total) continue;
            is_v[u] = i >= per_tensor;
            const int64_t j = is_v[u] ? i - per_tensor : i;
            const int64_t t = j / vecs_per_row;
            const int64_t c = j - t * vecs_per_row;
            const int64_t slot = __ldg(slot_mapping + t);
            if (slot < 0) continue;  // not cached
            if (slot >= capacity) {
                flag_error(dev_error, PKV_DEVERR_SLOT);
                continue;
            }
            v[u] = is_v[u] ? __ldg(value + j) : __ldg(key + j);
            if constexpr (HND) {
                const int64_t g = c / vecs_per_head, cv = c - g * vecs_per_head;
                const int64_t blk = slot / block_size, off = slot - blk * block_size;
                const int64_t heads = vecs_per_row / vecs_per_head;
                dst[u] = ((blk * heads + g) * block_size + off) * vecs_per_head + cv;
            } else {
                dst[u] = slot * vecs_per_row + c;
            }
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            if (dst[u] < 0) continue;
            if (is_v[u])
                v_cache[dst[u]] = v[u];
            else
                k_cache[dst[u]] = v[u];
        }
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int64_t row_bytes, int64_t capacity,
                                     int block_size, int64_t head_bytes, bool hnd,
                                     int32_t *dev_error, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t vecs_per_row = row_bytes / 16;
    const int64_t total = 2 * num_tokens * vecs_per_row;
    int64_t blocks = (total + int64_t(kThreads) * kVecPerThread - 1) /
                     (int64_t(kThreads) * kVecPerThread);
    const int64_t cap = int64_t(device_sm_count()) * 32;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto kern = hnd ? reshape_and_cache_kernel<true> : reshape_and_cache_kernel<false>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream,
                      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                      slot_mapping, num_tokens, vecs_per_row, capacity, block_size,
                      head_bytes / 16, dev_error);
}

}  // namespace pkv
