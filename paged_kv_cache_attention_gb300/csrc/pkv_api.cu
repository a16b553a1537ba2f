// pkv_api.cu -- the C ABI of libpkv: host-side validation, workspace sizing,
// TMA tensor-map encoding and kernel dispatch.  Nothing here touches device
// memory from the host or synchronises a stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kDefaultPartition = 512;
constexpr int kMaxPartition = 16384;
constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 3-D view of a pool or of q: {D elements, heads, rows}, bf16, 128-byte
// swizzled boxes of {64, box_heads, box_rows}.
pkv_status encode_rows_map(CUtensorMap *map, const void *base, int D, int heads, int64_t rows,
                           int box_heads, int box_rows) {
    auto enc = encoder();
    if (!enc) return PKV_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * heads};
    cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// TMA view of one paged pool whose box is one (page, kv head) half-row tile
// of bs rows x 64 dims.  NHD: {D, Hkv, num_blocks * bs}, box {64, 1, bs} at
// (x, head, page * bs).  HND: {D, bs, num_blocks * Hkv}, box {64, bs, 1} at
// (x, 0, page * Hkv + head).  Both land as bs rows of 128 bytes.
pkv_status encode_pool_map(CUtensorMap *map, const void *base, const pkv_cache_desc &c) {
    if (c.layout == PKV_NHD)
        return encode_rows_map(map, base, c.head_dim, c.num_kv_heads,
                               c.num_blocks * c.block_size, 1, c.block_size);
    auto enc = encoder();
    if (!enc) return PKV_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.block_size,
                          (cuuint64_t)(c.num_blocks * c.num_kv_heads)};
    cuuint64_t strides[2] = {(cuuint64_t)c.head_dim * 2,
                             (cuuint64_t)c.head_dim * 2 * c.block_size};
    cuuint32_t box[3] = {64, (cuuint32_t)c.block_size, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status check_cache(const pkv_cache_desc &c) {
    if (c.num_blocks <= 0 || c.block_size <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (c.dtype != PKV_F32 && c.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (c.layout != PKV_NHD && c.layout != PKV_HND) return PKV_ERR_UNSUPPORTED;
    switch (c.head_dim) {  // the head sizes the attention kernels take
        case 64: case 80: case 96: case 112: case 128: case 256: break;
        default: return PKV_ERR_UNSUPPORTED;
    }
    if (c.block_size != 16 && c.block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (c.num_blocks * (int64_t)c.block_size >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    if (c.num_blocks * (int64_t)c.num_kv_heads >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

int decode_num_parts(int max_seqlen, int P, int window_left) {
    int n = (max_seqlen + P - 1) / P;
    if (window_left >= 0) {
        const long long w = ((long long)window_left + 1 + P - 1) / P + 1;
        if (w < n) n = (int)w;
    }
    return n < 1 ? 1 : n;
}

struct DecodeLayout {
    size_t lse_off, o_off, total;
};

DecodeLayout decode_layout(int batch, int Hq, int D, int num_parts) {
    DecodeLayout L;
    const size_t units = (size_t)batch * Hq * num_parts;
    L.lse_off = 0;
    L.o_off = round_up(units * sizeof(float), 256);
    L.total = L.o_off + round_up(units * D * sizeof(float), 256);
    return L;
}

// Work list of the prefill kernel: a 256-byte header (item count), one int4
// per (query block, kv head), the per-request block offsets and the
// per-request first item.  A query
// block holds 2 tiles of 128 / G tokens.
struct PrefillLayout {
    int64_t max_items;
    size_t total;
};

PrefillLayout prefill_layout(int batch, int G, int num_kv_heads, int total_q) {
    PrefillLayout L;
    const int64_t tokens = G > 0 && G <= 128 ? 2 * (128 / G) : 1;
    L.max_items = ((int64_t)total_q / tokens + batch) * num_kv_heads;
    L.total = round_up(256 + (size_t)L.max_items * 16 + ((size_t)2 * batch + 1) * 4, 256);
    return L;
}

pkv_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return PKV_OK;
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    return PKV_ERR_CUDA;
}

}  // namespace

int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < kMaxDevices) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 148;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes) {
    struct Entry {
        const void *kernel;
        int device;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &x : done)
        if (x.kernel == kernel && x.device == dev && x.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back({kernel, dev, bytes});
    return e;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_OUT_OF_RANGE: return "PKV_ERR_OUT_OF_RANGE";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
        default: return "PKV_ERR_UNKNOWN";
    }
}

int pkv_version(void) { return 501; }

pkv_status pkv_get_device_error(const int32_t *dev_error, int32_t *bits, int clear,
                                void *stream) {
    if (!dev_error) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, dev_error, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (bits) *bits = word;
    if (clear && cudaMemsetAsync(const_cast<int32_t *>(dev_error), 0, sizeof word, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (word & (int32_t)PKV_DEVERR_TIMEOUT) return PKV_ERR_TIMEOUT;
    const int32_t metadata =
        (int32_t)(PKV_DEVERR_BLOCK_ID | PKV_DEVERR_SLOT | PKV_DEVERR_SEQLEN | PKV_DEVERR_POSITION);
    return (word & metadata) ? PKV_ERR_OUT_OF_RANGE : PKV_OK;
}

pkv_status pkv_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                 void *v_cache, const int64_t *slot_mapping, int64_t num_tokens,
                                 pkv_cache_desc cache, int32_t *dev_error, void *stream) {
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0 ||
        cache.head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache.dtype != PKV_F32 && cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache.layout != PKV_NHD && cache.layout != PKV_HND) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    const int64_t head_bytes = (int64_t)cache.head_dim * elem_bytes(cache.dtype);
    const int64_t row_bytes = (int64_t)cache.num_kv_heads * head_bytes;
    if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (cache.layout == PKV_HND && head_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    const int64_t capacity = cache.num_blocks * (int64_t)cache.block_size;
    return from_cuda(launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping,
                                              num_tokens, row_bytes, capacity, cache.block_size,
                                              head_bytes, cache.layout == PKV_HND, dev_error,
                                              static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_rope_cos_sin_table(float *cos_sin, int max_position, int rotary_dim,
                                  double base, double position_scale, double ntk_alpha,
                                  void *stream) {
    if (max_position < 0 || rotary_dim <= 0 || rotary_dim % 2 != 0) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(base) || base <= 0.0 || !std::isfinite(position_scale) ||
        position_scale <= 0.0 || !std::isfinite(ntk_alpha) || ntk_alpha <= 0.0)
        return PKV_ERR_INVALID_ARG;
    if (ntk_alpha != 1.0) {
        // NTK-aware scaling: raise the base so that the lowest frequency,
        // base^(-(rd - 2) / rd), is divided by ntk_alpha
        if (rotary_dim <= 2) return PKV_ERR_INVALID_ARG;
        base *= std::pow(ntk_alpha, (double)rotary_dim / (rotary_dim - 2));
        if (!std::isfinite(base) || base <= 0.0) return PKV_ERR_INVALID_ARG;
    }
    if (max_position == 0) return PKV_OK;
    if (!cos_sin || !aligned(cos_sin, 16)) return PKV_ERR_INVALID_ARG;
    return from_cuda(launch_rope_table(cos_sin, max_position, rotary_dim, base, position_scale,
                                       static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_rope_reshape_and_cache(void *query, void *key, const void *value, void *k_cache,
                                      void *v_cache, const int64_t *positions,
                                      const int64_t *slot_mapping, int64_t num_tokens,
                                      int num_qo_heads, pkv_cache_desc cache,
                                      const float *cos_sin, int max_position, int rotary_dim,
                                      int is_neox_style, int32_t *dev_error, void *stream) {
    if (num_tokens < 0 || num_qo_heads < 0 || max_position <= 0) return PKV_ERR_INVALID_ARG;
    if (cache.num_blocks <= 0 || cache.block_size <= 0 || cache.num_kv_heads <= 0 ||
        cache.head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache.dtype != PKV_F32 && cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache.layout != PKV_NHD && cache.layout != PKV_HND) return PKV_ERR_UNSUPPORTED;
    const int V = 16 / elem_bytes(cache.dtype);
    if (rotary_dim <= 0 || rotary_dim > cache.head_dim || rotary_dim % 2 != 0)
        return PKV_ERR_INVALID_ARG;
    if (rotary_dim % (2 * V) != 0 || cache.head_dim % V != 0) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_qo_heads * cache.head_dim > (1 << 24) ||
        (int64_t)cache.num_kv_heads * cache.head_dim > (1 << 24))
        return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !positions || !slot_mapping || !cos_sin ||
        (num_qo_heads > 0 && !query))
        return PKV_ERR_INVALID_ARG;
    if ((query && !aligned(query, 16)) || !aligned(key, 16) || !aligned(value, 16) ||
        !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(cos_sin, 16) ||
        !aligned(positions, 8) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    RopeParams p;
    p.query = query;
    p.key = key;
    p.value = value;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.positions = positions;
    p.slot_mapping = slot_mapping;
    p.cos_sin = reinterpret_cast<const float2 *>(cos_sin);
    p.dev_error = dev_error;
    p.num_tokens = num_tokens;
    p.capacity = cache.num_blocks * (int64_t)cache.block_size;
    p.max_position = max_position;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = cache.num_kv_heads;
    p.head_dim = cache.head_dim;
    p.rotary_dim = rotary_dim;
    p.block_size = cache.block_size;
    p.hnd = cache.layout == PKV_HND ? 1 : 0;
    return from_cuda(launch_rope_reshape_cache(p, cache.dtype, is_neox_style != 0,
                                               static_cast<cudaStream_t>(stream)));
}

size_t pkv_paged_decode_workspace_size(int batch, int num_qo_heads, int head_dim,
                                       int max_seqlen, int partition_size, int window_left) {
    if (batch <= 0 || num_qo_heads <= 0 || head_dim <= 0 || max_seqlen < 0) return 256;
    const int P = partition_size > 0 ? partition_size : kDefaultPartition;
    const int np = decode_num_parts(max_seqlen, P, window_left);
    return decode_layout(batch, num_qo_heads, head_dim, np).total;
}

pkv_status pkv_paged_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                            pkv_cache_desc cache, const int32_t *block_table,
                            int max_blocks_per_seq, const int32_t *cache_seqlens,
                            int max_seqlen, const float *sink, const float *alibi_slopes,
                            int batch, int num_qo_heads, int window_left, float sm_scale,
                            int partition_size, float *lse_out, void *workspace,
                            size_t workspace_bytes, int32_t *dev_error, void *stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (batch < 0 || batch > 65535 || num_qo_heads <= 0 || max_seqlen < 0 ||
        max_blocks_per_seq <= 0 || window_left < -1 || !std::isfinite(sm_scale))
        return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = num_qo_heads / cache.num_kv_heads;
    if (G > 16) return PKV_ERR_UNSUPPORTED;
    if (cache.dtype == PKV_F32 && cache.head_dim > 128) return PKV_ERR_UNSUPPORTED;
    const int P = partition_size > 0 ? partition_size : kDefaultPartition;
    if (partition_size < 0 || P % cache.block_size != 0 || P > kMaxPartition)
        return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !cache_seqlens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_table, 4) || !aligned(cache_seqlens, 4))
        return PKV_ERR_INVALID_ARG;
    const int np = decode_num_parts(max_seqlen, P, window_left);
    if (np > 65535) return PKV_ERR_UNSUPPORTED;  // grid.y limit
    const DecodeLayout lay = decode_layout(batch, num_qo_heads, cache.head_dim, np);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.total)
        return PKV_ERR_WORKSPACE;

    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.out = out;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table;
    p.seqlens = cache_seqlens;
    p.sink = sink;
    p.alibi = alibi_slopes;
    p.lse_out = lse_out;
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.lse_off);
    p.part_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.o_off);
    p.dev_error = dev_error;
    p.num_blocks = cache.num_blocks;
    p.batch = batch;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = cache.num_kv_heads;
    p.group = G;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_seqlen = max_seqlen;
    p.window_left = window_left;
    p.head_dim = cache.head_dim;
    p.hnd = cache.layout == PKV_HND ? 1 : 0;
    p.partition_size = P;
    p.num_parts = np;
    p.scale_log2 = sm_scale * 1.4426950408889634f;

    alignas(64) CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    if (cache.dtype == PKV_BF16) {
        if ((st = encode_pool_map(&tk, k_cache, cache)) != PKV_OK) return st;
        if ((st = encode_pool_map(&tv, v_cache, cache)) != PKV_OK) return st;
    }
    return from_cuda(launch_decode(p, cache, &tk, &tv, static_cast<cudaStream_t>(stream)));
}

size_t pkv_varlen_prefill_workspace_size(int batch, int num_qo_heads, int num_kv_heads,
                                         int total_q, int max_seqlen_q) {
    (void)max_seqlen_q;
    if (batch <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || total_q < 0 ||
        num_qo_heads % num_kv_heads != 0)
        return 256;
    const int G = num_qo_heads / num_kv_heads;
    return prefill_layout(batch, G, num_kv_heads, total_q).total;
}

}  // extern "C"

namespace {

// Shared by the paged and the contiguous prefill entry points.  kv_rows: the
// rows of the K/V views the tensor maps cover; kv_box_rows: rows per box (the
// page size, or 128 for contiguous rows).
// The bitmaps of the MInference sparse form (nullptr: dense attention).
struct SparseMask {
    const uint32_t *vbits, *sbits;
    const int32_t *vcnt, *scnt;
    int words;
};

pkv_status prefill_run(void *out, const void *q, const void *k, const void *v,
                       const pkv_cache_desc &cache, bool contiguous, int64_t kv_rows,
                       const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *cu_seq_lens_q, const int32_t *cu_seq_lens_k,
                       int max_seqlen_q, int max_seqlen_k, int total_q, const float *sink,
                       const float *alibi_slopes, int batch, int num_qo_heads, int causal,
                       int window_left, float sm_scale,
                       float *lse_out, void *workspace, size_t workspace_bytes,
                       int32_t *dev_error, void *stream, const SparseMask *sparse = nullptr,
                       int max_ctas = 0) {
    if (cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache.head_dim % 16 != 0 || (cache.head_dim > 128 && cache.head_dim != 256))
        return PKV_ERR_UNSUPPORTED;
    if (batch < 0 || num_qo_heads <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        total_q < 0 || max_blocks_per_seq <= 0 || window_left < -1 || !std::isfinite(sm_scale) ||
        max_ctas < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = num_qo_heads / cache.num_kv_heads;
    if (G > 16 || (G & (G - 1)) != 0) return PKV_ERR_UNSUPPORTED;
    if (batch == 0 || total_q == 0) return PKV_OK;
    if (!out || !q || (kv_rows > 0 && (!k || !v)) || (!contiguous && !block_table) ||
        !cu_seq_lens_q || !cu_seq_lens_k)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) ||
        (kv_rows > 0 && (!aligned(k, 16) || !aligned(v, 16))))
        return PKV_ERR_INVALID_ARG;
    if (kv_rows >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    const PrefillLayout lay = prefill_layout(batch, G, cache.num_kv_heads, total_q);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.total)
        return PKV_ERR_WORKSPACE;
    if (lay.max_items > (int64_t)1 << 30) return PKV_ERR_UNSUPPORTED;

    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.out = out;
    p.block_table = block_table;
    p.cu_q = cu_seq_lens_q;
    p.cu_k = cu_seq_lens_k;
    p.sink = sink;
    p.alibi = alibi_slopes;
    p.lse_out = lse_out;
    p.tiles = static_cast<int32_t *>(workspace);
    p.dev_error = dev_error;
    p.num_blocks = cache.num_blocks;
    p.batch = batch;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = cache.num_kv_heads;
    p.group = G;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.total_q = total_q;
    p.window_left = window_left;
    p.head_dim = cache.head_dim;
    p.hnd = (!contiguous && cache.layout == PKV_HND) ? 1 : 0;
    if (sparse) {
        p.vbits = sparse->vbits;
        p.sbits = sparse->sbits;
        p.vcnt = sparse->vcnt;
        p.scnt = sparse->scnt;
        p.bit_words = sparse->words;
    }
    p.causal = causal ? 1 : 0;
    p.total_k = contiguous ? (int)kv_rows : 0;
    p.rows_per_head = 128 / G;
    p.max_tiles = (int)lay.max_items;
    p.max_ctas = max_ctas;
    p.scale_log2 = sm_scale * 1.4426950408889634f;

    // With no contiguous keys at all every request clips to kv_len 0 and no
    // K/V tile is ever loaded; the K/V maps then cover one row of q only so
    // that they can be encoded.
    if (contiguous && kv_rows == 0) {
        k = v = q;
        kv_rows = 1;
    }
    alignas(64) CUtensorMap tq, tk, tv;
    const int box_rows = contiguous ? 128 : cache.block_size;
    pkv_status st;
    if ((st = encode_rows_map(&tq, q, cache.head_dim, num_qo_heads, total_q, G, 128 / G)) !=
        PKV_OK)
        return st;
    if (contiguous) {
        if ((st = encode_rows_map(&tk, k, cache.head_dim, cache.num_kv_heads, kv_rows, 1,
                                  box_rows)) != PKV_OK)
            return st;
        if ((st = encode_rows_map(&tv, v, cache.head_dim, cache.num_kv_heads, kv_rows, 1,
                                  box_rows)) != PKV_OK)
            return st;
    } else {
        if ((st = encode_pool_map(&tk, k, cache)) != PKV_OK) return st;
        if ((st = encode_pool_map(&tv, v, cache)) != PKV_OK) return st;
    }
    return from_cuda(launch_prefill(p, cache, contiguous, &tq, &tk, &tv,
                                    static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

pkv_status pkv_varlen_prefill(void *out, const void *q, const void *k_cache,
                              const void *v_cache, pkv_cache_desc cache,
                              const int32_t *block_table, int max_blocks_per_seq,
                              const int32_t *cu_seq_lens_q, const int32_t *cu_seq_lens_k,
                              int max_seqlen_q, int max_seqlen_k, int total_q,
                              const float *sink, const float *alibi_slopes, int batch,
                              int num_qo_heads, int causal, int window_left, float sm_scale,
                              float *lse_out, void *workspace, size_t workspace_bytes,
                              int max_ctas, int32_t *dev_error, void *stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    return prefill_run(out, q, k_cache, v_cache, cache, false,
                       cache.num_blocks * cache.block_size, block_table, max_blocks_per_seq,
                       cu_seq_lens_q, cu_seq_lens_k, max_seqlen_q, max_seqlen_k, total_q, sink,
                       alibi_slopes, batch, num_qo_heads, causal, window_left, sm_scale,
                       lse_out, workspace, workspace_bytes, dev_error, stream, nullptr,
                       max_ctas);
}

pkv_status pkv_varlen_prefill_contiguous(void *out, const void *q, const void *k, const void *v,
                                         int total_k, int num_kv_heads, int head_dim, int dtype,
                                         const int32_t *cu_seq_lens_q,
                                         const int32_t *cu_seq_lens_k, int max_seqlen_q,
                                         int max_seqlen_k, int total_q, const float *sink,
                                         const float *alibi_slopes, int batch,
                                         int num_qo_heads, int causal, int window_left,
                                         float sm_scale, float *lse_out, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_error,
                                         void *stream) {
    if (total_k < 0 || num_kv_heads <= 0 || head_dim <= 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    pkv_cache_desc cache;
    cache.num_blocks = 1;
    cache.block_size = 128;
    cache.num_kv_heads = num_kv_heads;
    cache.head_dim = head_dim;
    cache.dtype = dtype;
    cache.layout = PKV_NHD;
    return prefill_run(out, q, k, v, cache, true, total_k,
                       nullptr, max_seqlen_k / 64 + 2, cu_seq_lens_q, cu_seq_lens_k,
                       max_seqlen_q, max_seqlen_k, total_q, sink, alibi_slopes, batch,
                       num_qo_heads, causal, window_left, sm_scale, lse_out, workspace,
                       workspace_bytes, dev_error, stream);
}


pkv_status pkv_minference_sizes(int seq_len, int vertical_size, int slash_size,
                                double adaptive_budget, int num_sink_tokens,
                                int num_recent_diags, int *nv, int *ns) {
    if (seq_len <= 0 || num_sink_tokens < 0 || num_recent_diags < 0 || !nv || !ns)
        return PKV_ERR_INVALID_ARG;
    if (adaptive_budget > 0.0) {
        const int budget = (int)(seq_len * adaptive_budget);
        vertical_size = std::max(num_sink_tokens + 1, (int)(budget * 0.2));
        slash_size = std::max(num_recent_diags + 1, (int)(budget * 0.8));
    }
    if (vertical_size <= 0 || slash_size <= 0) return PKV_ERR_INVALID_ARG;
    *nv = std::min(vertical_size, seq_len);
    *ns = std::min(slash_size, seq_len);
    return PKV_OK;
}

}  // extern "C"

namespace {

struct MinferenceLayout {
    size_t stat, lse, vscore, sscore, spart, vidx, sidx, vbits, sbits, vcnt, scnt, cu, tiles,
        total;
};

MinferenceLayout minference_layout(int S, int Hq, int Hkv, int nv, int ns) {
    MinferenceLayout L;
    const size_t nblk = (size_t)(S + 127) / 128, W = (size_t)(S + 31) / 32;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    L.stat = take((size_t)Hq * nblk * 64 * 4 * 2);
    L.lse = take((size_t)Hq * 64 * 4);
    L.vscore = take((size_t)Hq * S * 4);
    L.sscore = take((size_t)Hq * S * 4);
    L.spart = take((size_t)Hq * nblk * 192 * 4);
    L.vidx = take((size_t)Hq * nv * 4);
    L.sidx = take((size_t)Hq * ns * 4);
    L.vbits = take((size_t)Hq * W * 4);
    L.sbits = take((size_t)Hq * W * 4);
    L.vcnt = take((size_t)Hq * (W + 1) * 4);
    L.scnt = take((size_t)Hq * (W + 1) * 4);
    L.cu = take(16);
    const int G = Hkv > 0 ? Hq / Hkv : 1;
    L.tiles = take(prefill_layout(1, G, Hkv, S).total);
    L.total = o;
    return L;
}

}  // namespace

extern "C" {

size_t pkv_minference_workspace_size(int seq_len, int num_qo_heads, int num_kv_heads,
                                     int vertical_size, int slash_size, double adaptive_budget,
                                     int num_sink_tokens, int num_recent_diags) {
    int nv = 0, ns = 0;
    if (num_qo_heads <= 0 || num_kv_heads <= 0 ||
        pkv_minference_sizes(seq_len, vertical_size, slash_size, adaptive_budget,
                             num_sink_tokens, num_recent_diags, &nv, &ns) != PKV_OK)
        return 256;
    return minference_layout(seq_len, num_qo_heads, num_kv_heads, nv, ns).total;
}

pkv_status pkv_minference_prefill(void *out, const void *q, const void *k, const void *v,
                                  int seq_len, int num_qo_heads, int num_kv_heads, int head_dim,
                                  int dtype, int vertical_size, int slash_size,
                                  double adaptive_budget, int num_sink_tokens,
                                  int num_recent_diags, float sm_scale,
                                  int32_t *vertical_indices, int32_t *slash_indices,
                                  void *workspace, size_t workspace_bytes, int32_t *dev_error,
                                  void *stream) {
    int nv = 0, ns = 0;
    pkv_status st = pkv_minference_sizes(seq_len, vertical_size, slash_size, adaptive_budget,
                                         num_sink_tokens, num_recent_diags, &nv, &ns);
    if (st != PKV_OK) return st;
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 ||
        !std::isfinite(sm_scale))
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim % 16 != 0 || head_dim < 64 || head_dim > 128) return PKV_ERR_UNSUPPORTED;
    if (seq_len > kMaxSparseKeys) return PKV_ERR_UNSUPPORTED;
    if (!out || !q || !k || !v) return PKV_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
        (vertical_indices && !aligned(vertical_indices, 4)) ||
        (slash_indices && !aligned(slash_indices, 4)))
        return PKV_ERR_INVALID_ARG;
    const MinferenceLayout L =
        minference_layout(seq_len, num_qo_heads, num_kv_heads, nv, ns);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total)
        return PKV_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    MinferenceParams m;
    std::memset(&m, 0, sizeof m);
    m.q = q;
    m.k = k;
    m.seq_len = seq_len;
    m.last_q = std::min(64, seq_len);
    m.num_qo_heads = num_qo_heads;
    m.num_kv_heads = num_kv_heads;
    m.head_dim = head_dim;
    m.num_blocks = (seq_len + 127) / 128;
    m.scale = sm_scale;
    const size_t nblk = (size_t)m.num_blocks;
    m.stat_m = reinterpret_cast<float *>(ws + L.stat);
    m.stat_l = m.stat_m + (size_t)num_qo_heads * nblk * 64;
    m.lse = reinterpret_cast<float *>(ws + L.lse);
    m.vscore = reinterpret_cast<float *>(ws + L.vscore);
    m.sscore = reinterpret_cast<float *>(ws + L.sscore);
    m.spart = reinterpret_cast<float *>(ws + L.spart);
    m.nv = nv;
    m.ns = ns;
    m.num_sink = num_sink_tokens;
    m.num_recent = num_recent_diags;
    m.vidx = vertical_indices ? vertical_indices : reinterpret_cast<int32_t *>(ws + L.vidx);
    m.sidx = slash_indices ? slash_indices : reinterpret_cast<int32_t *>(ws + L.sidx);
    m.words = (seq_len + 31) / 32;
    m.vbits = reinterpret_cast<uint32_t *>(ws + L.vbits);
    m.sbits = reinterpret_cast<uint32_t *>(ws + L.sbits);
    m.vcnt = reinterpret_cast<int32_t *>(ws + L.vcnt);
    m.scnt = reinterpret_cast<int32_t *>(ws + L.scnt);
    m.cu = reinterpret_cast<int32_t *>(ws + L.cu);
    cudaError_t e = launch_minference_pattern(m, dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    pkv_cache_desc cache;
    cache.num_blocks = 1;
    cache.block_size = 128;
    cache.num_kv_heads = num_kv_heads;
    cache.head_dim = head_dim;
    cache.dtype = dtype;
    cache.layout = PKV_NHD;
    const SparseMask mask{m.vbits, m.sbits, m.vcnt, m.scnt, m.words};
    return prefill_run(out, q, k, v, cache, true, seq_len, nullptr, seq_len / 64 + 2, m.cu,
                       m.cu, seq_len, seq_len, seq_len, nullptr, nullptr, 1, num_qo_heads, 1, -1,
                       sm_scale, nullptr, ws + L.tiles, L.total - L.tiles, dev_error, stream,
                       &mask);
}

}  // extern "C"
