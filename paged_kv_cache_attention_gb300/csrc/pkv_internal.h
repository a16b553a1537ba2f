// pkv_internal.h -- parameter blocks and launcher entry points shared by the
// C-ABI layer (pkv_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Split-KV decode: one CTA per (partition, kv head, sequence).
struct DecodeParams {
    const void *q;               // [B, Hq, D]
    void *out;                   // [B, Hq, D]
    const void *k_cache;         // pools (used by the kernels that do not use TMA)
    const void *v_cache;
    const int32_t *block_table;  // [B, max_blocks_per_seq]
    const int32_t *seqlens;      // [B]
    const float *sink;           // [Hq] or nullptr
    const float *alibi;          // [Hq] ALiBi slopes or nullptr
    float *lse_out;              // [B, Hq] or nullptr
    float *part_lse;             // [B, Hq, num_parts] (log2 units)
    float *part_o;               // [B, Hq, num_parts, D], normalised partial outputs
    int32_t *dev_error;
    int64_t num_blocks;
    int batch, num_qo_heads, num_kv_heads, group;
    int max_blocks_per_seq, max_seqlen;
    int window_left;
    int head_dim;                // D of q, out and the pools; the kernels pad it to 64/128/256
    int hnd;                     // pools in the HND layout (else NHD)
    int partition_size;
    int num_parts;               // grid.x: partitions per sequence the grid covers
    float scale_log2;            // sm_scale * log2(e)
};

// Varlen prefill on the paged pools, or on contiguous K/V ([total_k, Hkv, D]
// addressed by cu_k).
struct PrefillParams {
    const void *q;                 // [total_q, Hq, D]
    void *out;                     // [total_q, Hq, D]
    const int32_t *block_table;    // [B, max_blocks_per_seq]
    const int32_t *cu_q;           // [B+1]
    const int32_t *cu_k;           // [B+1]
    const float *sink;             // [Hq] or nullptr
    const float *alibi;            // [Hq] ALiBi slopes or nullptr
    float *lse_out;                // [total_q, Hq] or nullptr
    int32_t *tiles;                // work list, built on the device
    int32_t *dev_error;
    int64_t num_blocks;
    int batch, num_qo_heads, num_kv_heads, group;
    int max_blocks_per_seq, max_seqlen_q, max_seqlen_k, total_q;
    int window_left;
    int causal;                    // 1: keys j <= query position; 0: no upper bound
    int head_dim;                  // D <= 128 (tiles padded to 128 with zeros), or 256
    int hnd;                       // paged pools in the HND layout (else NHD)
    int total_k;                   // contiguous K/V: rows in the arrays (unused when paged)
    // MInference sparse form (contiguous K/V only): [Hq][bit_words] bitmaps of
    // the kept key columns and diagonals, and their per-word prefix counts
    // ([Hq][bit_words + 1]); vbits == nullptr for dense attention
    const uint32_t *vbits, *sbits;
    const int32_t *vcnt, *scnt;
    int bit_words;
    int rows_per_head;             // query tokens per 128-row tile (128 / group)
    int max_tiles;                 // capacity of the work list
    int max_ctas;                  // attention CTAs of the launch (0: one per SM)
    float scale_log2;
};

// hnd: pools in the HND layout; the copy then scatters each token's row by kv
// head (head_bytes each) to page rows of block_size.
cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int64_t row_bytes, int64_t capacity,
                                     int block_size, int64_t head_bytes, bool hnd,
                                     int32_t *dev_error, cudaStream_t stream);

// Returns cudaErrorNotSupported when no kernel matches the shape.
cudaError_t launch_decode(const DecodeParams &p, const pkv_cache_desc &cache,
                          const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                          cudaStream_t stream);

// MInference: the longest sequence the sparse prefill takes (its per-CTA
// list of 128-key tiles has 16-bit entries in 2 KB of shared memory).
constexpr int kMaxSparseKeys = 131072;

// MInference vertical + slash pattern of one sequence (minference.cu).
struct MinferenceParams {
    const void *q, *k;             // [S, Hq, D], [S, Hkv, D]
    int seq_len, last_q, num_qo_heads, num_kv_heads, head_dim;
    int num_blocks;                // ceil(S / 128) score blocks
    float scale;                   // logit = scale * <q, k>
    // workspace
    float *stat_m, *stat_l;        // [Hq][num_blocks][64] per-block row max, sum exp
    float *lse;                    // [Hq][64]
    float *vscore, *sscore;        // [Hq][S]
    float *spart;                  // [Hq][num_blocks][192] diagonal partials
    // selection
    int nv, ns, num_sink, num_recent;
    int32_t *vidx, *sidx;          // [Hq][nv], [Hq][ns], ascending
    // bitmaps for the attention
    int words;                     // ceil(S / 32)
    uint32_t *vbits, *sbits;       // [Hq][words]
    int32_t *vcnt, *scnt;          // [Hq][words + 1]
    int32_t *cu;                   // [2]: cu_seq_lens {0, S} of the one sequence
};

cudaError_t launch_minference_pattern(const MinferenceParams &p, int dtype, cudaStream_t stream);

// Rotary embedding fused with the cache write.
struct RopeParams {
    void *query;                   // [T, Hq, D], rotated in place (may be null if Hq == 0)
    void *key;                     // [T, Hkv, D], rotated in place
    const void *value;             // [T, Hkv, D]
    void *k_cache, *v_cache;       // NHD pools
    const int64_t *positions;      // [T]
    const int64_t *slot_mapping;   // [T]
    const float2 *cos_sin;         // [max_position][rotary_dim / 2] (cos, sin)
    int32_t *dev_error;
    int64_t num_tokens;
    int64_t capacity;              // num_blocks * block_size
    int64_t max_position;
    int num_qo_heads, num_kv_heads, head_dim, rotary_dim;
    int block_size;
    int hnd;                       // pools in the HND layout (else NHD)
};

cudaError_t launch_rope_table(float *table, int max_position, int rotary_dim, double base,
                              double position_scale, cudaStream_t stream);
cudaError_t launch_rope_reshape_cache(const RopeParams &p, int dtype, bool neox,
                                      cudaStream_t stream);

// head_dim 256: the attention kernel of prefill_wide.cu (64-key tiles; the
// contiguous tensor maps use 64-row boxes).
cudaError_t launch_prefill_wide(const PrefillParams &p, const pkv_cache_desc &cache,
                                bool contiguous, const CUtensorMap *tmap_q,
                                const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                cudaStream_t stream);

// contiguous: K/V are [total_k, Hkv, D] rows addressed by cu_k (the tensor
// maps use 128-row boxes, 64 for head_dim 256); otherwise paged pools of
// cache.block_size rows.
cudaError_t launch_prefill(const PrefillParams &p, const pkv_cache_desc &cache, bool contiguous,
                           const CUtensorMap *tmap_q, const CUtensorMap *tmap_k,
                           const CUtensorMap *tmap_v, cudaStream_t stream);

// Launch `kernel` with the programmatic-stream-serialization attribute: it may
// begin while the previous kernel on the stream finishes and must call
// pdl_wait() before reading that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `kernel` on the
// current device, done once per (kernel, device, size) and remembered.
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);

}  // namespace pkv
