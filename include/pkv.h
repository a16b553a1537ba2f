/*
 * pkv.h -- C ABI of libpkv: attention over a paged KV cache on GB300 (sm_103a).
 *
 * The operations, each an asynchronous launch sequence on the caller's
 * CUDA stream:
 *
 *   pkv_reshape_and_cache  write the new tokens' K/V rows into the paged pools
 *                          at the flat slots slot_mapping names
 *                          (vLLM attention.py, PagedAttention.forward: the
 *                          cache_ops.reshape_and_cache step);
 *   pkv_rope_reshape_and_cache  the same write preceded by the rotary
 *                          position embedding of query and key
 *                          (vLLM attention.py, PagedAttentionWithRoPE);
 *   pkv_minference_prefill vertical + slash sparse prefill of one sequence
 *                          (nano-vllm minference.py);
 *   pkv_paged_decode       one query token per sequence, attending to positions
 *                          0 .. cache_seqlens[b]-1 gathered through block_table
 *                          (transformers docs "paged_attention", decode path;
 *                          vLLM attention.py, single_query_cached_kv_attention
 *                          with 512-token split-KV partitions);
 *   pkv_varlen_prefill     varlen / chunk prefill, causal or not: request r
 *                          has q_len = cu_seq_lens_q[r+1]-cu_seq_lens_q[r]
 *                          queries over kv_len = cu_seq_lens_k[r+1]-
 *                          cu_seq_lens_k[r] keys read from the paged pools
 *                          (transformers docs "paged_attention", varlen path;
 *                          FlashInfer sink_attention_reference.py, varlen
 *                          mode);
 *   pkv_varlen_prefill_contiguous  the same attention with request r's keys in
 *                          rows cu_seq_lens_k[r] .. cu_seq_lens_k[r+1]-1 of
 *                          contiguous [total_k, num_kv_heads, head_dim] K and
 *                          V arrays (the docs' varlen path before the keys are
 *                          paged).
 *
 * What the attention computes (FlashInfer sink_attention_reference.py,
 * sink_softmax and sink_attention_unified): for request r, query row i and
 * query head h, with G = num_qo_heads / num_kv_heads and kv head g = h / G:
 *   qpos  = kv_len - q_len + i               (decode: kv_len - 1)
 *   keep key j iff j < kv_len, j <= qpos (causal only), and
 *                  (window_left < 0 or j >= qpos - window_left)
 *   s_j   = sm_scale * <q[i,h,:], k[j,g,:]>  (fp32)
 *           + alibi_slopes[h] * (j - qpos)   (only with ALiBi slopes: vLLM
 *                                     attention.py, PagedAttentionWithALiBi)
 *   o     = sum_j exp(s_j) v[j,g,:] / (sum_j exp(s_j) + exp(sink[h]))
 *   lse   = log(sum_j exp(s_j) + exp(sink[h]))           (natural log)
 * sink[h] is a logit, not scaled by sm_scale; sink == NULL means no sink.
 * A row that keeps no key gets o = 0 and lse = sink[h] (or -inf).
 *
 * Paged pool layout: k_cache and v_cache are each a contiguous
 *   [num_blocks, block_size, num_kv_heads, head_dim]   (PKV_NHD), or
 *   [num_blocks, num_kv_heads, block_size, head_dim]   (PKV_HND)
 * array.  Logical position p of sequence b lives in page
 * block_table[b * max_blocks_per_seq + p / block_size], row p % block_size;
 * its flat slot is page * block_size + p % block_size.  block_table entries
 * beyond a sequence's length may be -1 (unallocated) and are never read.
 *
 * Ownership: the caller allocates and owns every buffer; device pointers are
 * device memory, host values are plain ints/floats.  The library allocates
 * nothing and keeps no state between calls except a process-wide cache of
 * the driver's tensor-map encoder and of per-device attributes.  Scratch
 * space (split-KV partials) lives in the caller's workspace, whose size the
 * *_workspace_size functions give.  Apart from pkv_get_device_error, the
 * library never reads device memory from the host and never synchronises
 * the stream.
 *
 * Errors: arguments are validated on the host before anything is launched;
 * a non-zero pkv_status is returned and nothing runs.  Metadata that only the
 * device sees (a block id outside the pool, a slot outside the pool, a
 * sequence length larger than the declared maximum or an offset outside the
 * rows of q) is checked in the kernels: the offending page or row is skipped
 * and a PKV_DEVERR_* bit is OR-ed into *dev_error (a device int32 the caller
 * owns and zeroes; may be NULL).  No kernel traps.  pkv_get_device_error
 * reads that word back and turns it into a status (PKV_ERR_OUT_OF_RANGE).
 * The word is the caller's (not part of a workspace) so that one word can
 * collect the checks of every call of a step, cache writes included.
 *
 * What each call supports (head sizes, page sizes, dtypes, layouts, causal
 * or not, ALiBi, GQA group sizes) is listed with the call below; all calls
 * take block_size 16 or 32 and num_qo_heads % num_kv_heads == 0, and the
 * attention output has the dtype of the cache.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shape */
    PKV_ERR_UNSUPPORTED = 2, /* a shape or dtype this version has no kernel for */
    PKV_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
    PKV_ERR_CUDA = 4,        /* a CUDA call failed (launch, tensor-map encode, sync) */
    PKV_ERR_OUT_OF_RANGE = 5, /* pkv_get_device_error: the kernels found device
                                 metadata out of range (PKV_DEVERR_BLOCK_ID, _SLOT,
                                 _SEQLEN or _POSITION) and skipped it */
    PKV_ERR_TIMEOUT = 6      /* pkv_get_device_error: a bounded pipeline wait gave up
                                (PKV_DEVERR_TIMEOUT); the outputs of that call are
                                not valid */
} pkv_status;

typedef enum pkv_dtype { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Layout of each pool.  NHD: [num_blocks, block_size, num_kv_heads, head_dim]
 * (a token's row of all kv heads is contiguous).  HND: [num_blocks,
 * num_kv_heads, block_size, head_dim] (a page of one kv head is contiguous). */
typedef enum pkv_layout { PKV_NHD = 0, PKV_HND = 1 } pkv_layout;

/* Device-side error bits OR-ed into *dev_error. */
#define PKV_DEVERR_BLOCK_ID 1u /* block_table entry of an attended position outside [0, num_blocks) */
#define PKV_DEVERR_SLOT 2u     /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_SEQLEN 4u   /* a length above its declared maximum, negative, or
                                  beyond max_blocks_per_seq * block_size; a
                                  cu_seq_lens offset outside the rows of q / k */
#define PKV_DEVERR_TIMEOUT 8u  /* a bounded pipeline wait gave up */
#define PKV_DEVERR_POSITION 16u /* a rotary position outside [0, max_position) */

/* Description of the two paged pools (same shape and dtype). */
typedef struct pkv_cache_desc {
    int64_t num_blocks;   /* pages in each pool */
    int32_t block_size;   /* tokens per page: 16 or 32 */
    int32_t num_kv_heads; /* Hkv */
    int32_t head_dim;     /* D: 64, 80, 96, 112, 128 or 256 (see each call) */
    int32_t dtype;        /* pkv_dtype of the pools, q and out */
    int32_t layout;       /* pkv_layout of the pools */
} pkv_cache_desc;

/* Human-readable name of a pkv_status. */
PKV_API const char *pkv_status_string(int status);

/* Library ABI version (major * 100 + minor). */
PKV_API int pkv_version(void);

/*
 * get_device_error: the device-side check result of the calls issued so far.
 * Waits for `stream` to finish (cudaStreamSynchronize), reads the caller's
 * int32 error word dev_error (device memory; the word every call of this
 * library ORs its PKV_DEVERR_* bits into) and stores its bits in *bits
 * (host; may be NULL).  With clear != 0 the word is then reset to zero on
 * `stream`.  This is the one call of the library that synchronises and reads
 * device memory from the host.
 *
 * Returns PKV_OK when no bit is set; PKV_ERR_TIMEOUT when PKV_DEVERR_TIMEOUT
 * is set; otherwise PKV_ERR_OUT_OF_RANGE when a metadata bit is set (a block
 * id, slot, length or position outside its range: the kernels skipped the
 * offending page, row or token, so the outputs that depend on it are not the
 * attention the caller meant); PKV_ERR_INVALID_ARG for a NULL dev_error;
 * PKV_ERR_CUDA when the synchronisation or the copy fails.
 *
 * The pages put the cache write before the attention in one forward
 * (vLLM attention.py, PagedAttention.forward) and mark unallocated block
 * table entries with -1 (transformers docs "paged_attention", decode path);
 * this call is how a caller learns that such an entry, or any other device
 * metadata, was out of range.
 */
PKV_API pkv_status pkv_get_device_error(const int32_t *dev_error, int32_t *bits, int clear,
                                        void *stream);

/*
 * selftest_bounded_wait: a check of the library's bounded pipeline waits on
 * the current device.  Launches one warp on `stream` that waits on a shared-
 * memory barrier nothing arrives on; the wait gives up after its limit
 * (about 4e8 SM cycles, a fraction of a second), ORs PKV_DEVERR_TIMEOUT into
 * dev_error (device int32, caller-owned) and the kernel returns.  Afterwards
 * pkv_get_device_error reports PKV_ERR_TIMEOUT, and the context and stream
 * stay usable: this is the path every kernel of the library takes when one
 * of its pipeline waits runs out, here without a broken pipeline.
 * Returns PKV_ERR_INVALID_ARG for a NULL dev_error, PKV_ERR_CUDA if the
 * launch fails, else PKV_OK (asynchronous).
 */
PKV_API pkv_status pkv_selftest_bounded_wait(int32_t *dev_error, void *stream);

/*
 * reshape_and_cache: for every t in [0, num_tokens) with slot_mapping[t] >= 0,
 * copy row t of key and of value ([num_tokens, Hkv, D], contiguous, dtype of
 * the cache) into flat slot slot_mapping[t] of k_cache and v_cache.  The copy
 * is bit-exact.  A negative slot skips the token (stands for vLLM's to_cache
 * filter).  A slot >= num_blocks * block_size is skipped and sets
 * PKV_DEVERR_SLOT.  Two tokens with the same slot race (caller error).
 * All pointers must be 16-byte aligned.
 */
PKV_API pkv_status pkv_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                 void *v_cache, const int64_t *slot_mapping,
                                 int64_t num_tokens, pkv_cache_desc cache, int32_t *dev_error,
                                 void *stream);

/*
 * Rotary position embedding (vLLM attention.py, PagedAttentionWithRoPE:
 * rotary_dim, base, is_neox_style, rope_scaling), in two calls.
 *
 * rope_cos_sin_table: fill cos_sin ([max_position, rotary_dim / 2] pairs of
 * float32 (cos, sin), device memory owned by the caller, 16-byte aligned)
 * with the angles (pos / position_scale) * b^(-2i / rotary_dim) for
 * pos in [0, max_position) and i in [0, rotary_dim / 2), where
 * b = base * ntk_alpha^(rotary_dim / (rotary_dim - 2)).  The angles and
 * their cos/sin are computed in fp64 and rounded once to fp32.  Linear
 * scaling ("linear" rope_scaling) is position_scale = factor; NTK-aware
 * scaling (the reading taken of "dynamic" rope_scaling) is ntk_alpha =
 * the context stretch the caller wants, which divides the lowest frequency
 * by exactly ntk_alpha and keeps the highest; ntk_alpha = 1 is no NTK
 * scaling (then rotary_dim may be 2).  Build the table once per
 * configuration.
 */
PKV_API pkv_status pkv_rope_cos_sin_table(float *cos_sin, int max_position, int rotary_dim,
                                          double base, double position_scale, double ntk_alpha,
                                          void *stream);

/*
 * rope_reshape_and_cache: for every token t, at position positions[t]:
 *   - rotate the first rotary_dim dimensions of every q head of query
 *     ([num_tokens, num_qo_heads, head_dim]) and every kv head of key
 *     ([num_tokens, Hkv, head_dim]) in place: the pair (x_a, x_b) of
 *     frequency i turns by the table's angle, x_a' = x_a cos - x_b sin,
 *     x_b' = x_b cos + x_a sin, with (a, b) = (i, i + rotary_dim/2) when
 *     is_neox_style, else (2i, 2i + 1) (RoFormer's rotary embedding); the
 *     other dimensions are not touched;
 *   - then, as pkv_reshape_and_cache, store the rotated key row and the value
 *     row at flat slot slot_mapping[t] (negative: not cached).
 * Arithmetic in fp32, rounded to the dtype of the cache once.  positions and
 * slot_mapping are int64 device arrays; cos_sin is a table built by
 * pkv_rope_cos_sin_table with this rotary_dim and max_position rows.  A token
 * whose position is outside [0, max_position) is left untouched (query, key
 * and cache) and sets PKV_DEVERR_POSITION; a slot >= num_blocks * block_size
 * skips that token's cache write and sets PKV_DEVERR_SLOT.  query may be
 * NULL when num_qo_heads == 0.  Requirements: rotary_dim even, 0 < rotary_dim
 * <= head_dim and a multiple of 2 * (16 / element size) (16 for bf16, 8 for
 * fp32); head_dim a multiple of 16 / element size; every pointer 16-byte
 * aligned (positions and slot_mapping 8-byte).  head_dim is not limited to
 * 64 and 128 here.
 */
PKV_API pkv_status pkv_rope_reshape_and_cache(void *query, void *key, const void *value,
                                              void *k_cache, void *v_cache,
                                              const int64_t *positions,
                                              const int64_t *slot_mapping, int64_t num_tokens,
                                              int num_qo_heads, pkv_cache_desc cache,
                                              const float *cos_sin, int max_position,
                                              int rotary_dim, int is_neox_style,
                                              int32_t *dev_error, void *stream);

/*
 * Workspace bytes pkv_paged_decode needs: split-KV partials for
 * batch x num_qo_heads x P partitions, P = ceil(max_seqlen / partition_size)
 * (fewer with a window).  partition_size 0 means 512.
 */
PKV_API size_t pkv_paged_decode_workspace_size(int batch, int num_qo_heads, int head_dim,
                                       int max_seqlen, int partition_size, int window_left);

/*
 * paged_decode: out[b, h, :] for one query q[b, h, :] per sequence.
 *   out, q        [batch, num_qo_heads, head_dim], contiguous, cache dtype
 *   block_table   [batch, max_blocks_per_seq] int32 (device)
 *   cache_seqlens [batch] int32 (device): attended length L_b; the query sits
 *                 at position L_b - 1 (write the new token first, then pass
 *                 the length including it)
 *   max_seqlen    host int >= every cache_seqlens[b] (sizes the grid)
 *   sink          [num_qo_heads] fp32 (device) or NULL
 *   alibi_slopes  [num_qo_heads] fp32 (device) or NULL: with slopes the
 *                 logit of key j gains alibi_slopes[h] * (j - (L_b - 1))
 *   window_left   -1 for none, else keep keys j >= L_b - 1 - window_left
 *   head sizes: bf16 64/80/96/112/128/256, fp32 64/80/96/112/128 (the
 *                 kernels pad to 64, 128 or 256 with zeros; the padding reads
 *                 no memory)
 *   partition_size split-KV partition in tokens (0 = 512); a multiple of
 *                 block_size, at most 16384; partitions start at multiples of
 *                 it
 *   lse_out       [batch, num_qo_heads] fp32 (device) or NULL
 *   workspace     device scratch of at least pkv_paged_decode_workspace_size
 *                 bytes, 256-byte aligned; contents need no initialisation
 * Sequences longer than max_seqlen are clipped to it and set
 * PKV_DEVERR_SEQLEN.
 */
PKV_API pkv_status pkv_paged_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                            pkv_cache_desc cache, const int32_t *block_table,
                            int max_blocks_per_seq, const int32_t *cache_seqlens,
                            int max_seqlen, const float *sink, const float *alibi_slopes,
                            int batch, int num_qo_heads, int window_left, float sm_scale,
                            int partition_size, float *lse_out, void *workspace,
                            size_t workspace_bytes, int32_t *dev_error, void *stream);

/* Workspace bytes pkv_varlen_prefill needs (its work-tile list). */
PKV_API size_t pkv_varlen_prefill_workspace_size(int batch, int num_qo_heads, int num_kv_heads,
                                         int total_q, int max_seqlen_q);

/*
 * varlen_prefill: attention of every query row over its request's paged keys.
 *   out, q         [total_q, num_qo_heads, head_dim] bf16, contiguous
 *   cu_seq_lens_q  [batch+1] int32 (device), exclusive prefix sums of q_len
 *   cu_seq_lens_k  [batch+1] int32 (device), exclusive prefix sums of kv_len;
 *                  only the differences are used -- keys come from the pages
 *   max_seqlen_q/k host ints >= every q_len / kv_len
 *   total_q        host int == cu_seq_lens_q[batch]
 *   causal         1: key j <= qpos (the mask aligned to the end of kv);
 *                  0: no upper bound, window_left >= 0 still drops keys
 *                  before qpos - window_left (FlashInfer
 *                  sink_attention_reference.py, non-causal varlen mask)
 *   sink, alibi_slopes (bias alibi_slopes[h] * (j - qpos)), window_left,
 *   sm_scale, lse_out ([total_q, num_qo_heads]) as in
 *   paged_decode.  Causal rows whose position is negative (q_len > kv_len)
 *   keep no key.  Supported: bf16 pools, head_dim 64/80/96/112/128 (the
 *   tiles are padded to 128 with zeros), block_size 16 or 32,
 *   G = num_qo_heads / num_kv_heads a power of two <= 16; anything else
 *   returns PKV_ERR_UNSUPPORTED.
 *   max_ctas       host int: at most this many CTAs of the attention kernel
 *                  run at once (each takes one SM and draws work items until
 *                  none is left); 0 means one per SM.  A smaller number
 *                  leaves SMs free for work the caller runs beside the call
 *                  on another stream (a decode, for example); the result
 *                  does not depend on it.  Head size 256 ignores it.
 */
PKV_API pkv_status pkv_varlen_prefill(void *out, const void *q, const void *k_cache,
                              const void *v_cache, pkv_cache_desc cache,
                              const int32_t *block_table, int max_blocks_per_seq,
                              const int32_t *cu_seq_lens_q, const int32_t *cu_seq_lens_k,
                              int max_seqlen_q, int max_seqlen_k, int total_q,
                              const float *sink, const float *alibi_slopes, int batch,
                              int num_qo_heads, int causal, int window_left, float sm_scale,
                              float *lse_out, void *workspace, size_t workspace_bytes,
                              int max_ctas, int32_t *dev_error, void *stream);

/*
 * varlen_prefill_contiguous: varlen_prefill with the keys and values of all
 * requests packed, not paged.
 *   k, v           [total_k, num_kv_heads, head_dim] (dtype: PKV_BF16),
 *                  contiguous, 16-byte aligned device memory owned by the
 *                  caller; may be NULL when total_k == 0
 *   total_k        host int, rows of k and v (normally cu_seq_lens_k[batch])
 *   cu_seq_lens_k  [batch+1] int32 (device): request r's keys are rows
 *                  cu_seq_lens_k[r] .. cu_seq_lens_k[r+1]-1
 * Every other argument as in pkv_varlen_prefill, and the same workspace
 * (pkv_varlen_prefill_workspace_size).  A request whose rows run past total_k
 * is clipped to the rows that exist and PKV_DEVERR_SEQLEN is raised in
 * dev_error; nothing outside k and v is read.
 */
PKV_API pkv_status pkv_varlen_prefill_contiguous(void *out, const void *q, const void *k,
                                                 const void *v, int total_k, int num_kv_heads,
                                                 int head_dim, int dtype,
                                                 const int32_t *cu_seq_lens_q,
                                                 const int32_t *cu_seq_lens_k, int max_seqlen_q,
                                                 int max_seqlen_k, int total_q, const float *sink,
                                                 const float *alibi_slopes, int batch,
                                                 int num_qo_heads, int causal, int window_left,
                                                 float sm_scale, float *lse_out,
                                                 void *workspace, size_t workspace_bytes,
                                                 int32_t *dev_error, void *stream);

/*
 * MInference vertical + slash sparse prefill of one sequence (nano-vllm
 * minference.py, MInferencePolicy).  Two steps, both on the GPU:
 *   1. the pattern (estimate_pattern): the last min(64, S) queries attend
 *      causally to every key with logits sm_scale * <q, k>; each row's softmax
 *      probabilities are summed per key column (vertical scores) and per
 *      diagonal d = position - key (slash scores); the first num_sink_tokens
 *      columns and num_recent_diags diagonals count as +inf; the nv highest
 *      columns and ns highest diagonals of every query head are kept (equal
 *      scores: lower index first), in ascending order.  nv, ns: see
 *      pkv_minference_sizes.  Scores and sums in fp32.
 *   2. the attention: query row i (position i) keeps key j iff j <= i and
 *      (j is a kept column of its head, or i - j a kept diagonal); softmax
 *      over the kept keys; o = sum p v (a row keeping nothing gets 0).  The
 *      pages leave the sparse kernel itself to a library they do not show;
 *      this is the element-wise reading of "vertical + slash".
 *   q, out [S, num_qo_heads, head_dim], k, v [S, num_kv_heads, head_dim]:
 *   bf16, contiguous; head_dim 64..128 (multiple of 16); S <= 131072;
 *   num_qo_heads / num_kv_heads a power of two <= 16.
 *   vertical_indices [num_qo_heads, nv], slash_indices [num_qo_heads, ns]:
 *   optional int32 device outputs (NULL: kept in the workspace).
 *   workspace: pkv_minference_workspace_size bytes, 256-byte aligned.
 */
PKV_API pkv_status pkv_minference_sizes(int seq_len, int vertical_size, int slash_size,
                                        double adaptive_budget, int num_sink_tokens,
                                        int num_recent_diags, int *nv, int *ns);
/* nv, ns: with adaptive_budget > 0, b = (int)(S * adaptive_budget),
 * nv = max(num_sink + 1, (int)(0.2 b)), ns = max(num_recent + 1, (int)(0.8 b));
 * otherwise vertical_size, slash_size; both capped at S. */

PKV_API size_t pkv_minference_workspace_size(int seq_len, int num_qo_heads, int num_kv_heads,
                                             int vertical_size, int slash_size,
                                             double adaptive_budget, int num_sink_tokens,
                                             int num_recent_diags);

PKV_API pkv_status pkv_minference_prefill(void *out, const void *q, const void *k,
                                          const void *v, int seq_len, int num_qo_heads,
                                          int num_kv_heads, int head_dim, int dtype,
                                          int vertical_size, int slash_size,
                                          double adaptive_budget, int num_sink_tokens,
                                          int num_recent_diags, float sm_scale,
                                          int32_t *vertical_indices, int32_t *slash_indices,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *dev_error, void *stream);

/*
 * paged_decode_noalloc: paged_decode for callers that cannot allocate device
 * memory at the call site -- for example a plug-in whose host framework owns
 * all device memory and exposes no allocator to it, or a serving loop that
 * must not allocate once it is running.  The pages have no counterpart: this
 * entry point exists only for such callers.
 *
 * It takes the same arguments as pkv_paged_decode minus the workspace and
 * minus alibi_slopes (no ALiBi bias).  The
 * split-KV scratch is instead a fixed device array inside the library of
 * PKV_NOALLOC_DECODE_SCRATCH_BYTES bytes; every GPU that loads the library
 * holds that array until the process exits.  A problem whose scratch need
 * (pkv_paged_decode_workspace_size) exceeds it is rejected with
 * PKV_ERR_WORKSPACE before anything is launched.  The caller still provides
 * out, q, the pools and the metadata; nothing is allocated.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept for the life of the process: after a
 * cudaDeviceReset of that device the entry point must not be called again
 * (the reset unloads the array; the kept address would then be stale).  A
 * call with batch == 0 returns PKV_OK without touching the device.  All calls share the one array and it keeps the last call's
 * contents: nothing in it needs to start at zero, because every call writes
 * each partial it later reads.  Calls that can overlap on the GPU (concurrent
 * streams, or several host threads) race on the array: serialise them.
 */
#define PKV_NOALLOC_DECODE_SCRATCH_BYTES ((size_t)32 << 20)

PKV_API pkv_status pkv_paged_decode_noalloc(void *out, const void *q, const void *k_cache,
                                            const void *v_cache, pkv_cache_desc cache,
                                            const int32_t *block_table, int max_blocks_per_seq,
                                            const int32_t *cache_seqlens, int max_seqlen,
                                            const float *sink, int batch, int num_qo_heads,
                                            int window_left, float sm_scale,
                                            int partition_size, float *lse_out,
                                            int32_t *dev_error, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
