/*
 * pkv_oracle.c -- plain fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library: it is written separately, from the
 * definitions on the source pages, so that the two can be compared.
 *
 * Every step is a plain loop, in the order the definitions state it:
 *   - token -> request assignment by cumulative sequence lengths and the
 *     paged address of a logical position (transformers docs "paged_attention":
 *     "Varlen path" example and "Decode path" example);
 *   - logits s_j = sm_scale * <q, k_j>, computed on the exact values of the
 *     inputs widened to double (sink_attention_reference.py, FlashInfer tests:
 *     sink_attention_unified, the einsum followed by "* sm_scale");
 *   - GQA: query head h reads kv head h / (Hq / Hkv)
 *     (sink_attention_reference.py, repeat_interleave over the head axis;
 *     vLLM attention.py, PagedAttention.head_mapping);
 *   - causal mask aligned to the end of the kv sequence: the query in row i
 *     of a request sits at position kv_len - q_len + i and keeps key j iff
 *     j <= that position; a sliding window additionally needs
 *     position - window_left <= j (sink_attention_reference.py, varlen branch
 *     and the incremental-mode mask);
 *   - sink softmax: the per-query-head sink logit is one extra softmax column
 *     that is dropped after normalising, so the denominator gains exp(sink[h])
 *     (sink_attention_reference.py, sink_softmax);
 *   - ALiBi (optional): slope[h] * (j - position) is added to the scaled
 *     logit (vLLM attention.py, PagedAttentionWithALiBi);
 *   - o = sum_j p_j v_j (the final einsum).
 *
 * Readings where the pages are silent (they are listed with the design notes):
 *   - sink[h] is a logit in natural-log units and is not multiplied by
 *     sm_scale (it is concatenated after the logits were scaled);
 *   - a NULL sink means "no sink" (-inf); with no sink the result is the
 *     plain softmax;
 *   - a row with no attended key has output 0 (and lse = the sink, or -inf);
 *   - lse = log(sum_j exp(s_j) + exp(sink[h])), the full softmax
 *     denominator, natural log.
 *
 * Precision: every input value (fp32, or bf16 given as its 16 raw bits) is
 * widened exactly to double; all arithmetic is double; nothing is rounded.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* ------------------------------------------------------------------------ */
/* indexing                                                                  */
/* ------------------------------------------------------------------------ */

/* For every token t in [0, total), the request r with cu[r] <= t < cu[r+1].
 * Empty requests own no token.  Returns 0, or -1 if some token has no owner
 * (cu not covering [0, total)). */
int oracle_token_to_request(const int32_t *cu, int batch, int total, int32_t *out) {
    for (int t = 0; t < total; ++t) {
        out[t] = -1;
        for (int r = 0; r < batch; ++r) {
            if (cu[r] <= t && t < cu[r + 1]) {
                out[t] = r;
                break;
            }
        }
        if (out[t] < 0) return -1;
    }
    return 0;
}

/* Flat cache slot of logical position pos of sequence b: the page that the
 * block table names for that position, times the page size, plus the offset
 * inside the page.  Returns -1 for an unallocated (-1) page entry. */
int64_t oracle_slot(const int32_t *block_table, int max_blocks_per_seq, int b, int pos,
                    int block_size) {
    int32_t page = block_table[(int64_t)b * max_blocks_per_seq + pos / block_size];
    if (page < 0) return -1;
    return (int64_t)page * block_size + pos % block_size;
}

/* The cache write: row slot_mapping[t] of each pool receives row t of key and
 * value, bit for bit.  A negative slot means "do not cache this token"
 * (vLLM attention.py, PagedAttention.forward: the to_cache filter before
 * reshape_and_cache).  row_bytes is the size of one token's row
 * (num_kv_heads * head_dim * element size). */
void oracle_reshape_and_cache(const uint8_t *key, const uint8_t *value, uint8_t *k_cache,
                              uint8_t *v_cache, const int64_t *slot_mapping, int num_tokens,
                              int64_t row_bytes) {
    for (int t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        memcpy(k_cache + s * row_bytes, key + (int64_t)t * row_bytes, (size_t)row_bytes);
        memcpy(v_cache + s * row_bytes, value + (int64_t)t * row_bytes, (size_t)row_bytes);
    }
}

/* ------------------------------------------------------------------------ */
/* attention                                                                 */
/* ------------------------------------------------------------------------ */

static double widen(const void *base, int dtype, int64_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    /* bf16: the 16 bits are the upper half of an fp32 */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    /* outputs */
    double *out;           /* [nrows, Hq, D] */
    double *lse;           /* [nrows, Hq] or NULL */
    /* inputs */
    const void *q;         /* [total_q, Hq, D] */
    int q_dtype;
    const void *k_cache;   /* [num_blocks, block_size, Hkv, D] */
    const void *v_cache;
    int kv_dtype;
    int64_t num_blocks;
    int block_size, num_kv_heads, head_dim;
    const int32_t *block_table;
    int max_blocks_per_seq;
    const int32_t *cu_q;   /* [batch+1] */
    const int32_t *kv_lens;/* [batch] */
    int batch, num_qo_heads;
    const float *sink;     /* [Hq] or NULL */
    const float *alibi;    /* [Hq] ALiBi slopes or NULL */
    int causal, window_left;
    double sm_scale;
    const int32_t *rows;   /* which query rows to compute, or NULL = all */
    int nrows;
    /* work distribution */
    int64_t next_unit;
    pthread_mutex_t lock;
    int status;
} job_t;

/* One (query row, query head) output: the definition written out. */
static int attend_one(job_t *J, int out_row, int t, int h, double *s_buf) {
    const int Hq = J->num_qo_heads, Hkv = J->num_kv_heads, D = J->head_dim;
    /* which request owns query row t */
    int r = -1;
    for (int i = 0; i < J->batch; ++i)
        if (J->cu_q[i] <= t && t < J->cu_q[i + 1]) { r = i; break; }
    if (r < 0) return -1;
    const int q_len = J->cu_q[r + 1] - J->cu_q[r];
    const int kv_len = J->kv_lens[r];
    const int i_row = t - J->cu_q[r];
    const int64_t qpos = (int64_t)kv_len - q_len + i_row; /* the query's position */
    const int group = Hq / Hkv;

    {
        const int g = h / group;
        const double sink = J->sink ? (double)J->sink[h] : -INFINITY;
        double *o = J->out + ((int64_t)out_row * Hq + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;

        /* logits of the allowed keys; disallowed keys get -inf */
        double m = sink;
        int any = 0;
        for (int j = 0; j < kv_len; ++j) {
            int allowed = 1;
            if (J->causal && !((int64_t)j <= qpos)) allowed = 0;
            if (J->window_left >= 0 && !(qpos - J->window_left <= (int64_t)j)) allowed = 0;
            if (!allowed) { s_buf[j] = -INFINITY; continue; }
            int64_t slot = oracle_slot(J->block_table, J->max_blocks_per_seq, r, j, J->block_size);
            if (slot < 0 || slot >= J->num_blocks * J->block_size) return -2;
            const int64_t kbase = (slot * Hkv + g) * D;
            const int64_t qbase = ((int64_t)t * Hq + h) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += widen(J->q, J->q_dtype, qbase + d) * widen(J->k_cache, J->kv_dtype, kbase + d);
            s_buf[j] = J->sm_scale * dot;
            /* ALiBi: the scaled logit gains slope[h] times the signed distance
             * of the key from the query's position (vLLM attention.py,
             * PagedAttentionWithALiBi.set_attn_bias: bias[i][j] = j - i times
             * the head's slope, added to the scaled scores) */
            if (J->alibi) s_buf[j] += (double)J->alibi[h] * (double)((int64_t)j - qpos);
            if (s_buf[j] > m) m = s_buf[j];
            any = 1;
        }
        if (!any) {
            /* nothing attended: the sink column (if any) takes all the mass
             * and is dropped, so the output is 0 */
            if (J->lse) J->lse[(int64_t)out_row * Hq + h] = sink;
            return 0;
        }
        /* softmax over [s_0 .. s_{n-1}, sink], sink column dropped */
        double z = exp(sink - m); /* exp(-inf) = 0 when there is no sink */
        for (int j = 0; j < kv_len; ++j)
            if (s_buf[j] != -INFINITY) z += exp(s_buf[j] - m);
        for (int j = 0; j < kv_len; ++j) {
            if (s_buf[j] == -INFINITY) continue;
            const double p = exp(s_buf[j] - m) / z;
            int64_t slot = oracle_slot(J->block_table, J->max_blocks_per_seq, r, j, J->block_size);
            const int64_t vbase = (slot * Hkv + g) * D;
            for (int d = 0; d < D; ++d) o[d] += p * widen(J->v_cache, J->kv_dtype, vbase + d);
        }
        if (J->lse) J->lse[(int64_t)out_row * Hq + h] = m + log(z);
    }
    return 0;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    int64_t max_kv = 1;
    for (int r = 0; r < J->batch; ++r)
        if (J->kv_lens[r] > max_kv) max_kv = J->kv_lens[r];
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_kv);
    if (!s_buf) {
        pthread_mutex_lock(&J->lock);
        J->status = -3;
        pthread_mutex_unlock(&J->lock);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= (int64_t)J->nrows * J->num_qo_heads) break;
        const int row = (int)(u / J->num_qo_heads), h = (int)(u % J->num_qo_heads);
        int t = J->rows ? J->rows[row] : row;
        int st = attend_one(J, row, t, h, s_buf);
        if (st != 0) {
            pthread_mutex_lock(&J->lock);
            J->status = st;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(s_buf);
    return NULL;
}

/* Attention of every (listed) query row over its request's paged K/V.
 *
 * Decode is the special case cu_q = [0, 1, ..., batch] with kv_lens =
 * cache_seqlens: the single query sits at position kv_len - 1.
 *
 * rows: NULL computes all cu_q[batch] rows (nrows must equal that);
 * otherwise out row u is query row rows[u].
 * nthreads <= 0 uses every online core.  Returns 0; -1 if a row has no
 * request; -2 if an attended key's page is unallocated or out of the pool;
 * -3 on allocation failure; -4 on bad arguments. */
int oracle_attention(double *out, double *lse, const void *q, int q_dtype, const void *k_cache,
                     const void *v_cache, int kv_dtype, int64_t num_blocks, int block_size,
                     int num_kv_heads, int head_dim, const int32_t *block_table,
                     int max_blocks_per_seq, const int32_t *cu_q, const int32_t *kv_lens,
                     int batch, int num_qo_heads, const float *sink, const float *alibi,
                     int causal, int window_left, double sm_scale, const int32_t *rows,
                     int nrows, int nthreads) {
    if (num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || batch < 0 || nrows < 0)
        return -4;
    job_t J;
    memset(&J, 0, sizeof J);
    J.out = out; J.lse = lse; J.q = q; J.q_dtype = q_dtype;
    J.k_cache = k_cache; J.v_cache = v_cache; J.kv_dtype = kv_dtype;
    J.num_blocks = num_blocks; J.block_size = block_size;
    J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.block_table = block_table; J.max_blocks_per_seq = max_blocks_per_seq;
    J.cu_q = cu_q; J.kv_lens = kv_lens; J.batch = batch; J.num_qo_heads = num_qo_heads;
    J.sink = sink; J.alibi = alibi; J.causal = causal; J.window_left = window_left; J.sm_scale = sm_scale;
    J.rows = rows; J.nrows = nrows;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > (int64_t)nrows * num_qo_heads && nrows > 0)
        nthreads = nrows * num_qo_heads;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -3;
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

int oracle_online_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* ------------------------------------------------------------------------ */
/* rotary position embedding                                                 */
/* ------------------------------------------------------------------------ */

/* The rotary step that precedes the cache write (vLLM attention.py,
 * PagedAttentionWithRoPE.forward: rotary_emb(positions, query, key) with
 * head_size, rotary_dim, base, is_neox_style and a rope_scaling factor).
 * The page names those parameters but does not spell the rotation out; it is
 * the rotary position embedding of RoFormer (Su et al., 2021):
 *   - frequency i in [0, rotary_dim/2):  theta_i = base^(-2i / rotary_dim);
 *   - a token at position m turns the pair (x_a, x_b) of frequency i by the
 *     angle m' * theta_i, where m' = m / position_scale (linear position
 *     scaling; 1 means none):
 *         x_a' = x_a cos - x_b sin,   x_b' = x_b cos + x_a sin;
 *   - the pairs: neox style (a, b) = (i, i + rotary_dim/2), the two halves
 *     of the rotated part; otherwise (GPT-J style) (a, b) = (2i, 2i + 1);
 *   - dimensions rotary_dim .. head_dim-1 are not rotated.
 * The page's "dynamic" rope_scaling is read as NTK-aware scaling: to stretch
 * the usable context ntk_alpha times, the base is raised to
 *   base * ntk_alpha^(rotary_dim / (rotary_dim - 2)),
 * which divides the lowest frequency (i = rotary_dim/2 - 1) by exactly
 * ntk_alpha and leaves the highest (i = 0) alone; ntk_alpha = 1 is no
 * scaling.
 * x: [num_tokens, num_heads, head_dim] in dtype; out: the same shape, fp64,
 * every value exact up to the rounding of double arithmetic. */
void oracle_rope(double *out, const void *x, int dtype, int64_t num_tokens, int num_heads,
                 int head_dim, const int64_t *positions, int rotary_dim, double base,
                 double position_scale, double ntk_alpha, int neox) {
    const int half = rotary_dim / 2;
    if (ntk_alpha != 1.0) base = base * pow(ntk_alpha, (double)rotary_dim / (rotary_dim - 2));
    for (int64_t t = 0; t < num_tokens; ++t) {
        const double m = (double)positions[t] / position_scale;
        for (int h = 0; h < num_heads; ++h) {
            const int64_t row = (t * num_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) out[row + d] = widen(x, dtype, row + d);
            for (int i = 0; i < half; ++i) {
                const double theta = pow(base, -2.0 * i / rotary_dim);
                const double c = cos(m * theta), s = sin(m * theta);
                const int a = neox ? i : 2 * i;
                const int b = neox ? i + half : 2 * i + 1;
                const double xa = widen(x, dtype, row + a), xb = widen(x, dtype, row + b);
                out[row + a] = xa * c - xb * s;
                out[row + b] = xb * c + xa * s;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MInference vertical + slash sparse prefill                                */
/* ------------------------------------------------------------------------ */

/* Pattern scores (nano-vllm minference.py, MInferencePolicy.estimate_pattern):
 * the last `last_q` queries of a sequence of S tokens (positions
 * S - last_q .. S - 1) attend causally to all keys; each row's softmax
 * probabilities p_i(j) are summed
 *   - per key column:   vertical[h][j] = sum_i p_i(j)
 *   - per diagonal:     slash[h][d]    = sum_i p_i(pos_i - d),  d = pos_i - j.
 * q: [S, Hq, D], k: [S, Hkv, D] (query head h reads kv head h / (Hq / Hkv));
 * the logit is scale * <q, k>.  vertical, slash: [Hq, S] fp64 outputs. */
void oracle_minference_scores(double *vertical, double *slash, const void *q, const void *k,
                              int dtype, int S, int num_qo_heads, int num_kv_heads,
                              int head_dim, int last_q, double scale) {
    const int Hq = num_qo_heads, Hkv = num_kv_heads, D = head_dim;
    const int group = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    for (int h = 0; h < Hq; ++h) {
        const int kvh = h / group;
        double *vh = vertical + (int64_t)h * S, *sh = slash + (int64_t)h * S;
        for (int j = 0; j < S; ++j) vh[j] = sh[j] = 0.0;
        for (int i = 0; i < last_q; ++i) {
            const int pos = S - last_q + i;
            const int64_t qb = ((int64_t)pos * Hq + h) * D;
            double m = -INFINITY;
            for (int j = 0; j <= pos; ++j) {
                const int64_t kb = ((int64_t)j * Hkv + kvh) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += widen(q, dtype, qb + d) * widen(k, dtype, kb + d);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double z = 0.0;
            for (int j = 0; j <= pos; ++j) z += exp(s[j] - m);
            for (int j = 0; j <= pos; ++j) {
                const double p = exp(s[j] - m) / z;
                vh[j] += p;
                sh[pos - j] += p;
            }
        }
    }
    free(s);
}

/* Vertical + slash sparse attention of one sequence (the attention the
 * pattern selects): query row i (position i) keeps key j iff j <= i and
 * (j is a vertical index of its head, or i - j is a slash index of its
 * head); softmax over the kept keys, o = sum p v.  A row that keeps no key
 * gets 0.  vert: [Hq, nv] and slash_idx: [Hq, ns] key / diagonal indices.
 * out: [S, Hq, D] fp64. */
void oracle_sparse_attention(double *out, const void *q, const void *k, const void *v, int dtype,
                             int S, int num_qo_heads, int num_kv_heads, int head_dim,
                             const int32_t *vert, int nv, const int32_t *slash_idx, int ns,
                             double scale) {
    const int Hq = num_qo_heads, Hkv = num_kv_heads, D = head_dim;
    const int group = Hq / Hkv;
    uint8_t *isv = (uint8_t *)calloc((size_t)(S > 0 ? S : 1), 1);
    uint8_t *iss = (uint8_t *)calloc((size_t)(S > 0 ? S : 1), 1);
    double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    for (int h = 0; h < Hq; ++h) {
        const int kvh = h / group;
        memset(isv, 0, (size_t)S);
        memset(iss, 0, (size_t)S);
        for (int a = 0; a < nv; ++a) {
            const int j = vert[(int64_t)h * nv + a];
            if (j >= 0 && j < S) isv[j] = 1;
        }
        for (int a = 0; a < ns; ++a) {
            const int d = slash_idx[(int64_t)h * ns + a];
            if (d >= 0 && d < S) iss[d] = 1;
        }
        for (int i = 0; i < S; ++i) {
            double *o = out + ((int64_t)i * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            const int64_t qb = ((int64_t)i * Hq + h) * D;
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                if (!(isv[j] || iss[i - j])) { s[j] = -INFINITY; continue; }
                const int64_t kb = ((int64_t)j * Hkv + kvh) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += widen(q, dtype, qb + d) * widen(k, dtype, kb + d);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            if (m == -INFINITY) continue;
            double z = 0.0;
            for (int j = 0; j <= i; ++j)
                if (s[j] != -INFINITY) z += exp(s[j] - m);
            for (int j = 0; j <= i; ++j) {
                if (s[j] == -INFINITY) continue;
                const double p = exp(s[j] - m) / z;
                const int64_t vb = ((int64_t)j * Hkv + kvh) * D;
                for (int d = 0; d < D; ++d) o[d] += p * widen(v, dtype, vb + d);
            }
        }
    }
    free(isv);
    free(iss);
    free(s);
}
