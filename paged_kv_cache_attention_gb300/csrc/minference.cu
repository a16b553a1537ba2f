// minference.cu -- the vertical + slash pattern of MInference sparse prefill
// (nano-vllm minference.py, MInferencePolicy.estimate_pattern).
//
// For one sequence of S tokens: the last lq = min(64, S) queries attend
// causally to every key; each row's softmax probabilities are summed per key
// column (vertical scores) and per diagonal d = position - key (slash
// scores); the first num_sink columns and num_recent diagonals are forced in;
// the top nv columns and ns diagonals of every query head are kept, in
// ascending order.  The attention itself runs in prefill.cu (SPARSE form),
// masked by bitmaps of the kept columns and diagonals that this file builds.
//
// GB300 design.  Dot products on the tensor cores (mma.sync, bf16 in, fp32
// out), softmax and sums in fp32 (the page's softmax and sums are fp32):
//   mi_scores_kernel<1>  one CTA per (128-key block, query head): the lq
//                        query rows and the key block in shared memory,
//                        warp tiles of 64 rows x 32 keys; per row the
//                        block's maximum and sum of exponentials;
//   mi_lse_kernel        per (head, row) the log-sum-exp over the blocks;
//   mi_scores_kernel<2>  recomputes the block's logits, p = exp(s - lse);
//                        column sums -> vertical scores of the block's keys;
//                        diagonal sums of the block -> per-block partials;
//   mi_slash_kernel      adds each diagonal's (at most two) partials;
//   mi_topk_kernel       one CTA per (head, kind): radix select of the k-th
//                        largest score on the float bits, then a block-scan
//                        compaction that writes the kept indices in
//                        ascending order (equal scores: lower index first);
//   mi_bitmap_kernel     bitmaps of the kept columns / diagonals and their
//                        per-word prefix bit counts, for the attention's
//                        per-element masks and per-tile skipping.
// Every reduction runs in a fixed order: the pattern is deterministic.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kLastQ = 64;
constexpr int kBlk = 128;  // keys per score block
constexpr int kScoreThreads = 128;
constexpr int kDiagSpan = kLastQ + kBlk - 1;  // diagonals one block touches (<= 191)
constexpr int kDiagSlots = 192;
constexpr int kTopkThreads = 1024;

// ---------------------------------------------------------------------------
// scores
// ---------------------------------------------------------------------------
// One CTA per (128-key block, query head), 4 warps.  Q rows (lq <= 64) and the
// key block sit in shared memory as bf16 rows padded by 16 bytes (ldmatrix
// without bank conflicts); warp w computes S[64 x 32] for keys 32w..32w+31
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate): 4 m-tiles x 4 n-tiles.
// Then pass 1 writes the rows' block maxima and sums of exponentials, pass 2
// the probabilities' column sums and diagonal partials (through a [64][128]
// fp32 shared array, reduced in a fixed order).
constexpr int kPadRow = 16;  // bytes of padding per shared row

__host__ __device__ constexpr int mi_row_bytes(int D) { return D * 2 + kPadRow; }

template <int PASS>
__global__ void __launch_bounds__(kScoreThreads)
mi_scores_kernel(MinferenceParams p) {
    extern __shared__ __align__(16) uint8_t sm8[];
    const int D = p.head_dim;
    const int RB = mi_row_bytes(D);
    uint8_t *qs = sm8;                          // [kLastQ][RB]
    uint8_t *ks = sm8 + kLastQ * RB;            // [kBlk][RB]
    float *ps = reinterpret_cast<float *>(sm8 + (kLastQ + kBlk) * RB);  // [kLastQ][kBlk]
    float *red = ps + kLastQ * kBlk;            // [4 warps][kLastQ] x 2
    const int blk = blockIdx.x, h = blockIdx.y;
    const int S = p.seq_len, lq = p.last_q;
    const int G = p.num_qo_heads / p.num_kv_heads, g = h / G;
    const int j0 = blk * kBlk;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
    const int vec = D / 8;  // 16-byte vectors per row
    for (int e = t; e < kLastQ * vec; e += kScoreThreads) {
        const int i = e / vec, c = e - i * vec;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (i < lq)
            v = *reinterpret_cast<const uint4 *>(
                q + ((int64_t)(S - lq + i) * p.num_qo_heads + h) * D + c * 8);
        *reinterpret_cast<uint4 *>(qs + i * RB + c * 16) = v;
    }
    for (int e = t; e < kBlk * vec; e += kScoreThreads) {
        const int r = e / vec, c = e - r * vec;
        const int j = j0 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j < S)
            v = *reinterpret_cast<const uint4 *>(k + ((int64_t)j * p.num_kv_heads + g) * D + c * 8);
        *reinterpret_cast<uint4 *>(ks + r * RB + c * 16) = v;
    }
    __syncthreads();
    float acc[4][4][4];  // [m-tile][n-tile][fragment]
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
    const uint32_t qs_u = smem_u32(qs), ks_u = smem_u32(ks);
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t af[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int chunk = kk * 2 + (lane >> 4);
            ldsm_x4(qs_u + row * RB + chunk * 16, af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
        }
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // pairs of n-tiles: one ldmatrix x4 each
            // lanes 0-7: keys of n-tile 2np, k 0-7; 8-15: same keys, k 8-15;
            // 16-23: n-tile 2np+1, k 0-7; 24-31: n-tile 2np+1, k 8-15
            const int key = warp * 32 + np * 16 + ((lane >> 4) << 3) + (lane & 7);
            const int chunk = kk * 2 + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ks_u + key * RB + chunk * 16, b0, b1, b2, b3);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                mma_bf16_16816(acc[mt][2 * np], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
                mma_bf16_16816(acc[mt][2 * np + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2,
                               b3);
            }
        }
    }
    // logits (fragment c: row mt*16 + lane/4 + 8*(c>>1), key nt*8 + 2*(lane%4) + (c&1));
    // a key past the row's position (or past S) is masked
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = mt * 16 + (lane >> 2) + 8 * (c >> 1);
                const int j = j0 + warp * 32 + nt * 8 + 2 * (lane & 3) + (c & 1);
                acc[mt][nt][c] =
                    (i < lq && j <= S - lq + i) ? acc[mt][nt][c] * p.scale : -INFINITY;
            }
    if constexpr (PASS == 1) {
        // per row: block maximum and sum of exp(s - max) -- first within the
        // warp (the 4 lanes of a row), then over the 4 warps in fixed order
        float *rm = red, *rl = red + 4 * kLastQ;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float m = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    m = fmaxf(m, fmaxf(acc[mt][nt][2 * hf], acc[mt][nt][2 * hf + 1]));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                float l = 0.f;
                if (m != -INFINITY) {
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
                        l += expf(acc[mt][nt][2 * hf] - m) + expf(acc[mt][nt][2 * hf + 1] - m);
                }
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                const int i = mt * 16 + (lane >> 2) + 8 * hf;
                if ((lane & 3) == 0) {
                    rm[warp * kLastQ + i] = m;
                    rl[warp * kLastQ + i] = l;
                }
            }
        __syncthreads();
        for (int i = t; i < lq; i += kScoreThreads) {
            float M = -INFINITY;
            for (int w = 0; w < 4; ++w) M = fmaxf(M, rm[w * kLastQ + i]);
            float L = 0.f;
            if (M != -INFINITY)
                for (int w = 0; w < 4; ++w)
                    if (rm[w * kLastQ + i] != -INFINITY)
                        L += rl[w * kLastQ + i] * expf(rm[w * kLastQ + i] - M);
            const int64_t o = ((int64_t)h * p.num_blocks + blk) * kLastQ + i;
            p.stat_m[o] = M;
            p.stat_l[o] = L;
        }
    } else {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = mt * 16 + (lane >> 2) + 8 * hf;
                const float lse = i < lq ? p.lse[(int64_t)h * kLastQ + i] : 0.f;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float x = acc[mt][nt][2 * hf + e];
                        const int c = warp * 32 + nt * 8 + 2 * (lane & 3) + e;
                        ps[i * kBlk + c] = x == -INFINITY ? 0.f : expf(x - lse);
                    }
            }
        __syncthreads();
        // vertical: column sums over the rows, in row order
        for (int c = t; c < kBlk; c += kScoreThreads) {
            float sum = 0.f;
            for (int i = 0; i < lq; ++i) sum += ps[i * kBlk + c];
            if (j0 + c < S) p.vscore[(int64_t)h * S + j0 + c] = sum;
        }
        // slash: diagonal d = (S - lq + i) - (j0 + c); slot dd = d - dbase,
        // dbase = S - lq - j0 - (kBlk - 1), so c = i + (kBlk - 1) - dd
        for (int dd = t; dd < kDiagSlots; dd += kScoreThreads) {
            float sum = 0.f;
            if (dd < kDiagSpan) {
                const int ilo = max(0, dd - (kBlk - 1)), ihi = min(lq - 1, dd);
                for (int i = ilo; i <= ihi; ++i) sum += ps[i * kBlk + i + (kBlk - 1) - dd];
            }
            p.spart[((int64_t)h * p.num_blocks + blk) * kDiagSlots + dd] = sum;
        }
    }
}

__host__ constexpr int mi_scores_smem(int D) {
    return (kLastQ + kBlk) * mi_row_bytes(D) + kLastQ * kBlk * 4 + 8 * kLastQ * 4;
}

__global__ void mi_lse_kernel(MinferenceParams p) {
    const int h = blockIdx.x, i = threadIdx.x;
    if (i >= p.last_q) return;
    float M = -INFINITY;
    for (int b = 0; b < p.num_blocks; ++b)
        M = fmaxf(M, p.stat_m[((int64_t)h * p.num_blocks + b) * kLastQ + i]);
    float L = 0.f;
    for (int b = 0; b < p.num_blocks; ++b) {
        const int64_t o = ((int64_t)h * p.num_blocks + b) * kLastQ + i;
        if (p.stat_m[o] != -INFINITY) L += p.stat_l[o] * expf(p.stat_m[o] - M);
    }
    p.lse[(int64_t)h * kLastQ + i] = M + logf(L);  // every row keeps key 0: L > 0
}

__global__ void mi_slash_kernel(MinferenceParams p) {
    const int h = blockIdx.y;
    const int d = blockIdx.x * blockDim.x + threadIdx.x;
    const int S = p.seq_len, lq = p.last_q;
    if (d >= S) return;
    // blocks whose diagonal span holds d: j0 in [S - lq - d - 127, S - 1 - d]
    const int lo = S - lq - d - (kBlk - 1), hi = S - 1 - d;
    const int blo = max(0, (lo + kBlk - 1) >= 0 ? (lo + kBlk - 1) / kBlk : 0);
    const int bhi = min(p.num_blocks - 1, hi / kBlk);
    float sum = 0.f;
    for (int b = blo; b <= bhi; ++b) {
        const int j0 = b * kBlk;
        const int dd = d - (S - lq - j0 - (kBlk - 1));
        if (dd >= 0 && dd < kDiagSpan)
            sum += p.spart[((int64_t)h * p.num_blocks + b) * kDiagSlots + dd];
    }
    p.sscore[(int64_t)h * S + d] = sum;
}

// ---------------------------------------------------------------------------
// top-k: blockIdx.x = head, blockIdx.y = 0 vertical / 1 slash
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t score_key(const float *s, int j, int n_force) {
    // scores are >= 0 (sums of probabilities): their bits order like the
    // values; forced entries are +inf
    return j < n_force ? 0x7f800000u : __float_as_uint(fmaxf(s[j], 0.f));
}

__device__ int block_exclusive_scan(int v, int *scratch, int &total) {
    // scratch: kTopkThreads / 32 ints
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kTopkThreads / 32 ? scratch[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        if (lane < kTopkThreads / 32) scratch[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    total = scratch[kTopkThreads / 32 - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kTopkThreads) mi_topk_kernel(MinferenceParams p) {
    __shared__ int hist[256];
    __shared__ int scratch[kTopkThreads / 32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remain;
    const int h = blockIdx.x, kind = blockIdx.y;
    const int S = p.seq_len;
    const float *s = (kind == 0 ? p.vscore : p.sscore) + (int64_t)h * S;
    const int k = kind == 0 ? p.nv : p.ns;
    const int n_force = kind == 0 ? p.num_sink : p.num_recent;
    int32_t *out = (kind == 0 ? p.vidx : p.sidx) + (int64_t)h * k;
    const int t = threadIdx.x;
    if (t == 0) {
        s_prefix = 0u;
        s_remain = k;
    }
    __syncthreads();
    // radix select, 8 bits at a time from the top: the k-th largest key
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = t; b < 256; b += kTopkThreads) hist[b] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
        for (int j = t; j < S; j += kTopkThreads) {
            const uint32_t key = score_key(s, j, n_force);
            if ((key & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        if (t == 0) {
            int remain = s_remain, b = 255;
            for (; b > 0; --b) {
                if (hist[b] >= remain) break;
                remain -= hist[b];
            }
            s_remain = remain;
            s_prefix = prefix | ((uint32_t)b << shift);
        }
        __syncthreads();
    }
    const uint32_t T = s_prefix;  // the k-th largest key
    const int need_eq = s_remain;  // keys equal to T to keep (the lowest indices)
    // compaction in index order
    int eq_base = 0, out_base = 0;
    for (int c0 = 0; c0 < S; c0 += kTopkThreads) {
        const int j = c0 + t;
        const uint32_t key = j < S ? score_key(s, j, n_force) : 0u;
        const bool eq = j < S && key == T;
        int eq_total;
        const int eq_rank = eq_base + block_exclusive_scan(eq ? 1 : 0, scratch, eq_total);
        const bool sel = j < S && (key > T || (eq && eq_rank < need_eq));
        int sel_total;
        const int at = out_base + block_exclusive_scan(sel ? 1 : 0, scratch, sel_total);
        if (sel && at < k) out[at] = j;
        eq_base += eq_total;
        out_base += sel_total;
    }
}

// ---------------------------------------------------------------------------
// bitmaps: one CTA per (head, kind)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTopkThreads) mi_bitmap_kernel(MinferenceParams p) {
    __shared__ int scratch[kTopkThreads / 32];
    const int h = blockIdx.x, kind = blockIdx.y;
    const int W = p.words;
    uint32_t *bits = (kind == 0 ? p.vbits : p.sbits) + (int64_t)h * W;
    int32_t *cnt = (kind == 0 ? p.vcnt : p.scnt) + (int64_t)h * (W + 1);
    const int32_t *idx = (kind == 0 ? p.vidx : p.sidx);
    const int k = kind == 0 ? p.nv : p.ns;
    for (int w = threadIdx.x; w < W; w += kTopkThreads) bits[w] = 0u;
    __syncthreads();
    for (int a = threadIdx.x; a < k; a += kTopkThreads) {
        const int j = idx[(int64_t)h * k + a];
        if (j >= 0 && j < p.seq_len) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    // cnt[w] = set bits in words [0, w)
    int base = 0;
    for (int w0 = 0; w0 < W; w0 += kTopkThreads) {
        const int w = w0 + threadIdx.x;
        const int c = w < W ? __popc(bits[w]) : 0;
        int total;
        const int before = block_exclusive_scan(c, scratch, total);
        if (w < W) cnt[w] = base + before;
        base += total;
    }
    if (threadIdx.x == 0) cnt[W] = base;
    if (h == 0 && kind == 0 && threadIdx.x == 0) {  // cu_seq_lens of the one sequence
        p.cu[0] = 0;
        p.cu[1] = p.seq_len;
    }
}

}  // namespace

cudaError_t launch_minference_pattern(const MinferenceParams &p, int dtype, cudaStream_t stream) {
    if (dtype != PKV_BF16 || p.head_dim % 16 != 0 || p.head_dim > 256)
        return cudaErrorNotSupported;
    const int smem = mi_scores_smem(p.head_dim);
    dim3 grid(p.num_blocks, p.num_qo_heads);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(mi_scores_kernel<1>), smem);
    if (e != cudaSuccess) return e;
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(mi_scores_kernel<2>), smem);
    if (e != cudaSuccess) return e;
    mi_scores_kernel<1><<<grid, kScoreThreads, smem, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mi_lse_kernel<<<p.num_qo_heads, kLastQ, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mi_scores_kernel<2><<<grid, kScoreThreads, smem, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mi_slash_kernel<<<dim3((p.seq_len + 255) / 256, p.num_qo_heads), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mi_topk_kernel<<<dim3(p.num_qo_heads, 2), kTopkThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mi_bitmap_kernel<<<dim3(p.num_qo_heads, 2), kTopkThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
