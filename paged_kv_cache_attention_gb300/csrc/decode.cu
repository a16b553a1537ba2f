// decode.cu -- split-KV paged decode.
//
// One query token per sequence attends to positions 0..L-1 of its paged K/V
// (transformers docs "paged_attention", decode path: block_table and
// cache_seqlens).  The sequence is cut into fixed partitions of P tokens
// aligned to absolute positions (vLLM attention.py: _PARTITION_SIZE = 512 and
// the paged_attention_v2 split), each partition is reduced to a normalised
// partial output and a log-sum-exp, and a second kernel merges the partitions
// and adds the per-head sink to the denominator (FlashInfer
// sink_attention_reference.py, sink_softmax: the sink is one extra softmax
// column whose value row is zero).
//
// GB300 design (bf16): one CTA per (kv head, partition, sequence), heads
// fastest in launch order so the CTAs reading one page run side by side; the
// G query heads of a kv head share every K/V byte fetched from HBM.  Each of
// the 2 warps owns every other page of the partition and streams it through a
// private 2-stage ring of shared-memory stages filled by TMA (one 3-D tiled box per
// 64-dim half of a page, 128-byte swizzle, evict-first L2 policy).  The dot
// products run on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32
// accumulate): S = Q K^T with the (zero-padded) query heads as the 16 rows,
// then O^T += V^T P^T, whose B fragment is exactly the C fragment of S, so P
// never leaves registers.  The online softmax works in log2 units with the
// scale folded in.  fp32 caches take a CUDA-core kernel: per token a
// warp-shuffle dot product per head.
#include <cfloat>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

// Small CTAs (2 warps, 2 stages of K+V per warp, ~38 KB of shared memory)
// let 5-6 CTAs share an SM, so one CTA's start-up latency is covered by the
// others' streaming; measured on GB300 this beat 4- and 8-warp CTAs and deeper
// per-warp rings.
constexpr int kDecWarps = 2;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kMaxGroup = 16;
constexpr int kMaxPartition = 16384;
constexpr float kNegInf = -INFINITY;

__device__ __forceinline__ int clipped_seqlen(const DecodeParams &p, int b, int block_size,
                                              bool report) {
    int L = p.seqlens[b];
    const long long cap_blocks = (long long)p.max_blocks_per_seq * block_size;
    int cap = p.max_seqlen;
    if (cap_blocks < cap) cap = (int)cap_blocks;
    if (L < 0) {
        if (report) flag_error(p.dev_error, PKV_DEVERR_SEQLEN);
        L = 0;
    }
    if (L > cap) {
        if (report) flag_error(p.dev_error, PKV_DEVERR_SEQLEN);
        L = cap;
    }
    return L;
}

// First attended position: the window keeps keys j >= L - 1 - window_left.
__device__ __forceinline__ int window_start(int L, int window_left) {
    if (window_left < 0) return 0;
    const int s = L - 1 - window_left;
    return s > 0 ? s : 0;
}

// The partition a CTA of the partition grid (x = kv head, y = partition
// slot, z = sequence) takes, and its token range [tok_lo, tok_hi).  Sequence
// b has n_b partitions (absolute P-aligned blocks meeting [start, L)); slot z
// takes the z-th of them.  (Measured on GB300: this sequence-major order beat
// a partition-major order and one that launched every sequence's partial
// last partition at the end.)  Returns false for an unused slot.
__device__ __forceinline__ bool decode_partition(const DecodeParams &p, int b, int z,
                                                 int block_size, bool report, int &L,
                                                 int &pidx, int &tok_lo, int &tok_hi) {
    L = clipped_seqlen(p, b, block_size, report);
    tok_lo = tok_hi = 0;
    const int start = window_start(L, p.window_left);
    const int P = p.partition_size;
    const int n = L > 0 ? (L - 1) / P - start / P + 1 : 0;
    pidx = z;
    if (pidx >= n) return false;
    const int part = start / P + pidx;
    tok_lo = max(part * P, start);
    tok_hi = min((part + 1) * P, L);
    return tok_lo < tok_hi;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023);
    return reinterpret_cast<uint8_t *>(a);
}

__device__ __forceinline__ uint32_t ld_b32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// Combine the per-warp softmax states of one CTA and write the partition's
// normalised output and log-sum-exp (log2 units).  s_o holds the warps'
// O accumulators already rescaled to the common maximum.
__device__ __forceinline__ void write_partition_rows(const DecodeParams &p, int b, int g,
                                                     int pidx, int D, int Ds, const float *s_m,
                                                     const float *s_l, const float *s_o) {
    const int G = p.group;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D, d = i - h * D;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w * kMaxGroup + h]);
        float Ls = 0.f;
        if (M != kNegInf) {
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w)
                Ls += exp2f(s_m[w * kMaxGroup + h] - M) * s_l[w * kMaxGroup + h];
        }
        const int hq = g * G + h;
        const int64_t idx = ((int64_t)b * p.num_qo_heads + hq) * p.num_parts + pidx;
        p.part_o[idx * D + d] = Ls > 0.f ? s_o[h * Ds + d] / Ls : 0.f;
        if (d == 0) p.part_lse[idx] = Ls > 0.f ? M + log2f(Ls) : kNegInf;
    }
}

// D: the head size (row stride of part_o); Ds: the row stride of s_o (D
// padded to the kernel's tile width).
template <int Ds>
__device__ __forceinline__ void write_partition(const DecodeParams &p, int b, int g, int pidx,
                                                int D, const float *s_m, const float *s_l,
                                                const float *s_o) {
    if (D == Ds)  // the usual case: divide by a compile-time width
        write_partition_rows(p, b, g, pidx, Ds, Ds, s_m, s_l, s_o);
    else
        write_partition_rows(p, b, g, pidx, D, Ds, s_m, s_l, s_o);
}

// ---------------------------------------------------------------------------
// bf16: TMA-fed tensor-core partition kernel
// ---------------------------------------------------------------------------
template <int D, int BS, int NHT, int NST>
struct DecTC {
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = BS * 128;            // one 64-dim half of a page
    static constexpr int PAGE_BYTES = HALVES * HALF_BYTES;  // one (page, kv head) of K or V
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;      // K + V
    static constexpr int RING_BYTES = kDecWarps * NST * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_BYTES;
    static constexpr int M_OFF = BAR_OFF + kDecWarps * NST * 8;
    static constexpr int L_OFF = M_OFF + kDecWarps * kMaxGroup * 4;
    static constexpr int BLK_OFF = L_OFF + kDecWarps * kMaxGroup * 4;
    // the block ids of one partition (partition_size / BS entries) follow,
    // sized at launch: with 512-token partitions a CTA needs ~34 KB and six
    // fit on an SM (five when the array was sized for the largest partition;
    // measured on GB300, six take the B64 batch from 0.110 to 0.106 ms and
    // the mixed step's decode from 0.486 to 0.472 ms)
    static constexpr int SMEM_FIXED = 1024 + BLK_OFF;
    static_assert(kMaxGroup * D * 4 <= RING_BYTES, "merge scratch must fit in the ring");
};

template <int D, int BS, int NHT, int NST, bool HND>
__global__ void __launch_bounds__(kDecThreads)
decode_bf16_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    using C = DecTC<D, BS, NHT, NST>;
    constexpr int NT = BS / 8;   // 8-token column tiles of S per page
    constexpr int KS = BS / 16;  // 16-token k-steps of PV per page
    constexpr int DK = D / 16;   // 16-dim k-steps of QK / m-tiles of PV

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    int *s_blk = reinterpret_cast<int *>(smem + C::BLK_OFF);
    float *s_m = reinterpret_cast<float *>(smem + C::M_OFF);
    float *s_l = reinterpret_cast<float *>(smem + C::L_OFF);

    // grid: x = kv head (fastest, so the heads reading one page run together),
    // y = partition slot, z = sequence (decode_partition)
    pdl_trigger();  // the merge kernel may launch once every CTA has started
    pdl_wait();     // the previous kernel on the stream (a cache write) has finished
    const int b = blockIdx.z, g = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L, pidx, tok_lo, tok_hi;
    if (!decode_partition(p, b, blockIdx.y, BS, blockIdx.y == 0 && g == 0 && threadIdx.x == 0,
                          L, pidx, tok_lo, tok_hi))
        return;  // this slot holds no attended key
    const int pg_lo = tok_lo / BS;
    const int npages = (tok_hi - 1) / BS - pg_lo + 1;

    const uint32_t ring = smem_u32(smem);
    const uint32_t bars = ring + C::BAR_OFF;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecWarps * NST; ++i) mbar_init(bars + 8 * i, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks_per_seq + pg_lo;
    for (int i = threadIdx.x; i < npages; i += kDecThreads) {
        int id = bt[i];
        if (id < 0 || id >= p.num_blocks) {
            flag_error(p.dev_error, PKV_DEVERR_BLOCK_ID);
            id = -1;
        }
        s_blk[i] = id;
    }
    __syncthreads();

    // pages of this warp: i = warp + j * kDecWarps
    const int nmine = npages > warp ? (npages - warp + kDecWarps - 1) / kDecWarps : 0;
    const uint32_t wring = ring + warp * NST * C::STAGE_BYTES;
    const uint32_t wbars = bars + warp * NST * 8;
    const uint64_t policy = l2_policy_evict_first();

    auto issue = [&](int j) {
        const int i = warp + j * kDecWarps;
        const int s = j % NST;
        const uint32_t bar = wbars + 8 * s;
        const int blk = s_blk[i];
        if (blk < 0) {  // invalid page: complete the phase without data
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
        const uint32_t dst = wring + s * C::STAGE_BYTES;
        // box coordinates of (page, kv head): NHD (x, head, page * BS), HND
        // (x, 0, page * Hkv + head)
        const int cy = HND ? 0 : g;
        const int cz = HND ? blk * p.num_kv_heads + g : blk * BS;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
            tma_load_3d_hint(dst + h * C::HALF_BYTES, &tmk, bar, h * 64, cy, cz, policy);
            tma_load_3d_hint(dst + C::PAGE_BYTES + h * C::HALF_BYTES, &tmv, bar, h * 64, cy, cz,
                             policy);
        }
    };
    if (lane == 0)
        for (int j = 0; j < NST && j < nmine; ++j) issue(j);

    // Q as the A operand (rows = query heads of this kv head, zero-padded to 16)
    const int gq = lane >> 2, tq = lane & 3;
    const int G = p.group;
    // D is the tile width; the head size Dh <= D is a multiple of 16, so a
    // 16-dim k-step lies wholly inside or wholly past it (past it: zeros,
    // matching the zero-filled columns the TMA boxes bring beyond Dh)
    const int Dh = p.head_dim;
    const __nv_bfloat16 *qb =
        static_cast<const __nv_bfloat16 *>(p.q) + ((int64_t)b * p.num_qo_heads + g * G) * Dh;
    uint32_t qa[DK][4];
#pragma unroll
    for (int kk = 0; kk < DK; ++kk) {
        const int d0 = kk * 16 + 2 * tq;
        const bool in = kk * 16 < Dh;
        const bool h0 = in && gq < G, h1 = in && (NHT > 1) && (gq + 8 < G);
        qa[kk][0] = h0 ? ld_b32(qb + gq * Dh + d0) : 0u;
        qa[kk][1] = h1 ? ld_b32(qb + (gq + 8) * Dh + d0) : 0u;
        qa[kk][2] = h0 ? ld_b32(qb + gq * Dh + d0 + 8) : 0u;
        qa[kk][3] = h1 ? ld_b32(qb + (gq + 8) * Dh + d0 + 8) : 0u;
    }

    float oacc[NHT][DK][4];
#pragma unroll
    for (int ht = 0; ht < NHT; ++ht)
#pragma unroll
        for (int mt = 0; mt < DK; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[ht][mt][e] = 0.f;
    float m_run[NHT], l_run[NHT], al2[NHT];
    bool head_ok[NHT];
#pragma unroll
    for (int ht = 0; ht < NHT; ++ht) {
        m_run[ht] = kNegInf;
        l_run[ht] = 0.f;
        head_ok[ht] = ht * 8 + gq < G;
        // ALiBi slope of this lane's head row, in log2 units (0: no bias)
        al2[ht] = (p.alibi && head_ok[ht]) ? p.alibi[g * G + ht * 8 + gq] * kLog2e : 0.f;
    }
    const int qpos = L - 1;  // the decode query's position

    int consumed = 0;
    for (int j = 0; j < nmine; ++j) {
        const int i = warp + j * kDecWarps;
        const int s = j % NST;
        if (!warp_wait_bounded(wbars + 8 * s, (j / NST) & 1, p.dev_error)) break;
        consumed = j + 1;
        const int blk = s_blk[i];
        if (blk >= 0) {
            const uint32_t kb = wring + s * C::STAGE_BYTES;
            const uint32_t vb = kb + C::PAGE_BYTES;
            const int tok0 = (pg_lo + i) * BS;
            // Rows outside [tok_lo, tok_hi) of a boundary page may hold any
            // bits; zero their V rows so a zero probability never meets a
            // non-finite value in the PV product.
            if (tok0 < tok_lo || tok0 + BS > tok_hi) {
                for (int e = lane; e < C::HALVES * BS * 8; e += 32) {
                    const int h = e / (BS * 8);
                    const int r = (e / 8) % BS;
                    const int c = e % 8;
                    const int tok = tok0 + r;
                    if (tok < tok_lo || tok >= tok_hi)
                        st_shared_zero16(vb + h * C::HALF_BYTES + sw128(r, c));
                }
                __syncwarp();
            }
            // S = Q K^T  (rows: heads; columns: 8 tokens per tile)
            float sacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
                for (int kp = 0; kp < D / 32; ++kp) {
                    const int c = kp * 4 + (lane >> 3);
                    const int r = nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + (c >> 3) * C::HALF_BYTES + sw128(r, c & 7), b0, b1, b2, b3);
                    mma_bf16_16816(sacc[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2],
                                   qa[2 * kp][3], b0, b1);
                    mma_bf16_16816(sacc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1],
                                   qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
                }
            }
            // online softmax (log2 units), one head row per lane quad
#pragma unroll
            for (int ht = 0; ht < NHT; ++ht) {
                float mx = kNegInf;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tok0 + nt * 8 + 2 * tq + e;
                        const bool ok = head_ok[ht] && tok >= tok_lo && tok < tok_hi;
                        const float sv =
                            ok ? fmaf(sacc[nt][2 * ht + e], p.scale_log2,
                                      al2[ht] * (float)(tok - qpos))
                               : kNegInf;
                        sacc[nt][2 * ht + e] = sv;
                        mx = fmaxf(mx, sv);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[ht], mx);
                const float msub = m_new == kNegInf ? 0.f : m_new;
                const float alpha = fast_exp2(m_run[ht] - msub);
                float psum = 0.f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = fast_exp2(sacc[nt][2 * ht + e] - msub);
                        sacc[nt][2 * ht + e] = pv;
                        psum += pv;
                    }
                l_run[ht] = l_run[ht] * alpha + psum;
                m_run[ht] = m_new;
                // O^T columns of this lane are heads ht*8 + 2tq and +1
                const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * tq);
                const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);
#pragma unroll
                for (int mt = 0; mt < DK; ++mt) {
                    oacc[ht][mt][0] *= a0;
                    oacc[ht][mt][1] *= a1;
                    oacc[ht][mt][2] *= a0;
                    oacc[ht][mt][3] *= a1;
                }
            }
            // O^T += V^T P^T
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t pb0[NHT], pb1[NHT];
#pragma unroll
                for (int ht = 0; ht < NHT; ++ht) {
                    pb0[ht] = pack_bf16(sacc[2 * ks][2 * ht], sacc[2 * ks][2 * ht + 1]);
                    pb1[ht] = pack_bf16(sacc[2 * ks + 1][2 * ht], sacc[2 * ks + 1][2 * ht + 1]);
                }
                const int jm = lane >> 3;
                const int r = ks * 16 + ((jm >> 1) << 3) + (lane & 7);
#pragma unroll
                for (int mt = 0; mt < DK; ++mt) {
                    const int c = mt * 2 + (jm & 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb + (c >> 3) * C::HALF_BYTES + sw128(r, c & 7), a0, a1, a2, a3);
#pragma unroll
                    for (int ht = 0; ht < NHT; ++ht)
                        mma_bf16_16816(oacc[ht][mt], a0, a1, a2, a3, pb0[ht], pb1[ht]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && j + NST < nmine) {
            fence_proxy_async_smem();
            issue(j + NST);
        }
    }
    // After a timed-out wait, give the copies still in flight a bounded
    // chance to land before the shared memory is reused.
    if (consumed < nmine) {
        const int last = min(nmine, consumed + NST);
        for (int j = consumed + 1; j < last; ++j)
            mbar_wait_bounded(wbars + 8 * (j % NST), (j / NST) & 1, p.dev_error);
    }

#pragma unroll
    for (int ht = 0; ht < NHT; ++ht) {
        l_run[ht] += __shfl_xor_sync(0xffffffffu, l_run[ht], 1);
        l_run[ht] += __shfl_xor_sync(0xffffffffu, l_run[ht], 2);
    }
    __syncthreads();  // every warp is done with the ring: reuse it for the merge
    float *s_o = reinterpret_cast<float *>(smem);
    if (tq == 0) {
#pragma unroll
        for (int ht = 0; ht < NHT; ++ht) {
            s_m[warp * kMaxGroup + ht * 8 + gq] = m_run[ht];
            s_l[warp * kMaxGroup + ht * 8 + gq] = l_run[ht];
        }
    }
    if (NHT == 1) {  // heads 8..15 are absent
        if (lane < 8) {
            s_m[warp * kMaxGroup + 8 + lane] = kNegInf;
            s_l[warp * kMaxGroup + 8 + lane] = 0.f;
        }
    }
    for (int i = threadIdx.x; i < kMaxGroup * D; i += kDecThreads) s_o[i] = 0.f;
    __syncthreads();
#pragma unroll
    for (int ht = 0; ht < NHT; ++ht) {
        const int hc0 = ht * 8 + 2 * tq, hc1 = hc0 + 1;
        float M0 = kNegInf, M1 = kNegInf;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            M0 = fmaxf(M0, s_m[w * kMaxGroup + hc0]);
            M1 = fmaxf(M1, s_m[w * kMaxGroup + hc1]);
        }
        const float f0 = M0 == kNegInf ? 0.f : exp2f(s_m[warp * kMaxGroup + hc0] - M0);
        const float f1 = M1 == kNegInf ? 0.f : exp2f(s_m[warp * kMaxGroup + hc1] - M1);
#pragma unroll
        for (int mt = 0; mt < DK; ++mt) {
            const int d0 = mt * 16 + gq, d1 = d0 + 8;
            if (f0 != 0.f) {
                atomicAdd(&s_o[hc0 * D + d0], oacc[ht][mt][0] * f0);
                atomicAdd(&s_o[hc0 * D + d1], oacc[ht][mt][2] * f0);
            }
            if (f1 != 0.f) {
                atomicAdd(&s_o[hc1 * D + d0], oacc[ht][mt][1] * f1);
                atomicAdd(&s_o[hc1 * D + d1], oacc[ht][mt][3] * f1);
            }
        }
    }
    __syncthreads();
    write_partition<D>(p, b, g, pidx, Dh, s_m, s_l, s_o);
}

// ---------------------------------------------------------------------------
// fp32: CUDA-core partition kernel (warp-shuffle dot products)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kDecThreads)
decode_f32_kernel(const DecodeParams p, int block_size) {
    constexpr int DPL = D / 32;  // dims per lane: lane + 32 * i
    __shared__ float s_m[kDecWarps * kMaxGroup], s_l[kDecWarps * kMaxGroup];
    __shared__ float s_o[kMaxGroup * D];

    pdl_trigger();  // the merge kernel may launch once every CTA has started
    pdl_wait();     // the previous kernel on the stream has finished
    const int b = blockIdx.z, g = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L, pidx, tok_lo, tok_hi;
    if (!decode_partition(p, b, blockIdx.y, block_size,
                          blockIdx.y == 0 && g == 0 && threadIdx.x == 0, L, pidx, tok_lo, tok_hi))
        return;

    const int G = p.group, Hkv = p.num_kv_heads;
    const int Dh = p.head_dim;  // <= D; dims past it are zero in q and skipped in k, v
    const float *qb = static_cast<const float *>(p.q) + ((int64_t)b * p.num_qo_heads + g * G) * Dh;
    float q[kMaxGroup][DPL], o[kMaxGroup][DPL], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        m[h] = kNegInf;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            q[h][i] = (h < G && lane + 32 * i < Dh) ? qb[h * Dh + lane + 32 * i] : 0.f;
            o[h][i] = 0.f;
        }
    }
    const float *kc = static_cast<const float *>(p.k_cache);
    const float *vc = static_cast<const float *>(p.v_cache);
    const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks_per_seq;
    for (int tok = tok_lo + warp; tok < tok_hi; tok += kDecWarps) {
        const int blk = bt[tok / block_size];
        if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0) flag_error(p.dev_error, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        const int64_t base =
            p.hnd ? (((int64_t)blk * Hkv + g) * block_size + tok % block_size) * Dh
                  : (((int64_t)blk * block_size + tok % block_size) * Hkv + g) * Dh;
        float k[DPL], v[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            const bool in = lane + 32 * i < Dh;
            k[i] = in ? kc[base + lane + 32 * i] : 0.f;
            v[i] = in ? vc[base + lane + 32 * i] : 0.f;
        }
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
            if (h >= G) break;
            float part_dot = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) part_dot = fmaf(q[h][i], k[i], part_dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                part_dot += __shfl_xor_sync(0xffffffffu, part_dot, off);
            const float bias = p.alibi ? p.alibi[g * G + h] * kLog2e * (float)(tok - (L - 1)) : 0.f;
            const float s = fmaf(part_dot, p.scale_log2, bias);
            const float m_new = fmaxf(m[h], s);
            const float alpha = exp2f(m[h] - m_new);
            const float pe = exp2f(s - m_new);
            l[h] = l[h] * alpha + pe;
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[h][i] = fmaf(o[h][i], alpha, pe * v[i]);
            m[h] = m_new;
        }
    }
    if (lane < kMaxGroup) {
        float mv = kNegInf, lv = 0.f;
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h == lane) {
                mv = m[h];
                lv = l[h];
            }
        s_m[warp * kMaxGroup + lane] = mv;
        s_l[warp * kMaxGroup + lane] = lv;
    }
    for (int i = threadIdx.x; i < kMaxGroup * D; i += kDecThreads) s_o[i] = 0.f;
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        if (h >= G) break;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w * kMaxGroup + h]);
        const float f = M == kNegInf ? 0.f : exp2f(m[h] - M);
        if (f != 0.f) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) atomicAdd(&s_o[h * D + lane + 32 * i], o[h][i] * f);
        }
    }
    __syncthreads();
    write_partition<D>(p, b, g, pidx, Dh, s_m, s_l, s_o);
}

// ---------------------------------------------------------------------------
// merge of the partitions + sink + cast
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ OutT from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

constexpr int kMergeThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *scratch) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, scratch[w]) : r + scratch[w];
    return r;
}

template <typename OutT>
__global__ void __launch_bounds__(kMergeThreads)
decode_merge_kernel(const DecodeParams p, int D, int block_size) {
    extern __shared__ float s_w[];  // [num_parts] partition weights
    __shared__ float scratch[kMergeThreads / 32];
    pdl_wait();  // the partition kernel's partials
    const int h = blockIdx.x, b = blockIdx.y;
    const int L = clipped_seqlen(p, b, block_size, false);
    const int start = window_start(L, p.window_left);
    const int P = p.partition_size;
    const int n = L > 0 ? (L - 1) / P - start / P + 1 : 0;
    const int64_t base = ((int64_t)b * p.num_qo_heads + h) * p.num_parts;
    const float *lp = p.part_lse + base;
    const float sink_l2 = p.sink ? p.sink[h] * kLog2e : kNegInf;

    float M = sink_l2;
    for (int i = threadIdx.x; i < n; i += kMergeThreads) M = fmaxf(M, lp[i]);
    M = block_reduce(M, true, scratch);
    float sum = 0.f;
    for (int i = threadIdx.x; i < n; i += kMergeThreads) {
        const float w = M == kNegInf ? 0.f : exp2f(lp[i] - M);
        s_w[i] = w;
        sum += w;
    }
    sum = block_reduce(sum, false, scratch);
    const float lam = sum + (M == kNegInf ? 0.f : exp2f(sink_l2 - M));
    __syncthreads();
    // Weighted sum over the partitions: thread (r, c) accumulates a 4-wide
    // column slice c of partition rows r, r + R, r + 2R, ... (coalesced 16-byte
    // loads, R partition rows in flight per pass); the R partial rows are
    // then added in shared memory.
    OutT *out = static_cast<OutT *>(p.out) + ((int64_t)b * p.num_qo_heads + h) * D;
    const float *po = p.part_o + base * D;
    const int cols = D / 4;                  // float4 slices per row
    const int R = kMergeThreads / cols;      // partition rows per pass
    const int c = threadIdx.x % cols, r = threadIdx.x / cols;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lam > 0.f) {
        int i = r;
        for (; i + R < n; i += 2 * R) {  // two rows in flight per thread
            const float w0 = s_w[i], w1 = s_w[i + R];
            const float4 v0 = *reinterpret_cast<const float4 *>(po + (int64_t)i * D + 4 * c);
            const float4 v1 = *reinterpret_cast<const float4 *>(po + (int64_t)(i + R) * D + 4 * c);
            if (w0 != 0.f) {
                acc.x = fmaf(w0, v0.x, acc.x); acc.y = fmaf(w0, v0.y, acc.y);
                acc.z = fmaf(w0, v0.z, acc.z); acc.w = fmaf(w0, v0.w, acc.w);
            }
            if (w1 != 0.f) {
                acc.x = fmaf(w1, v1.x, acc.x); acc.y = fmaf(w1, v1.y, acc.y);
                acc.z = fmaf(w1, v1.z, acc.z); acc.w = fmaf(w1, v1.w, acc.w);
            }
        }
        if (i < n) {
            const float w0 = s_w[i];
            const float4 v0 = *reinterpret_cast<const float4 *>(po + (int64_t)i * D + 4 * c);
            if (w0 != 0.f) {
                acc.x = fmaf(w0, v0.x, acc.x); acc.y = fmaf(w0, v0.y, acc.y);
                acc.z = fmaf(w0, v0.z, acc.z); acc.w = fmaf(w0, v0.w, acc.w);
            }
        }
    }
    __shared__ float4 s_acc[kMergeThreads];
    s_acc[threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.x < cols) {
        float4 t = s_acc[threadIdx.x];
        for (int k = 1; k < R; ++k) {
            const float4 u = s_acc[k * cols + threadIdx.x];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float inv = lam > 0.f ? 1.f / lam : 0.f;
        out[4 * threadIdx.x + 0] = from_f32<OutT>(t.x * inv);
        out[4 * threadIdx.x + 1] = from_f32<OutT>(t.y * inv);
        out[4 * threadIdx.x + 2] = from_f32<OutT>(t.z * inv);
        out[4 * threadIdx.x + 3] = from_f32<OutT>(t.w * inv);
    }
    if (p.lse_out && threadIdx.x == 0) {
        float lse;
        if (lam > 0.f)
            lse = (M + log2f(lam)) * kLn2;
        else
            lse = p.sink ? p.sink[h] : kNegInf;
        p.lse_out[(int64_t)b * p.num_qo_heads + h] = lse;
    }
}

// Merge with one warp per (sequence, query head), for batches with many
// heads and few partitions each (short sequences): no block-wide barriers.
// Lane l owns the columns [l * D/32, (l+1) * D/32); partition weights are
// computed 32 at a time, one per lane, and broadcast with shuffles.
template <typename OutT, int D>
__global__ void __launch_bounds__(kMergeThreads)
decode_merge_warp_kernel(const DecodeParams p, int block_size) {
    constexpr int VEC = D / 32;  // columns per lane: 2, 4 or 8
    pdl_wait();  // the partition kernel's partials
    const int lane = threadIdx.x & 31;
    const int64_t unit = (int64_t)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
    if (unit >= (int64_t)p.batch * p.num_qo_heads) return;
    const int b = (int)(unit / p.num_qo_heads), h = (int)(unit % p.num_qo_heads);
    const int L = clipped_seqlen(p, b, block_size, false);
    const int start = window_start(L, p.window_left);
    const int P = p.partition_size;
    const int n = L > 0 ? (L - 1) / P - start / P + 1 : 0;
    const int64_t base = ((int64_t)b * p.num_qo_heads + h) * p.num_parts;
    const float *lp = p.part_lse + base;
    const float sink_l2 = p.sink ? p.sink[h] * kLog2e : kNegInf;

    float M = sink_l2;
    for (int i = lane; i < n; i += 32) M = fmaxf(M, lp[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float sum = 0.f;
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    const float *po = p.part_o + base * D + lane * VEC;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const float w_mine = (M == kNegInf || c0 + lane >= n) ? 0.f : exp2f(lp[c0 + lane] - M);
        sum += w_mine;
        const int cnt = min(32, n - c0);
        for (int k = 0; k < cnt; ++k) {
            const float w = __shfl_sync(0xffffffffu, w_mine, k);
            const float *row = po + (int64_t)(c0 + k) * D;
            if constexpr (VEC == 8) {
                const float4 v4 = *reinterpret_cast<const float4 *>(row);
                const float4 u4 = *reinterpret_cast<const float4 *>(row + 4);
                acc[0] = fmaf(w, v4.x, acc[0]);
                acc[1] = fmaf(w, v4.y, acc[1]);
                acc[2] = fmaf(w, v4.z, acc[2]);
                acc[3] = fmaf(w, v4.w, acc[3]);
                acc[4] = fmaf(w, u4.x, acc[4]);
                acc[5] = fmaf(w, u4.y, acc[5]);
                acc[6] = fmaf(w, u4.z, acc[6]);
                acc[7] = fmaf(w, u4.w, acc[7]);
            } else if constexpr (VEC == 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(row);
                acc[0] = fmaf(w, v4.x, acc[0]);
                acc[1] = fmaf(w, v4.y, acc[1]);
                acc[2] = fmaf(w, v4.z, acc[2]);
                acc[3] = fmaf(w, v4.w, acc[3]);
            } else {
                const float2 v2 = *reinterpret_cast<const float2 *>(row);
                acc[0] = fmaf(w, v2.x, acc[0]);
                acc[1] = fmaf(w, v2.y, acc[1]);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lam = sum + (M == kNegInf ? 0.f : exp2f(sink_l2 - M));
    const float inv = lam > 0.f ? 1.f / lam : 0.f;
    OutT *out = static_cast<OutT *>(p.out) + ((int64_t)b * p.num_qo_heads + h) * D + lane * VEC;
#pragma unroll
    for (int v = 0; v < VEC; ++v) out[v] = from_f32<OutT>(acc[v] * inv);
    if (p.lse_out && lane == 0) {
        float lse;
        if (lam > 0.f)
            lse = (M + log2f(lam)) * kLn2;
        else
            lse = p.sink ? p.sink[h] : kNegInf;
        p.lse_out[(int64_t)b * p.num_qo_heads + h] = lse;
    }
}

template <typename OutT>
cudaError_t launch_merge(const DecodeParams &p, int D, int BS, cudaStream_t stream) {
    // many heads with few partitions: warp per head; otherwise CTA per head
    const int64_t units = (int64_t)p.batch * p.num_qo_heads;
    if (p.num_parts <= 64 && units >= 8LL * device_sm_count() &&
        (D == 64 || D == 128 || D == 256)) {
        const unsigned blocks = (unsigned)((units + kMergeThreads / 32 - 1) / (kMergeThreads / 32));
        if (D == 64)
            return launch_pdl(decode_merge_warp_kernel<OutT, 64>, dim3(blocks),
                              dim3(kMergeThreads), 0, stream, p, BS);
        if (D == 128)
            return launch_pdl(decode_merge_warp_kernel<OutT, 128>, dim3(blocks),
                              dim3(kMergeThreads), 0, stream, p, BS);
        return launch_pdl(decode_merge_warp_kernel<OutT, 256>, dim3(blocks), dim3(kMergeThreads),
                          0, stream, p, BS);
    }
    const int merge_smem = p.num_parts * (int)sizeof(float);
    auto k = decode_merge_kernel<OutT>;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(k), merge_smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(p.num_qo_heads, p.batch), dim3(kMergeThreads),
                      (size_t)merge_smem, stream, p, D, BS);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return ensure_dynamic_smem(reinterpret_cast<const void *>(kernel), bytes);
}

template <int D, int BS, int NHT, int NST>
cudaError_t launch_tc(const DecodeParams &p, const CUtensorMap *tk, const CUtensorMap *tv,
                      cudaStream_t stream) {
    using C = DecTC<D, BS, NHT, NST>;
    auto kern = p.hnd ? decode_bf16_tc_kernel<D, BS, NHT, NST, true>
                      : decode_bf16_tc_kernel<D, BS, NHT, NST, false>;
    const int smem = C::SMEM_FIXED + (p.partition_size / BS) * 4;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_kv_heads, p.num_parts, p.batch);
    return launch_pdl(kern, grid, dim3(kDecThreads), smem, stream, p, *tk, *tv);
}

template <int D, int BS>
cudaError_t launch_tc_g(const DecodeParams &p, const CUtensorMap *tk, const CUtensorMap *tv,
                        cudaStream_t stream) {
    constexpr int NST = 2;
    if (p.group <= 8) return launch_tc<D, BS, 1, NST>(p, tk, tv, stream);
    return launch_tc<D, BS, 2, NST>(p, tk, tv, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, const pkv_cache_desc &cache,
                          const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                          cudaStream_t stream) {
    // D: the head size; T: the kernel's tile width (D rounded up to 64, 128
    // or 256; the padded dims are zeros and cost no HBM traffic)
    const int D = cache.head_dim, BS = cache.block_size;
    const int T = D <= 64 ? 64 : D <= 128 ? 128 : 256;
    cudaError_t e = cudaSuccess;
    if (p.group > kMaxGroup || p.partition_size > kMaxPartition) return cudaErrorNotSupported;
    if (D % 16 != 0 || D > 256 || p.head_dim != D) return cudaErrorNotSupported;
    if (cache.dtype == PKV_F32) {
        dim3 grid(p.num_kv_heads, p.num_parts, p.batch);
        if (T == 64)
            e = launch_pdl(decode_f32_kernel<64>, grid, dim3(kDecThreads), 0, stream, p, BS);
        else if (T == 128)
            e = launch_pdl(decode_f32_kernel<128>, grid, dim3(kDecThreads), 0, stream, p, BS);
        else
            return cudaErrorNotSupported;
    } else {
        if (T == 64 && BS == 16)
            e = launch_tc_g<64, 16>(p, tmap_k, tmap_v, stream);
        else if (T == 64 && BS == 32)
            e = launch_tc_g<64, 32>(p, tmap_k, tmap_v, stream);
        else if (T == 128 && BS == 16)
            e = launch_tc_g<128, 16>(p, tmap_k, tmap_v, stream);
        else if (T == 128 && BS == 32)
            e = launch_tc_g<128, 32>(p, tmap_k, tmap_v, stream);
        else if (T == 256 && BS == 16)
            e = launch_tc_g<256, 16>(p, tmap_k, tmap_v, stream);
        else if (T == 256 && BS == 32)
            e = launch_tc_g<256, 32>(p, tmap_k, tmap_v, stream);
        else
            return cudaErrorNotSupported;
    }
    if (e != cudaSuccess) return e;
    if (cache.dtype == PKV_F32) return launch_merge<float>(p, D, BS, stream);
    return launch_merge<__nv_bfloat16>(p, D, BS, stream);
}

}  // namespace pkv
