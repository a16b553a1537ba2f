// prefill.cu -- varlen / chunk prefill on the paged pools (or on contiguous
// K/V rows), on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: for request r (q_len queries, kv_len keys addressed by
// cu_seq_lens_q / cu_seq_lens_k, transformers docs "paged_attention", varlen
// path) query row i sits at position kv_len - q_len + i and attends causally
// (and within window_left) to its request's keys, read from the pages named by
// block_table; the per-head sink joins the softmax denominator (FlashInfer
// sink_attention_reference.py, varlen branch and sink_softmax).  Without the
// causal bound a row keeps every key at or after position - window_left (the
// same reference's non-causal varlen mask).  With ALiBi slopes the scaled
// logit of key j gains slope[head] * (j - position) (vLLM attention.py,
// PagedAttentionWithALiBi).  The contiguous form reads request
// r's keys from rows cu_k[r] .. cu_k[r+1]-1 of [total_k, Hkv, D] arrays, as in
// the docs' varlen path.
//
// GB300 design.  One CTA takes NQ = 2 query tiles of 128 rows of one request
// and one kv head.  The G query heads of the kv head are packed into the rows
// (row = token * G + head), so every K/V byte staged in shared memory serves
// 256 query rows.  Warp roles:
//   warp 0      TMA producer: Q tiles once; per 128-key tile one 3-D box per
//               (page, 64-dim half) of K and of V into a 2-stage ring
//               (128-byte swizzle); pages past the end are fetched out of
//               bounds, which fills zeros;
//   warp 1      owns TMEM; one thread issues tcgen05.mma (each group of 8
//               k-steps from one PTX block, descriptors built once):
//                 S_x = Q_x K^T   (A, B K-major in smem, fp32 in TMEM; with
//                                  ALiBi one more k-step adds the bias)
//                 O_x += P_x V    (A = P in TMEM as bf16, B = V MN-major)
//   warps 2-17  softmax, eight per query tile: two per TMEM lane quarter,
//               each owning half of its 32 rows' 128 key columns (thread =
//               row = TMEM lane).  They read S with tcgen05.ld, mask, combine
//               their partial row maxima through shared memory, rescale O in
//               TMEM only when the maximum grows by more than 2^8, write P
//               back to TMEM in place of S, and finally normalise O (sink
//               included) and store it.
// A small single-CTA kernel first builds the work list on the device
// (counting sort by key-tile count, heaviest first).
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"
#include "prefill_common.cuh"

namespace pkv {

namespace {

constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // keys per tile
constexpr int kHeadDim = 128;
constexpr int kNQ = 2;        // query tiles per CTA
constexpr int kStages = 2;    // K and V ring depth
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxSparseTiles = kMaxSparseKeys / kTileN;
static_assert(kTileN / 16 == 8 && kHeadDim / 16 == 8, "MMA groups of 8 k-steps");

struct PfLayout {
    static constexpr int Q_BYTES = kTileM * kHeadDim * 2;   // 32 KB
    static constexpr int T_BYTES = kTileN * kHeadDim * 2;   // 32 KB per K or V tile
    static constexpr int HALF = kTileN * 128;               // one 64-dim half: 16 KB
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + kNQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + kStages * T_BYTES;
    // ALiBi as one more k-step of S = Q K^T: 16-wide K-major blocks without
    // swizzle (8x8 core matrices: 128 bytes between the two k-halves, 256
    // bytes between 8-row groups).  Row r of the Q block holds the head's
    // slope / scale split into three bf16 parts; key row n of the K block holds
    // n (the key's offset in its tile) three times, so the extra k-step adds
    // slope / scale * n to every score.
    static constexpr int AB_BYTES = 128 * 16 * 2;
    static constexpr int OFF_QA = OFF_V + kStages * T_BYTES;
    static constexpr int OFF_KA = OFF_QA + AB_BYTES;
    static constexpr int OFF_BAR = OFF_KA + AB_BYTES;
    // barriers
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + kStages;
    static constexpr int B_VFULL = B_KEMPTY + kStages;
    static constexpr int B_VEMPTY = B_VFULL + kStages;
    static constexpr int B_VFIX = B_VEMPTY + kStages;  // [kStages] tail rows of V zeroed
    static constexpr int B_SFULL = B_VFIX + kStages;
    static constexpr int B_PFULL = B_SFULL + kNQ;
    static constexpr int B_ODONE = B_PFULL + kNQ;
    static constexpr int B_DRAIN = B_ODONE + kNQ;  // the MMAs in flight, after a failed wait
    // a CTA takes work items one after another (persistent form):
    static constexpr int B_QEMPTY = B_DRAIN + 1;   // every S of the item done: Q may be reloaded
    static constexpr int B_OFREE = B_QEMPTY + 1;   // [kNQ] the epilogue has read O_x
    static constexpr int RING = 4;                 // item indices handed from the producer
    static constexpr int B_IFULL = B_OFREE + kNQ;  // [RING] slot written
    static constexpr int B_IEMPTY = B_IFULL + RING;  // [RING] slot read by the MMA thread and
                                                     // the 16 softmax warps
    static constexpr int NBARS = B_IEMPTY + RING;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    // row-max exchange between the two warps sharing a row ([2][kNQ][128][2]
    // floats, double-buffered by key-tile parity) and the row-sum exchange
    // ([2][kNQ][128][2], double-buffered by item parity)
    static constexpr int OFF_XMAX = OFF_TMEM + 16;
    static constexpr int OFF_XL = OFF_XMAX + 2 * kNQ * 128 * 2 * 4;
    static constexpr int OFF_RING = OFF_XL + 2 * kNQ * 128 * 2 * 4;  // [RING] item indices
    // sparse form: the key tiles the item attends ([kMaxSparseTiles] uint16)
    // and their number
    static constexpr int OFF_LIST = OFF_RING + RING * 4;
    static constexpr int OFF_NLIST = OFF_LIST + kMaxSparseTiles * 2;
    // the row pairs' wait status, double-buffered like the maxima
    static constexpr int OFF_XOK = OFF_NLIST + 16;
    static constexpr int SMEM = 1024 + OFF_XOK + 2 * kNQ * 128 * 2 * 4;
    static constexpr int SOFT_WARPS = 8;  // per query tile: 2 per TMEM lane quarter
    static constexpr int THREADS = 64 + kNQ * SOFT_WARPS * 32;
    static constexpr int TMEM_COLS = 512;  // O_0, O_1, S_0, S_1: 128 columns each
};

__host__ __device__ constexpr int o_col(int x) { return x * 128; }
__host__ __device__ constexpr int s_col(int x) { return kNQ * 128 + x * 128; }

using pf::align1024;
using pf::st_shared_zero16;

// Per-CTA geometry of one work item: its request and the key tiles its two
// query tiles attend.
struct Geo : pf::Geo {
    int kt_lo, ntiles;
};

__device__ __forceinline__ Geo make_geo(const PrefillParams &p, int4 item, int block_size,
                                        bool contiguous, bool report) {
    Geo G;
    static_cast<pf::Geo &>(G) = pf::item_geo(p, item, block_size, contiguous, report);
    pf::key_tiles(p, G, G.t0, G.t0 + kNQ * p.rows_per_head, kTileN, G.kt_lo, G.ntiles);
    return G;
}

// ---------------------------------------------------------------------------
// work list: items {request, first query token, kv head, cost}: requests by
// the cost (key tiles) of their heaviest query block, heaviest first, and
// inside a request its query blocks by cost, heaviest first (the persistent
// CTAs draw the items in this order, so the cheap ones come last).  Single
// CTA.
// ---------------------------------------------------------------------------
constexpr int kSchedThreads = 1024;
constexpr int kBuckets = 1024;

__device__ __forceinline__ int item_cost(const PrefillParams &p, int q_len, int kv_len, int t0) {
    const int tokens = kNQ * p.rows_per_head;
    const int t_end = min(t0 + tokens, q_len);
    const int qpos_min = kv_len - q_len + t0;
    const int hi = p.causal ? min(kv_len, kv_len - q_len + t_end) : kv_len;
    int lo = 0;
    if (p.window_left >= 0) lo = max(0, qpos_min - p.window_left);
    if (hi <= lo) return 0;
    return (hi - 1) / kTileN - lo / kTileN + 1;
}

__global__ void __launch_bounds__(kSchedThreads) prefill_schedule_kernel(const PrefillParams p) {
    __shared__ int hist[kBuckets];
    __shared__ int wsum[kSchedThreads / 32];
    __shared__ int total_pairs_s;
    int *count = p.tiles;                                      // [0]: number of items
    int4 *items = reinterpret_cast<int4 *>(p.tiles + 64);      // 256-byte header
    int *offs = p.tiles + 64 + 4 * p.max_tiles;                // [batch + 1] pair offsets,
                                                               // then [batch] first items
    const int tid = threadIdx.x;
    const int tokens = kNQ * p.rows_per_head;
    pdl_trigger();  // the attention kernel (launched as a dependent) may start launching
    pdl_wait();     // the previous kernel on the stream has finished
    if (tid == 0) {
        *pf::abort_word(p) = 0;    // the attention launch's abort word
        *pf::item_counter(p) = 0;  // items drawn by persistent attention CTAs
    }

    // 1. pairs (request, q block) per request, exclusive prefix sum
    int carry = 0;
    for (int base = 0; base < p.batch; base += kSchedThreads) {
        const int r = base + tid;
        int n = 0;
        if (r < p.batch) {
            // the one place that sees every request: report its bad offsets
            int qs, ql;
            pf::q_rows(p, r, qs, ql, true);
            n = (ql + tokens - 1) / tokens;
        }
        // block scan
        int v = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, v, off);
            if ((tid & 31) >= off) v += o;
        }
        if ((tid & 31) == 31) wsum[tid >> 5] = v;
        __syncthreads();
        if (tid < 32) {
            int w = tid < kSchedThreads / 32 ? wsum[tid] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, w, off);
                if (tid >= off) w += o;
            }
            if (tid < kSchedThreads / 32) wsum[tid] = w;
        }
        __syncthreads();
        const int excl = carry + v - n + ((tid >> 5) ? wsum[(tid >> 5) - 1] : 0);
        if (r < p.batch) offs[r] = excl;
        const int block_total = wsum[kSchedThreads / 32 - 1];
        __syncthreads();
        carry += block_total;
    }
    if (tid == 0) {
        offs[p.batch] = carry;
        total_pairs_s = carry;
    }
    for (int i = tid; i < kBuckets; i += kSchedThreads) hist[i] = 0;
    __syncthreads();
    const int total_pairs = total_pairs_s;
    const int n_items = min(total_pairs * p.num_kv_heads, p.max_tiles);

    // locate the request of pair i by binary search over offs
    auto pair_of = [&](int i, int &r, int &t0, int &cost) {
        int lo = 0, hi = p.batch;  // offs[lo] <= i < offs[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (offs[mid] <= i) lo = mid; else hi = mid;
        }
        r = lo;
        t0 = (i - offs[r]) * tokens;
        int qs, ql;
        pf::q_rows(p, r, qs, ql, false);
        const int kl = pf::clip_len64((long long)p.cu_k[r + 1] - p.cu_k[r], p.max_seqlen_k,
                                      nullptr, false);
        cost = min(item_cost(p, ql, kl, t0), kBuckets - 1);
    };

    // The heaviest query block of request r (causal: the last one; with a
    // window all are about equal, so the first is checked too).
    auto request_cost = [&](int r) {
        const int nq = offs[r + 1] - offs[r];
        int qs, ql;
        pf::q_rows(p, r, qs, ql, false);
        const int kl = pf::clip_len64((long long)p.cu_k[r + 1] - p.cu_k[r], p.max_seqlen_k,
                                      nullptr, false);
        const int c = max(item_cost(p, ql, kl, 0), item_cost(p, ql, kl, (nq - 1) * tokens));
        return min(c, kBuckets - 1);
    };
    // 2. histogram of request costs (each request yields its blocks x
    //    num_kv_heads items)
    for (int r = tid; r < p.batch; r += kSchedThreads) {
        const int nq = offs[r + 1] - offs[r];
        if (nq > 0) atomicAdd(&hist[request_cost(r)], nq * p.num_kv_heads);
    }
    __syncthreads();
    // 3. exclusive scan from the heaviest bucket down: thread t takes bucket
    //    kBuckets - 1 - t (warp scans, then a scan of the warp totals)
    {
        static_assert(kBuckets == kSchedThreads, "one bucket per thread");
        const int bk = kBuckets - 1 - tid, lane = tid & 31, wid = tid >> 5;
        const int h = hist[bk];
        int v = h;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
        }
        if (lane == 31) wsum[wid] = v;
        __syncthreads();
        if (tid < 32) {
            int w = wsum[tid];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, w, off);
                if (tid >= off) w += o;
            }
            wsum[tid] = w;
        }
        __syncthreads();
        hist[bk] = v - h + (wid ? wsum[wid - 1] : 0);
    }
    __syncthreads();
    // 4. requests in order of their heaviest block, heaviest first; inside a
    //    request its query blocks from the heaviest down, each with its kv
    //    heads side by side.  The CTAs running at one time then work on one
    //    or two requests, whose K/V stays in L2 while all their query blocks
    //    read it.  On the 4 x 2048-token prefill of the mixed step (235 MB
    //    of algorithmic bytes) the launch moves 221 MB through DRAM this way,
    //    against 755 MB with the items ordered by their own cost across all
    //    requests (measured on GB300).
    int *first = offs + p.batch + 1;  // [batch] first item of each request
    for (int r = tid; r < p.batch; r += kSchedThreads) {
        const int nq = offs[r + 1] - offs[r];
        first[r] = nq > 0 ? atomicAdd(&hist[request_cost(r)], nq * p.num_kv_heads) : 0;
    }
    __syncthreads();
    for (int i = tid; i < total_pairs; i += kSchedThreads) {
        int r, t0, c;
        pair_of(i, r, t0, c);
        const int nq = offs[r + 1] - offs[r], blk = i - offs[r];
        for (int g = 0; g < p.num_kv_heads; ++g) {
            const int pos = first[r] + (nq - 1 - blk) * p.num_kv_heads + g;
            if (pos < p.max_tiles) items[pos] = make_int4(r, t0, g, c);
        }
    }
    if (tid == 0) *count = n_items;
}

// ---------------------------------------------------------------------------
// bitmaps of the sparse form
// ---------------------------------------------------------------------------
// Bits [lo, lo + 64) of a bitmap of `words` 32-bit words (bit j of the map is
// bit j & 31 of word j >> 5); bits outside the map read 0.
__device__ __forceinline__ uint64_t bits64(const uint32_t *bits, int words, int lo) {
    const int w = lo >> 5;  // floor, also for negative lo
    const int off = lo & 31;
    auto word = [&](int i) -> uint64_t {
        return (i >= 0 && i < words) ? (uint64_t)__ldg(bits + i) : 0ull;
    };
    const uint64_t a = word(w) | (word(w + 1) << 32);
    const uint64_t b = word(w + 2);
    return off ? (a >> off) | (b << (64 - off)) : a;
}

// Is any bit of [lo, hi] (inclusive, clipped to the map) set?  cnt[w] is the
// number of set bits in words [0, w).
__device__ __forceinline__ bool bit_range_any(const uint32_t *bits, const int32_t *cnt, int lo,
                                              int hi) {
    if (lo < 0) lo = 0;
    if (hi < lo) return false;
    const int wl = lo >> 5, wh = hi >> 5;
    const uint32_t ml = ~0u << (lo & 31), mh = ~0u >> (31 - (hi & 31));
    if (wl == wh) return (__ldg(bits + wl) & ml & mh) != 0;
    if (__ldg(bits + wl) & ml) return true;
    if (__ldg(bits + wh) & mh) return true;
    return __ldg(cnt + wh) - __ldg(cnt + wl + 1) > 0;
}

// ---------------------------------------------------------------------------
// the attention kernel
// ---------------------------------------------------------------------------
// BS: rows per page of the paged pools; CONTIG: K/V are contiguous rows
// addressed by cu_k (then BS = 128, one box per 64-dim half per tile);
// ALIBI: the logits gain slope[head] * (key - position); HND: paged pools in
// the HND layout; SPARSE: MInference vertical + slash attention of one
// contiguous sequence (key j kept for the row at position i iff j <= i and
// the vertical bitmap of its head has j or the slash bitmap has i - j); key
// tiles holding no kept key of the item's heads are skipped.
template <int BS, bool CONTIG, bool ALIBI, bool HND, bool SPARSE = false>
__global__ void __launch_bounds__(PfLayout::THREADS, 1)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Lay = PfLayout;
    constexpr int NPG = kTileN / BS;  // pages per key tile
    // The dense forms are persistent: a CTA takes work item blockIdx.x, then
    // draws further items from a counter of the work list until none is left,
    // keeping its barriers, tensor memory and shared-memory layout; every
    // barrier's phase carries on from item to item.  The sparse form takes
    // one item per CTA (its per-item list of key tiles is built by the whole
    // CTA before the roles split).
    constexpr bool PERSIST = !SPARSE;
    // items a CTA may take (one: the compiler then sees straight-line code)
    constexpr int kMaxItems = PERSIST ? (1 << 30) : 1;

    pdl_wait();  // the work list: the attention grid launches while it is built
    const int n_items = p.tiles[0];
    if ((int)blockIdx.x >= n_items) return;  // beyond the work list
    const int4 *items = reinterpret_cast<const int4 *>(p.tiles + 64);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + Lay::OFF_Q, sK = sbase + Lay::OFF_K, sV = sbase + Lay::OFF_V;
    const uint32_t sQA = sbase + Lay::OFF_QA, sKA = sbase + Lay::OFF_KA;
    const uint32_t bars = sbase + Lay::OFF_BAR;
    auto bar = [&](int i) { return bars + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_TMEM);
    volatile int *ring = reinterpret_cast<volatile int *>(smem + Lay::OFF_RING);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *const abort = pf::abort_word(p);  // zeroed by the work-list kernel
    const int G = p.group;
    const int TPR = p.rows_per_head;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lay::NBARS; ++i) {
            uint32_t count = 1;
            if ((i >= Lay::B_PFULL && i < Lay::B_PFULL + kNQ) ||
                (i >= Lay::B_OFREE && i < Lay::B_OFREE + kNQ))
                count = Lay::SOFT_WARPS * 32;
            if (i >= Lay::B_IEMPTY && i < Lay::B_IEMPTY + Lay::RING)
                count = 1 + kNQ * Lay::SOFT_WARPS;  // the MMA thread + one per softmax warp
            mbar_init(bar(i), count);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
        tc::tmem_relinquish();
    }
    if constexpr (ALIBI) {
        // the ALiBi k-step's blocks (see PfLayout): element (row r, k) at
        // byte (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
        // The key side holds r for k < 3; the query side's k < 3 entries
        // depend on the item's kv head and are written by the producer per
        // item, the rest stay zero
        for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
            const int r = i >> 4, k = i & 15;
            const int off = (r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
            *reinterpret_cast<__nv_bfloat16 *>(smem + Lay::OFF_KA + off) =
                __float2bfloat16_rn(k < 3 ? (float)r : 0.f);
            *reinterpret_cast<__nv_bfloat16 *>(smem + Lay::OFF_QA + off) = __float2bfloat16_rn(0.f);
        }
        fence_proxy_async_smem();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    uint16_t *s_list = reinterpret_cast<uint16_t *>(smem + Lay::OFF_LIST);
    int *s_nlist = reinterpret_cast<int *>(smem + Lay::OFF_NLIST);
    if constexpr (SPARSE) {
        // the key tiles with at least one kept key for some row of the item
        // (a superset is harmless: every key of a tile is masked per element)
        const Geo geo = make_geo(p, items[blockIdx.x], BS, CONTIG, false);
        if (threadIdx.x == 0) *s_nlist = 0;
        __syncthreads();
        const int t_end = min(geo.t0 + kNQ * p.rows_per_head, geo.q_len);
        const int pos_lo = geo.kv_len - geo.q_len + geo.t0;
        const int pos_hi = geo.kv_len - geo.q_len + t_end - 1;
        for (int jt = threadIdx.x; jt < geo.ntiles; jt += blockDim.x) {
            const int k0 = (geo.kt_lo + jt) * kTileN;
            const int k1 = min(k0 + kTileN - 1, pos_hi);  // causal
            bool need = false;
            for (int hl = 0; hl < G && !need; ++hl) {
                const int head = geo.g * G + hl;
                need = bit_range_any(p.vbits + (int64_t)head * p.bit_words,
                                     p.vcnt + (int64_t)head * (p.bit_words + 1), k0, k1) ||
                       bit_range_any(p.sbits + (int64_t)head * p.bit_words,
                                     p.scnt + (int64_t)head * (p.bit_words + 1),
                                     max(pos_lo - (k0 + kTileN - 1), 0), pos_hi - k0);
            }
            if (need) s_list[jt] = 1; else s_list[jt] = 0;
        }
        __syncthreads();
        if (warp == 0) {  // compact the flags, in order
            int base = 0;
            for (int c0 = 0; c0 < geo.ntiles; c0 += 32) {
                const int jt = c0 + lane;
                const bool f = jt < geo.ntiles && s_list[jt];
                const uint32_t m = __ballot_sync(0xffffffffu, f);
                __syncwarp();
                if (f) s_list[base + __popc(m & ((1u << lane) - 1))] = (uint16_t)jt;
                __syncwarp();
                base += __popc(m);
            }
            if (lane == 0) *s_nlist = base;
        }
        __syncthreads();
    }

    // One work item as every role sees it: its geometry, the key tiles it
    // processes and their order.  Key tiles in processing order (offsets
    // from kt_lo): with ALiBi they run from the query's end backwards (the
    // nearest keys carry the largest bias, so the first tile usually holds
    // the row maximum and its P = 2^0 is exact in bf16); the sparse form runs
    // its list of tiles, also from the end (its rows are dominated by their
    // nearest, slash, keys).
    struct Work {
        Geo geo;
        int ntiles;  // key tiles processed
        bool tail;   // the last key tile runs past kv_len
    };
    auto work_of = [&](int idx, bool report) {
        Work w;
        w.geo = make_geo(p, items[idx], BS, CONTIG, report);
        w.ntiles = SPARSE ? *s_nlist : w.geo.ntiles;
        w.tail = w.geo.ntiles > 0 && (w.geo.kt_lo + w.geo.ntiles) * kTileN > w.geo.kv_len;
        return w;
    };
    auto tile_of = [&](const Work &w, int j) {
        if constexpr (SPARSE) return (int)s_list[w.ntiles - 1 - j];
        return ALIBI ? w.ntiles - 1 - j : j;
    };
    auto is_tail = [&](const Work &w, int j) {
        return w.tail && tile_of(w, j) == w.geo.ntiles - 1;
    };
    // The n-th item of this CTA for the MMA thread and the softmax warps: the
    // producer draws it and hands its index over through a ring of shared
    // slots (-1: none left; -2: a wait gave up).  Each consumer releases the
    // slot once it has read it.  whole_warp: every lane waits and reads.
    auto item_at = [&](int n, bool whole_warp) -> int {
        if constexpr (!PERSIST) return n == 0 ? (int)blockIdx.x : -1;
        const int s = n % Lay::RING;
        const uint32_t par = (uint32_t)(n / Lay::RING) & 1;
        const bool ok = whole_warp ? warp_wait_bounded(bar(Lay::B_IFULL + s), par, p.dev_error, abort)
                                   : mbar_wait_bounded(bar(Lay::B_IFULL + s), par, p.dev_error, abort);
        if (!ok) return -2;
        const int idx = ring[s];
        if (whole_warp) __syncwarp();
        if (!whole_warp || lane == 0) mbar_arrive(bar(Lay::B_IEMPTY + s));
        return idx;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        // box coordinates of (page, kv head): NHD (x, head, page * BS),
        // HND (x, 0, page * Hkv + head); one past the pool reads zeros
        const int oob_row = HND ? (int)(p.num_blocks * p.num_kv_heads) : (int)(p.num_blocks * BS);
        int kt = 0;          // key tiles loaded so far, all items: ring stage kt % 2
        int qn = 0;          // Q loads so far
        int nk = 0, nv = 0;  // key / value tile loads issued (for the drain)
        bool alive = true;
        for (int n = 0; alive && n < kMaxItems; ++n) {
            int idx;
            if constexpr (PERSIST) {
                const int s = n % Lay::RING;
                if (n >= Lay::RING) {  // slot s last held item n - RING
                    alive = warp_wait_bounded(bar(Lay::B_IEMPTY + s),
                                              (uint32_t)(n / Lay::RING - 1) & 1, p.dev_error,
                                              abort);
                    if (!alive) break;
                }
                int drawn = 0;
                if (lane == 0)
                    drawn = n == 0 ? (int)blockIdx.x
                                   : (int)gridDim.x + atomicAdd(pf::item_counter(p), 1);
                idx = __shfl_sync(0xffffffffu, drawn, 0);
                if (idx >= n_items) idx = -1;
                if (lane == 0) {
                    ring[s] = idx;
                    mbar_arrive(bar(Lay::B_IFULL + s));
                }
            } else {
                idx = n == 0 ? (int)blockIdx.x : -1;
            }
            if (idx < 0) break;
            const Work w = work_of(idx, lane == 0);
            const Geo &geo = w.geo;
            if (w.ntiles == 0) continue;
            // Q (and the query side of the ALiBi k-step) may be rewritten
            // once every S product of the previous item is done
            if (qn > 0) {
                alive = warp_wait_bounded(bar(Lay::B_QEMPTY), (uint32_t)(qn - 1) & 1,
                                          p.dev_error, abort);
                if (!alive) break;
            }
            if constexpr (ALIBI) {
                // the query side's k < 3 entries: row r holds the slope of
                // head g * G + r % G divided by the scale, split into three
                // bf16 parts (hi + mid + lo to about 2^-24 relative); the
                // block serves both query tiles.  Lane l < G loads slope l.
                float a = 0.f;
                if (lane < G) a = p.alibi[geo.g * G + lane] * kLog2e / p.scale_log2;
                for (int r = lane; r < 128; r += 32) {
                    const float ar = __shfl_sync(0xffffffffu, a, r % G);
                    const float hi = __bfloat162float(__float2bfloat16_rn(ar));
                    const float mid = __bfloat162float(__float2bfloat16_rn(ar - hi));
                    const float parts[3] = {hi, mid, ar - hi - mid};
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const int off = (r >> 3) * 256 + (r & 7) * 16 + k * 2;
                        *reinterpret_cast<__nv_bfloat16 *>(smem + Lay::OFF_QA + off) =
                            __float2bfloat16_rn(parts[k]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(Lay::B_Q), kNQ * Lay::Q_BYTES);
                for (int x = 0; x < kNQ; ++x)
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sQ + x * Lay::Q_BYTES + h * Lay::HALF, &tmq, bar(Lay::B_Q),
                                    h * 64, geo.g * G, geo.q_start + geo.t0 + x * TPR);
            }
            ++qn;
            const int32_t *bt = p.block_table + (int64_t)geo.r * p.max_blocks_per_seq;
            const int cy = HND ? 0 : geo.g;
            const int pg0 = geo.kt_lo * NPG;       // first page of the item's key range
            const int npages_kv = (geo.kv_len + BS - 1) / BS;
            int ids_batch = -1, ids_row = oob_row;  // lane l: pool row of page pg0 + 32*batch + l
            for (int j = 0; j < w.ntiles && alive; ++j) {
                const int t = kt + j;
                const int s = t & 1;
                const uint32_t ph = (t >> 1) & 1;
                const int key0 = (geo.kt_lo + tile_of(w, j)) * kTileN;
                const int rel = tile_of(w, j) * NPG;
                if (!CONTIG && (rel >> 5) != ids_batch) {  // 32 block ids per warp-wide load
                    ids_batch = rel >> 5;
                    const int pg = pg0 + ids_batch * 32 + lane;
                    ids_row = oob_row;
                    if (pg < npages_kv) {
                        const int blk = bt[pg];
                        if (blk < 0 || blk >= p.num_blocks)
                            flag_error(p.dev_error, PKV_DEVERR_BLOCK_ID);
                        else
                            ids_row = HND ? blk * p.num_kv_heads + geo.g : blk * BS;
                    }
                }
                int row = __shfl_sync(0xffffffffu, ids_row, ((rel & 31) + min(lane >> 1, NPG - 1)) & 31);
                if constexpr (CONTIG) row = p.cu_k[geo.r] + key0;  // rows past kv_len are masked
                // K
                alive = warp_wait_bounded(bar(Lay::B_KEMPTY + s), ph ^ 1, p.dev_error, abort);
                if (!alive) break;
                if (lane == 0) mbar_arrive_expect_tx(bar(Lay::B_KFULL + s), Lay::T_BYTES);
                __syncwarp();
                if (lane < 2 * NPG) {
                    const int pg = lane >> 1, h = lane & 1;
                    tma_load_3d(sK + s * Lay::T_BYTES + h * Lay::HALF + pg * BS * 128, &tmk,
                                bar(Lay::B_KFULL + s), h * 64, cy, row);
                }
                ++nk;
                // V
                alive = warp_wait_bounded(bar(Lay::B_VEMPTY + s), ph ^ 1, p.dev_error, abort);
                if (!alive) break;
                if (lane == 0) mbar_arrive_expect_tx(bar(Lay::B_VFULL + s), Lay::T_BYTES);
                __syncwarp();
                if (lane < 2 * NPG) {
                    const int pg = lane >> 1, h = lane & 1;
                    tma_load_3d(sV + s * Lay::T_BYTES + h * Lay::HALF + pg * BS * 128, &tmv,
                                bar(Lay::B_VFULL + s), h * 64, cy, row);
                }
                ++nv;
                if (is_tail(w, j)) {
                    // rows at or past kv_len of the last value tile may hold any
                    // bits: zero them so P = 0 never meets a non-finite value
                    alive = warp_wait_bounded(bar(Lay::B_VFULL + s), ph, p.dev_error, abort);
                    if (!alive) break;
                    const int first = max(geo.kv_len - key0, 0);
                    const uint32_t vb = sV + s * Lay::T_BYTES;
                    for (int e = first * 16 + lane; e < kTileN * 16; e += 32) {
                        const int rr = e >> 4, c = e & 15;
                        st_shared_zero16(vb + (c >> 3) * Lay::HALF + sw128(rr, c & 7));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(Lay::B_VFIX + s));
                }
            }
            kt += w.ntiles;
        }
        // Let the MMA issuer's last "stage empty" arrivals land before the
        // CTA can exit.
        for (int t = max(0, kt - kStages); t < kt && alive; ++t) {
            const uint32_t ph = (t >> 1) & 1;
            alive = warp_wait_bounded(bar(Lay::B_KEMPTY + (t & 1)), ph, p.dev_error, abort) &&
                    warp_wait_bounded(bar(Lay::B_VEMPTY + (t & 1)), ph, p.dev_error, abort);
        }
        if (!alive) {
            // a wait gave up: let this warp's copies still in flight land
            // (bounded) before the CTA's shared memory is released
            if (qn > 0) warp_wait_bounded(bar(Lay::B_Q), (uint32_t)(qn - 1) & 1, p.dev_error);
            for (int t = max(0, nk - kStages); t < nk; ++t)
                warp_wait_bounded(bar(Lay::B_KFULL + (t & 1)), (t >> 1) & 1, p.dev_error);
            for (int t = max(0, nv - kStages); t < nv; ++t)
                warp_wait_bounded(bar(Lay::B_VFULL + (t & 1)), (t >> 1) & 1, p.dev_error);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Order per key tile j:  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): the next
        // S of a query tile only waits for that tile's own PV (S_x(j+1) is
        // written where P_x(j) lives), not for the other tile's softmax.
        // Across items the same rule holds for the first S of an item (it
        // waits for the previous item's last PV of that tile), and the first
        // PV of an item, which overwrites O_x, waits until the previous item's
        // epilogue has read O_x.
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16_f32(kTileM, kTileN, 0, 0);
            constexpr uint32_t idO = tc::idesc_bf16_f32(kTileM, kHeadDim, 0, 1);
            const int ksteps = p.head_dim / 16;  // k-steps past the head size multiply zeros
            // The issuing thread shares its SM sub-partition with four busy
            // softmax warps, so every instruction it spends per MMA delays
            // the tensor pipe: the descriptors are built once, and per tile,
            // stage and k-step only their start-address field (bytes / 16,
            // bits 0-13, never carrying out) moves by a constant.
            const uint64_t dq0 = tc::smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(sK, 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(sV, Lay::HALF, 1024);
            const uint64_t dqa = tc::smem_desc_noswz(sQA, 128, 256);
            const uint64_t dka = tc::smem_desc_noswz(sKA, 128, 256);
            auto issue_s = [&](int x, int s) {
                const uint64_t dq = dq0 + (uint64_t)((x * Lay::Q_BYTES) >> 4);
                const uint64_t dk = dk0 + (uint64_t)((s * Lay::T_BYTES) >> 4);
                const uint32_t d = tmem + s_col(x);
                auto kstep = [&](int kk) {
                    const uint32_t koff = ((kk >> 2) * Lay::HALF + (kk & 3) * 32) >> 4;
                    tc::mma_ss(d, dq + koff, dk + koff, idS, kk > 0 ? 1u : 0u);
                };
                if (ksteps == kHeadDim / 16) {
                    tc::mma_ss8<Lay::HALF>(d, dq, dk, idS, 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                        if (kk >= ksteps) break;
                        kstep(kk);
                    }
                }
                if constexpr (ALIBI) tc::mma_ss(d, dqa, dka, idS, 1u);
                tc::commit(bar(Lay::B_SFULL + x));
            };
            int kt = 0;       // key tiles consumed so far, all items
            int gstep = 0;    // (key tile, query tile) steps so far: phases of S/P/O barriers
            int qn = 0;       // items with key tiles so far
            int vfn[kStages] = {0, 0};  // tail fixes consumed per stage
            bool alive = true;
            for (int n = 0; alive && n < kMaxItems; ++n) {
                const int idx = item_at(n, false);
                if (idx < 0) {
                    alive = idx == -1;
                    break;
                }
                const Work w = work_of(idx, false);
                if (w.ntiles == 0) continue;
                alive = mbar_wait_bounded(bar(Lay::B_Q), (uint32_t)qn & 1, p.dev_error, abort) &&
                        mbar_wait_bounded(bar(Lay::B_KFULL + (kt & 1)), (kt >> 1) & 1,
                                          p.dev_error, abort);
                if (!alive) break;
                tc::fence_after_sync();
                for (int x = 0; x < kNQ && alive; ++x) {
                    if (gstep > 0) {  // the previous item's last P_x lives where S_x goes
                        alive = mbar_wait_bounded(bar(Lay::B_ODONE + x), (gstep - 1) & 1,
                                                  p.dev_error, abort);
                        tc::fence_after_sync();
                    }
                    if (alive) issue_s(x, kt & 1);
                }
                if (!alive) break;
                tc::commit(bar(Lay::B_KEMPTY + (kt & 1)));
                if (w.ntiles == 1) tc::commit(bar(Lay::B_QEMPTY));
                for (int j = 0; j < w.ntiles && alive; ++j) {
                    const int t = kt + j, g = gstep + j;
                    const int s = t & 1;
                    const uint32_t ph = (t >> 1) & 1;
                    const int sn = (t + 1) & 1;
                    const uint32_t phn = ((t + 1) >> 1) & 1;
                    const bool more = j + 1 < w.ntiles;
                    for (int x = 0; x < kNQ && alive; ++x) {
                        alive = mbar_wait_bounded(bar(Lay::B_PFULL + x), g & 1, p.dev_error, abort);
                        if (!alive) break;
                        tc::fence_after_sync();
                        if (x == 0) {
                            if (is_tail(w, j)) {
                                alive = mbar_wait_bounded(bar(Lay::B_VFIX + s), vfn[s] & 1,
                                                          p.dev_error, abort);
                                ++vfn[s];
                            } else {
                                alive = mbar_wait_bounded(bar(Lay::B_VFULL + s), ph, p.dev_error,
                                                          abort);
                            }
                            if (!alive) break;
                            tc::fence_after_sync();
                        }
                        if (j == 0 && qn > 0) {  // the previous item's epilogue has read O_x
                            alive = mbar_wait_bounded(bar(Lay::B_OFREE + x), (qn - 1) & 1,
                                                      p.dev_error, abort);
                            if (!alive) break;
                            tc::fence_after_sync();
                        }
                        {
                            const uint64_t dv = dv0 + (uint64_t)((s * Lay::T_BYTES) >> 4);
                            const uint32_t dO = tmem + o_col(x), aP = tmem + s_col(x);
                            tc::mma_ts8(dO, aP, dv, idO, j > 0 ? 1u : 0u);
                        }
                        tc::commit(bar(Lay::B_ODONE + x));
                        if (more) {
                            if (x == 0) {
                                alive = mbar_wait_bounded(bar(Lay::B_KFULL + sn), phn, p.dev_error,
                                                          abort);
                                if (!alive) break;
                            }
                            // P_x(j) lives where S_x(j+1) goes: PV_x(j) must be done
                            alive = mbar_wait_bounded(bar(Lay::B_ODONE + x), g & 1, p.dev_error,
                                                      abort);
                            if (!alive) break;
                            tc::fence_after_sync();
                            issue_s(x, sn);
                            if (x == kNQ - 1) {
                                tc::commit(bar(Lay::B_KEMPTY + sn));
                                if (j + 2 == w.ntiles) tc::commit(bar(Lay::B_QEMPTY));
                            }
                        }
                    }
                    if (!alive) break;
                    tc::commit(bar(Lay::B_VEMPTY + s));
                }
                kt += w.ntiles;
                gstep += w.ntiles;
                ++qn;
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Eight warps per query tile.  A warp may only touch the TMEM lane
        // quarter (warp % 4), so each quarter has two warps, and they split
        // every row's 128 key columns: warp half hc owns columns
        // [64 hc, 64 hc + 64) of S, [32 hc, 32 hc + 32) of the packed P and
        // [64 hc, 64 hc + 64) of O.  The two halves of a row exchange their
        // partial maxima (and, at the end, row sums) through shared memory
        // under a 64-thread named barrier.
        const int w = warp - 2;
        const int x = w / Lay::SOFT_WARPS;
        const int quarter = warp & 3;
        const int hc = (w % Lay::SOFT_WARPS) >> 2;
        const int row = quarter * 32 + lane;
        const int tok_local = row / G;
        const int h_local = row - tok_local * G;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + s_col(x) + hc * 64;
        const uint32_t tP = tmem + lane_off + s_col(x) + hc * 32;
        const uint32_t tO = tmem + lane_off + o_col(x) + hc * 64;
        const uint32_t pair_bar = 1 + x * 4 + quarter;
        float *xmax = reinterpret_cast<float *>(smem + Lay::OFF_XMAX);
        float *xl = reinterpret_cast<float *>(smem + Lay::OFF_XL);
        const float sl2 = p.scale_log2;
        const int wl = p.window_left;
        int gstep = 0;  // key-tile steps of this query tile so far, all items
        bool alive = true;
        for (int n = 0; alive && n < kMaxItems; ++n) {
        const int idx = item_at(n, true);
        if (idx < 0) break;
        const Work wk = work_of(idx, false);
        const Geo &geo = wk.geo;
        const int ntiles = wk.ntiles;
        const int tok = geo.t0 + x * TPR + tok_local;
        const bool row_valid = tok < geo.q_len;
        const int qpos = geo.kv_len - geo.q_len + tok;
        const int cpos = p.causal ? qpos : (1 << 30);  // causal upper bound on keys
        const int head = geo.g * G + h_local;
        // ALiBi slope of this row's head in log2 units
        const float al2 = ALIBI ? p.alibi[head] * kLog2e : 0.f;

        float m_run = kNegInf, l_run = 0.f;
        for (int j = 0; j < ntiles; ++j) {
            const int g = gstep + j;
            const int key0 = (geo.kt_lo + tile_of(wk, j)) * kTileN + hc * 64;  // first key of this half
            uint64_t keep = ~0ull;  // sparse form: bit c keeps key key0 + c
            if constexpr (SPARSE) {
                // vertical bits of keys [key0, key0 + 64) and slash bits of the
                // diagonals qpos - key0 - c, c = 0..63 (reversed into key
                // order); loaded before the wait for S so the two overlap
                keep = bits64(p.vbits + (int64_t)head * p.bit_words, p.bit_words, key0) |
                       __brevll(bits64(p.sbits + (int64_t)head * p.bit_words, p.bit_words,
                                       qpos - key0 - 63));
            }
            // a warp whose wait gave up still meets its partner at the pair
            // barrier below, and both leave together
            const bool s_ok = warp_wait_bounded(bar(Lay::B_SFULL + x), g & 1, p.dev_error, abort);
            tc::fence_after_sync();
            const bool full = !SPARSE && (key0 + 63 <= cpos) && (key0 + 64 <= geo.kv_len) &&
                              (wl < 0 || key0 >= qpos - wl);
            // keys this row keeps: [klo, khi] (inclusive), relative to key0
            const int khi = min(cpos, geo.kv_len - 1) - key0;
            const int klo = wl < 0 ? -1 : qpos - wl - key0;
            uint32_t ra[32], rb[32];
            tc::ld_32x32b_x32(tS, ra);
            tc::ld_32x32b_x32(tS + 32, rb);
            tc::wait_ld();
            // ALiBi: the extra k-step of S added slope / scale * (key - kt0),
            // kt0 = the tile's first key; the row's part slope * (kt0 - qpos)
            // joins here (log2 units)
            const float ct = ALIBI ? al2 * (float)(key0 - hc * 64 - qpos) : 0.f;
            auto apply_mask = [&]() {
                if constexpr (SPARSE) {
                    // fold the causal / length range [klo, khi] into the keep bits,
                    // then one bit test per element (none when every key is kept)
                    const int lo = max(klo, 0), hi = min(khi, 63);
                    const uint64_t range = hi < lo ? 0ull
                                                   : ((~0ull) >> (63 - hi)) & ((~0ull) << lo);
                    keep &= range;
                    if (keep != ~0ull) {
                        const uint32_t keep_a = (uint32_t)keep, keep_b = (uint32_t)(keep >> 32);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (!((keep_a >> i) & 1u)) ra[i] = __float_as_uint(kNegInf);
                            if (!((keep_b >> i) & 1u)) rb[i] = __float_as_uint(kNegInf);
                        }
                    }
                } else if (!full) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (!(i <= khi && i >= klo)) ra[i] = __float_as_uint(kNegInf);
                        if (!(i + 32 <= khi && i + 32 >= klo)) rb[i] = __float_as_uint(kNegInf);
                    }
                }
            };
            apply_mask();
            uint64_t ps2[2] = {0ull, 0ull};
            float mine;
            {
                float mx4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    mx4[i & 1] = fmax3(mx4[i & 1], __uint_as_float(ra[2 * i]),
                                       __uint_as_float(ra[2 * i + 1]));
                    mx4[2 + (i & 1)] = fmax3(mx4[2 + (i & 1)], __uint_as_float(rb[2 * i]),
                                             __uint_as_float(rb[2 * i + 1]));
                }
                mine = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            }
            float *slot = xmax + (((g & 1) * kNQ + x) * 128 + row) * 2;
            slot[hc] = mine;
            int *okslot = reinterpret_cast<int *>(smem + Lay::OFF_XOK) +
                          (((g & 1) * kNQ + x) * 128 + row) * 2;
            okslot[hc] = s_ok;
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            // both warps of the pair read both flags: they leave together
            alive = s_ok && okslot[hc ^ 1];
            if (!alive) break;
            const float mx = fmaxf(mine, slot[hc ^ 1]);
            const float m_tile = fmaf(mx, sl2, ct);
            // Lazy rescale: O is rescaled only when the maximum grows by more
            // than the threshold.  ALiBi and the sparse form rescale on any
            // growth, so the row's largest P stays 2^0 (see the tile order
            // above).
            const bool grow = m_tile > m_run + ((ALIBI || SPARSE) ? 0.f : kRescaleThreshold);
            // tcgen05.ld/st are warp-collective: the warp rescales together,
            // lanes whose maximum did not grow enough multiply by 1
            if (__any_sync(0xffffffffu, grow)) {
                const float alpha = grow ? fast_exp2(m_run - m_tile) : 1.f;
                l_run *= alpha;
                if (j > 0) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r16[16];
                        tc::ld_32x32b_x16(tO + c * 16, r16);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            r16[i] = __float_as_uint(__uint_as_float(r16[i]) * alpha);
                        tc::st_32x32b_x16(tO + c * 16, r16);
                    }
                }
                if (grow) m_run = m_tile;
            }
            {
                // P = 2^(s * scale + ct - m) as bf16 (masked keys hold -inf:
                // 2^-inf = 0).  With ALiBi the row's largest P, where it sets a
                // fresh maximum, is 2^0 up to rounding far below bf16's step.
                const float msub = m_run == kNegInf ? 0.f : m_run;
                const uint64_t scale2 = f2_pack(sl2, sl2), neg2 = f2_pack(ct - msub, ct - msub);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t *src = h ? rb : ra;  // packed in place: pair i -> word i
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(src[2 * i]),
                                                 __uint_as_float(src[2 * i + 1])),
                                         scale2, neg2),
                                  t0, t1);
                        const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        ps2[i & 1] = f2_add(ps2[i & 1], f2_pack(p0, p1));
                        src[i] = pack_bf16(p0, p1);
                    }
                    tc::st_32x32b_x16(tP + h * 16, src);
                }
            }
            float s0, s1, s2, s3;
            f2_unpack(ps2[0], s0, s1);
            f2_unpack(ps2[1], s2, s3);
            l_run += (s0 + s1) + (s2 + s3);
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(bar(Lay::B_PFULL + x));
        }
        // epilogue: combine the two halves' sums, normalise (sink in the
        // denominator) and store this warp's 64 output columns
        bool have_o = ntiles > 0 && alive;
        if (have_o) {
            have_o = warp_wait_bounded(bar(Lay::B_ODONE + x), (gstep + ntiles - 1) & 1,
                                       p.dev_error, abort);
            tc::fence_after_sync();
        }
        float *lslot = xl + (((n & 1) * kNQ + x) * 128 + row) * 2;
        lslot[hc] = l_run;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float l_tot = l_run + lslot[hc ^ 1];
        const float sink_l2 = p.sink ? p.sink[head] * kLog2e : kNegInf;
        const float M = fmaxf(m_run, sink_l2);
        float oscale = 0.f, lse = kNegInf;
        if (M != kNegInf) {
            const float f = fast_exp2(m_run - M);
            const float Z = l_tot * f + fast_exp2(sink_l2 - M);
            oscale = f / Z;
            lse = (M + log2f(Z)) * kLn2;
        }
        // the head size Dh <= 128 is a multiple of 16: the stores below skip
        // whole 8-column vectors past it (those columns of O are zero padding)
        const int Dh = p.head_dim;
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) +
                              ((int64_t)(geo.q_start + tok) * p.num_qo_heads + head) * Dh +
                              hc * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t r32[32];
            if (have_o) {  // warp-uniform: every lane takes part in the load
                tc::ld_32x32b_x32(tO + c * 32, r32);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) r32[i] = 0u;
            }
            if (row_valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = 8 * i;
                    if (hc * 64 + c * 32 + e >= Dh) break;
                    dst[i] = make_uint4(
                        pack_bf16(__uint_as_float(r32[e + 0]) * oscale, __uint_as_float(r32[e + 1]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 2]) * oscale, __uint_as_float(r32[e + 3]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 4]) * oscale, __uint_as_float(r32[e + 5]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 6]) * oscale, __uint_as_float(r32[e + 7]) * oscale));
                }
            }
        }
        if (row_valid && hc == 0 && p.lse_out)
            p.lse_out[(int64_t)(geo.q_start + tok) * p.num_qo_heads + head] = lse;
        if (ntiles > 0) {  // O_x has been read: the next item's first PV may overwrite it
            tc::fence_before_sync();
            mbar_arrive(bar(Lay::B_OFREE + x));
            gstep += ntiles;
        }
        }  // items
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        // If a wait of this launch gave up, MMAs this CTA issued may still
        // be running: the issuing thread lets them finish (bounded) before
        // tensor memory is released.  (Here rather than in the MMA loop, where
        // the extra code slowed the loop by 1-2 %.)
        // (the word is re-read through the kernel parameter, so that no
        // register holds its address through the roles' loops)
        if (lane == 0 && *reinterpret_cast<volatile int32_t *>(p.tiles + 1) != 0) {
            tc::commit(bar(Lay::B_DRAIN));
            mbar_wait_bounded(bar(Lay::B_DRAIN), 0, p.dev_error);
        }
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Lay::TMEM_COLS);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return ensure_dynamic_smem(reinterpret_cast<const void *>(kernel), bytes);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, const pkv_cache_desc &cache, bool contiguous,
                           const CUtensorMap *tmap_q, const CUtensorMap *tmap_k,
                           const CUtensorMap *tmap_v, cudaStream_t stream) {
    if (cache.dtype != PKV_BF16 || cache.head_dim % 16 != 0 ||
        (cache.head_dim > kHeadDim && cache.head_dim != 256))
        return cudaErrorNotSupported;
    cudaError_t e = launch_pdl(prefill_schedule_kernel, dim3(1), dim3(kSchedThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    if (cache.head_dim == 256)
        return launch_prefill_wide(p, cache, contiguous, tmap_q, tmap_k, tmap_v, stream);
    if (p.max_tiles <= 0) return cudaSuccess;
    // the dense forms are persistent: one CTA per SM (or the caller's cap),
    // each drawing work items until none is left; the sparse form takes one
    // item per CTA
    const int ctas = p.max_ctas > 0 ? p.max_ctas : device_sm_count();
    const int persistent_grid = p.max_tiles < ctas ? p.max_tiles : ctas;
    auto go = [&](auto kern, bool persistent) -> cudaError_t {
        cudaError_t e2 = set_smem(kern, PfLayout::SMEM);
        if (e2 != cudaSuccess) return e2;
        const int grid = persistent ? persistent_grid : p.max_tiles;
        return launch_pdl(kern, dim3(grid), dim3(PfLayout::THREADS), PfLayout::SMEM, stream, p,
                          *tmap_q, *tmap_k, *tmap_v);
    };
    auto paged = [&](auto alibi_tag) -> cudaError_t {
        constexpr bool AL = decltype(alibi_tag)::value;
        if (cache.block_size == 16)
            return p.hnd ? go(prefill_tc_kernel<16, false, AL, true>, true)
                         : go(prefill_tc_kernel<16, false, AL, false>, true);
        if (cache.block_size == 32)
            return p.hnd ? go(prefill_tc_kernel<32, false, AL, true>, true)
                         : go(prefill_tc_kernel<32, false, AL, false>, true);
        return cudaErrorNotSupported;
    };
    if (contiguous && p.vbits)
        return go(prefill_tc_kernel<kTileN, true, false, false, true>, false);
    if (contiguous)
        return p.alibi ? go(prefill_tc_kernel<kTileN, true, true, false>, true)
                       : go(prefill_tc_kernel<kTileN, true, false, false>, true);
    return p.alibi ? paged(std::true_type{}) : paged(std::false_type{});
}

}  // namespace pkv
