// prefill_wide.cu -- varlen / chunk prefill for head_dim 256 on the
// 5th-generation tensor cores (tcgen05 + TMEM).
//
// Same attention as prefill.cu (transformers docs "paged_attention", varlen
// path; FlashInfer sink_attention_reference.py, varlen branch and
// sink_softmax; vLLM attention.py: ALiBi, head sizes up to 256), same work
// list (one request, one kv head, two query tiles of 128 GQA-packed rows per
// item), same masks and numerics.  What changes with 256 dims is the budget:
//   * an O accumulator of a 128-row tile takes 256 of the SM's 512 TMEM
//     columns, so one CTA holds one query tile.  A work item runs on a
//     cluster of two CTAs, one per query tile, over the union of the two
//     tiles' key ranges (a key tile past one tile's causal range is masked
//     for it);
//   * the key tiles stay 128 wide, so that S = Q K^T runs as N = 128 MMAs at
//     the tensor pipe's full rate (an N = 64 MMA takes as long as an N = 128
//     one); S is double-buffered in the other 256 TMEM columns, and the MMA
//     issuer computes S(j+1) while the softmax warps work on S(j);
//   * a K or V tile of 128 keys x 256 dims is 64 KB, so shared memory holds
//     Q (64 KB) and a ring of four 32 KB units, each 128 keys x 128 dims (one
//     half of a K or V tile): 192 KB.  The units are filled in the order the
//     MMAs consume them -- K(0), K(1), V(0), K(2), V(1), ... -- and both CTAs
//     of the cluster need the same ones: each CTA loads one 64-dim chunk of
//     every unit and multicasts it to both, so an SM issues half the TMA
//     boxes (on 16-row pages, 8 boxes of 2 KB per unit).  A unit's slot is
//     refilled once the MMAs of both CTAs have read it.
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps
// 2..9 softmax (two per TMEM lane quarter, each owning 64 of a row's 128 key
// columns and 128 of its 256 output columns).
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"
#include "prefill_common.cuh"

namespace pkv {

namespace {

using pf::kNegInf;

constexpr int kD = 256;
constexpr int kTileM = 128;
constexpr int kTileN = 128;                // keys per tile
constexpr int kSlots = 4;                  // ring units
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct WideLayout {
    static constexpr int Q_BYTES = kTileM * kD * 2;       // 64 KB
    static constexpr int Q_CHUNK = kTileM * 128;          // one 64-dim chunk: 16 KB
    static constexpr int U_BYTES = kTileN * 128 * 2;      // one unit, 128 dims: 32 KB
    static constexpr int U_CHUNK = kTileN * 128;          // one 64-dim chunk of it: 16 KB
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + Q_BYTES;
    static constexpr int OFF_BAR = OFF_RING + kSlots * U_BYTES;
    static constexpr int B_Q = 0;
    static constexpr int B_FULL = 1;
    static constexpr int B_EMPTY = B_FULL + kSlots;  // two arrivals: the MMAs of both CTAs
    // A parity wait is only valid within one phase of the barrier, so the
    // barriers that can have two completions outstanding come in pairs:
    // SFULL / PFULL / ODONE [g & 1] complete step g (phase g >> 1); VFIX[u]
    // the zeroed tail of the value unit in ring slot u.
    static constexpr int B_VFIX = B_EMPTY + kSlots;
    static constexpr int B_SFULL = B_VFIX + kSlots;
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_ODONE = B_PFULL + 2;
    static constexpr int B_DRAIN = B_ODONE + 2;  // the MMAs in flight, after a failed wait
    static constexpr int NBARS = B_DRAIN + 1;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    // row-max exchange [2 (step parity)][128][2] and row-sum exchange
    // [128][2] between the two warps of a row
    static constexpr int OFF_XMAX = OFF_TMEM + 16;
    static constexpr int OFF_XL = OFF_XMAX + 2 * 128 * 2 * 4;
    // the row pairs' wait status ([2][128][2] ints, double-buffered like the
    // maxima)
    static constexpr int OFF_XOK = OFF_XL + 128 * 2 * 4;
    static constexpr int SMEM = 1024 + OFF_XOK + 2 * 128 * 2 * 4;
    static constexpr int SOFT_THREADS = 256;
    static constexpr int THREADS = 64 + SOFT_THREADS;
    static constexpr int TMEM_COLS = 512;  // O: 0..255, S0: 256..383, S1: 384..511
    static constexpr int O_COL = 0;
};
static_assert(WideLayout::SMEM <= 227 * 1024, "shared memory budget");

__host__ __device__ constexpr int s_col(int b) { return 256 + b * 128; }

// ---------------------------------------------------------------------------
// the two-CTA cluster
// ---------------------------------------------------------------------------
constexpr uint16_t kPairMask = 0x3;  // both CTAs of the cluster

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// every thread of both CTAs arrives, then waits for all the others
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the barrier initialisations of this CTA become visible to the cluster
__device__ __forceinline__ void fence_barrier_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// A 3-D tile load whose box lands at the same shared-memory offset in every
// CTA of `mask`, each CTA's barrier at offset `bar` receiving its bytes.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int c0, int c1, int c2,
                                                 uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "h"(mask)
        : "memory");
}
// Arrive once on the barrier at offset `bar` of every CTA of `mask` when the
// MMAs this thread issued so far are done.
__device__ __forceinline__ void commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster"
        ".b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// The key tiles of query tile x of the item (none when the tile holds no
// query row of the request).
struct TileRange {
    int kt_lo, n;
};

__device__ __forceinline__ TileRange tile_range(const PrefillParams &p, const pf::Geo &G,
                                                int x) {
    TileRange t;
    const int tb = G.t0 + x * p.rows_per_head;
    pf::key_tiles(p, G, tb, tb + p.rows_per_head, kTileN, t.kt_lo, t.n);
    if (tb >= G.q_len) t.n = 0;
    return t;
}

// The key tiles the two query tiles of an item attend together (the union of
// their ranges; both CTAs of the item's cluster compute the same one).
__device__ __forceinline__ TileRange pair_range(const TileRange &a, const TileRange &b) {
    if (a.n == 0) return b;
    if (b.n == 0) return a;
    TileRange u;
    u.kt_lo = min(a.kt_lo, b.kt_lo);
    u.n = max(a.kt_lo + a.n, b.kt_lo + b.n) - u.kt_lo;
    return u;
}

template <int BS, bool CONTIG, bool ALIBI, bool HND>
__global__ void __launch_bounds__(WideLayout::THREADS, 1)
prefill_wide_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
    using Lay = WideLayout;
    constexpr int NPG = kTileN / BS;  // pages per key tile

    pdl_wait();  // the work list
    // clusters of two consecutive CTAs: one work item, CTA rank x = its
    // query tile
    const int pair = (int)blockIdx.x >> 1;
    if (pair >= p.tiles[0]) return;  // beyond the work list (both CTAs of the cluster)
    const int4 item = reinterpret_cast<const int4 *>(p.tiles + 64)[pair];
    const int x = (int)cluster_rank();

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = pf::align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + Lay::OFF_Q, sR = sbase + Lay::OFF_RING;
    const uint32_t bars = sbase + Lay::OFF_BAR;
    auto bar = [&](int i) { return bars + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_TMEM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const pf::Geo geo = pf::item_geo(p, item, BS, CONTIG, threadIdx.x == 0 && x == 0);
    int32_t *const abort = pf::abort_word(p);
    const TileRange t = pair_range(tile_range(p, geo, 0), tile_range(p, geo, 1));
    const int G = p.group;
    const int TPR = p.rows_per_head;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lay::NBARS; ++i) {
            uint32_t count = 1;
            if (i == Lay::B_PFULL || i == Lay::B_PFULL + 1) count = Lay::SOFT_THREADS;
            if (i >= Lay::B_EMPTY && i < Lay::B_EMPTY + kSlots) count = 2;
            mbar_init(bar(i), count);
        }
        fence_barrier_init_cluster();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    // both CTAs' barriers are initialised before either multicasts a copy or
    // commits to the other's barriers
    cluster_sync();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // Key tiles in processing order (ALiBi: from the query's end backwards, so
    // the nearest keys set the row maximum first) and the partial last tile.
    auto tile_of = [&](int n, int j) { return ALIBI ? n - 1 - j : j; };
    auto is_tail = [&](int j) {
        return t.n > 0 && (t.kt_lo + t.n) * kTileN > geo.kv_len && tile_of(t.n, j) == t.n - 1;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The units go in the order K(0) | K(1) V(0) | K(2) V(1) | ... | V(n-1),
        // two units (dims 0..127, 128..255) per key tile; unit u sits in ring
        // slot u % 4.  This CTA loads 64-dim chunk x of every unit, for both.
        const int32_t *bt = p.block_table + (int64_t)geo.r * p.max_blocks_per_seq;
        const int cy = HND ? 0 : geo.g;
        const int oob_row = HND ? (int)(p.num_blocks * p.num_kv_heads) : (int)(p.num_blocks * BS);
        const int npages_kv = (geo.kv_len + BS - 1) / BS;
        bool alive = true;
        int u = 0;
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        int ids_batch = -1, ids_row = oob_row;
        // the pool row of the page this lane loads (lane) in key tile `tile`
        auto page_row = [&](int tile) -> int {
            if constexpr (CONTIG) {
                return p.cu_k[geo.r] + (t.kt_lo + tile) * kTileN;  // rows past kv_len are masked
            } else {
                const int rel = tile * NPG;
                if ((rel >> 5) != ids_batch) {  // 32 block ids per warp-wide load
                    ids_batch = rel >> 5;
                    const int pg = t.kt_lo * NPG + ids_batch * 32 + lane;
                    ids_row = oob_row;
                    if (pg < npages_kv) {
                        const int blk = bt[pg];
                        if (blk < 0 || blk >= p.num_blocks) {
                            if (x == 0) flag_error(p.dev_error, PKV_DEVERR_BLOCK_ID);
                        } else {
                            ids_row = HND ? blk * p.num_kv_heads + geo.g : blk * BS;
                        }
                    }
                }
                return __shfl_sync(0xffffffffu, ids_row, ((rel & 31) + min(lane, NPG - 1)) & 31);
            }
        };
        // one unit: half h of the K (tm = &tmk) or V tile whose page rows the
        // lanes hold; a value unit of the partial last tile gets its rows at
        // or past kv_len zeroed in this CTA's copy (they may hold any bits, and
        // P = 0 must never meet a non-finite value)
        auto load_unit = [&](const CUtensorMap *tm, int row, int h, int tail_first) {
            const int slot = u & (kSlots - 1);
            const uint32_t ph = (u >> 2) & 1;
            // both CTAs' MMAs are done with the slot's previous unit
            alive = warp_wait_bounded(bar(Lay::B_EMPTY + slot), ph ^ 1, p.dev_error, abort);
            if (!alive) return;
            const uint32_t dst = sR + slot * Lay::U_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(bar(Lay::B_FULL + slot), Lay::U_BYTES);
            __syncwarp();
            if (lane < NPG)
                tma_load_3d_pair(dst + x * Lay::U_CHUNK + lane * BS * 128, tm,
                                 bar(Lay::B_FULL + slot), (2 * h + x) * 64, cy, row, kPairMask);
            ++u;
            if (tail_first >= 0) {
                alive = warp_wait_bounded(bar(Lay::B_FULL + slot), ph, p.dev_error, abort);
                if (!alive) return;
                for (int e = tail_first * 16 + lane; e < kTileN * 16; e += 32) {
                    const int rr = e >> 4, c = e & 15;
                    pf::st_shared_zero16(dst + (c >> 3) * Lay::U_CHUNK + sw128(rr, c & 7));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Lay::B_VFIX + slot));
            }
        };
        if (t.n > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(Lay::B_Q), Lay::Q_BYTES);
                for (int c = 0; c < kD / 64; ++c)
                    tma_load_3d(sQ + c * Lay::Q_CHUNK, &tmq, bar(Lay::B_Q), c * 64, geo.g * G,
                                geo.q_start + geo.t0 + x * TPR);
            }
            int row_cur = page_row(tile_of(t.n, 0));
            for (int h = 0; h < 2 && alive; ++h) load_unit(&tmk, row_cur, h, -1);
            for (int j = 0; j < t.n && alive; ++j) {
                int row_next = row_cur;
                if (j + 1 < t.n) {
                    row_next = page_row(tile_of(t.n, j + 1));
                    for (int h = 0; h < 2 && alive; ++h) load_unit(&tmk, row_next, h, -1);
                }
                const int key0 = (t.kt_lo + tile_of(t.n, j)) * kTileN;
                const int first = is_tail(j) ? max(geo.kv_len - key0, 0) : -1;
                for (int h = 0; h < 2 && alive; ++h) load_unit(&tmv, row_cur, h, first);
                row_cur = row_next;
            }
        }
        // let both MMA issuers' last arrivals land before the CTA can exit
        for (int k = max(0, u - kSlots); k < u && alive; ++k)
            alive = warp_wait_bounded(bar(Lay::B_EMPTY + (k & (kSlots - 1))), (k >> 2) & 1,
                                      p.dev_error, abort);
        if (!alive) {
            // a wait gave up: let the copies still in flight into this CTA
            // land (bounded) before its shared memory is released
            if (t.n > 0) warp_wait_bounded(bar(Lay::B_Q), 0, p.dev_error);
            for (int k = max(0, u - kSlots); k < u; ++k)
                warp_wait_bounded(bar(Lay::B_FULL + (k & (kSlots - 1))), (k >> 2) & 1,
                                  p.dev_error);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && t.n > 0) {
            constexpr uint32_t idS = tc::idesc_bf16_f32(kTileM, kTileN, 0, 0);
            constexpr uint32_t idO = tc::idesc_bf16_f32(kTileM, 128, 0, 1);
            bool alive = true;
            int u = 0, g = 0;
            uint32_t vfix_par = 0;  // bit u: parity of the next tail fix in slot u
            // S(g) = Q K^T into buffer g & 1, from the two K units of its tile
            auto issue_s = [&]() {
                const int b = g & 1;
                for (int h = 0; h < 2 && alive; ++h) {
                    const int slot = u & (kSlots - 1);
                    alive = mbar_wait_bounded(bar(Lay::B_FULL + slot), (u >> 2) & 1, p.dev_error,
                                              abort);
                    if (!alive) return;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t a = tc::smem_desc_sw128(
                            sQ + (2 * h + (kk >> 2)) * Lay::Q_CHUNK + off, 16, 1024);
                        const uint64_t bd = tc::smem_desc_sw128(
                            sR + slot * Lay::U_BYTES + (kk >> 2) * Lay::U_CHUNK + off, 16, 1024);
                        tc::mma_ss(tmem + s_col(b), a, bd, idS, (h > 0 || kk > 0) ? 1u : 0u);
                    }
                    commit_pair(bar(Lay::B_EMPTY + slot), kPairMask);
                    ++u;
                }
                if (alive) tc::commit(bar(Lay::B_SFULL + b));
            };
            // O += P(g) V, one 128-column half of O per V unit
            auto issue_pv = [&](bool first, bool tail) {
                const int b = g & 1;
                for (int h = 0; h < 2 && alive; ++h) {
                    const int slot = u & (kSlots - 1);
                    if (tail) {
                        alive = mbar_wait_bounded(bar(Lay::B_VFIX + slot), (vfix_par >> slot) & 1,
                                                  p.dev_error, abort);
                        vfix_par ^= 1u << slot;
                    } else {
                        alive = mbar_wait_bounded(bar(Lay::B_FULL + slot), (u >> 2) & 1,
                                                  p.dev_error, abort);
                    }
                    if (!alive) return;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < kTileN / 16; ++kk) {
                        const uint64_t bd = tc::smem_desc_sw128(
                            sR + slot * Lay::U_BYTES + kk * 2048, Lay::U_CHUNK, 1024);
                        tc::mma_ts(tmem + Lay::O_COL + h * 128, tmem + s_col(b) + kk * 8, bd,
                                   idO, (!first || kk > 0) ? 1u : 0u);
                    }
                    commit_pair(bar(Lay::B_EMPTY + slot), kPairMask);
                    ++u;
                }
                if (alive) tc::commit(bar(Lay::B_ODONE + b));
            };
            // S(g) overwrites P(g - 2): PV(g - 2) must be done
            auto free_s = [&]() {
                if (g < 2) return;
                const int k = g - 2;
                alive = mbar_wait_bounded(bar(Lay::B_ODONE + (k & 1)), (k >> 1) & 1, p.dev_error,
                                          abort);
                tc::fence_after_sync();
            };
            alive = mbar_wait_bounded(bar(Lay::B_Q), 0, p.dev_error, abort);
            if (alive) {
                tc::fence_after_sync();
                issue_s();
            }
            for (int j = 0; j < t.n && alive; ++j) {
                if (j + 1 < t.n) {
                    g = j + 1;
                    free_s();
                    if (alive) issue_s();
                }
                g = j;
                if (!alive) break;
                alive = mbar_wait_bounded(bar(Lay::B_PFULL + (g & 1)), (g >> 1) & 1, p.dev_error,
                                          abort);
                if (!alive) break;
                tc::fence_after_sync();
                issue_pv(j == 0, is_tail(j));
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Two warps per TMEM lane quarter: half hc owns key columns
        // [64 hc, 64 hc + 64) of S, packed P columns [32 hc, 32 hc + 32) and
        // output columns [128 hc, 128 hc + 128).
        const int w = warp - 2;
        const int quarter = warp & 3;
        const int hc = w >> 2;
        const int row = quarter * 32 + lane;
        const int tok_local = row / G;
        const int h_local = row - tok_local * G;
        const int head = geo.g * G + h_local;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t pair_bar = 1 + quarter;
        float *xmax = reinterpret_cast<float *>(smem + Lay::OFF_XMAX);
        float *xl = reinterpret_cast<float *>(smem + Lay::OFF_XL);
        const float sl2 = p.scale_log2;
        const int wl = p.window_left;
        const float al2 = ALIBI ? p.alibi[head] * kLog2e : 0.f;
        const float sink_l2 = p.sink ? p.sink[head] * kLog2e : kNegInf;
        bool alive = true, o_ok = true;
        const int tok = geo.t0 + x * TPR + tok_local;
        const bool row_valid = tok < geo.q_len;
        const int qpos = geo.kv_len - geo.q_len + tok;
        const int cpos = p.causal ? qpos : (1 << 30);  // causal upper bound on keys
        float m_run = kNegInf, l_run = 0.f;
        for (int j = 0; j < t.n && alive; ++j) {
            const int g = j;
            const int b = g & 1;
            // a warp whose wait gave up still meets its partner at the pair
            // barrier below, and both leave together
            const bool s_wait = warp_wait_bounded(bar(Lay::B_SFULL + b), (g >> 1) & 1,
                                                  p.dev_error, abort);
            const bool s_ok = o_ok && s_wait;
            tc::fence_after_sync();
            const int key0 = (t.kt_lo + tile_of(t.n, j)) * kTileN + hc * 64;
            const bool full = (key0 + 63 <= cpos) && (key0 + 64 <= geo.kv_len) &&
                              (wl < 0 || key0 >= qpos - wl);
            const int khi = min(cpos, geo.kv_len - 1) - key0;
            const int klo = wl < 0 ? -1 : qpos - wl - key0;
            uint32_t ra[2][32];
            // loaded even after a failed wait (the values are then unused)
            tc::ld_32x32b_x32(tmem + lane_off + s_col(b) + hc * 64, ra[0]);
            tc::ld_32x32b_x32(tmem + lane_off + s_col(b) + hc * 64 + 32, ra[1]);
            tc::wait_ld();
            if (!full) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (!(i <= khi && i >= klo)) ra[i >> 5][i & 31] = __float_as_uint(kNegInf);
            }
            float mx4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
            if constexpr (ALIBI) {
                // x = s * scale + slope * (key - position), packed pairs
                const float b0 = al2 * (float)(key0 - qpos);
                const uint64_t sc2 = f2_pack(sl2, sl2), step2 = f2_pack(4.f * al2, 4.f * al2);
                uint64_t bc[2] = {f2_pack(b0, b0 + al2),
                                  f2_pack(b0 + 2.f * al2, b0 + 3.f * al2)};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    uint32_t &r0 = ra[i >> 4][(2 * i) & 31], &r1 = ra[i >> 4][(2 * i + 1) & 31];
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(r0), __uint_as_float(r1)), sc2,
                                     bc[i & 1]),
                              x0, x1);
                    bc[i & 1] = f2_add(bc[i & 1], step2);
                    r0 = __float_as_uint(x0);
                    r1 = __float_as_uint(x1);
                    mx4[i & 3] = fmax3(mx4[i & 3], x0, x1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    mx4[i & 3] = fmax3(mx4[i & 3], __uint_as_float(ra[i >> 4][(2 * i) & 31]),
                                       __uint_as_float(ra[i >> 4][(2 * i + 1) & 31]));
            }
            const float mine = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            float *slot = xmax + ((g & 1) * 128 + row) * 2;
            slot[hc] = mine;
            int *okslot = reinterpret_cast<int *>(smem + Lay::OFF_XOK) +
                          ((g & 1) * 128 + row) * 2;
            okslot[hc] = s_ok;
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            // both warps of the pair read both flags: they leave together
            alive = s_ok && okslot[hc ^ 1];
            if (!alive) break;
            const float mx = fmaxf(mine, slot[hc ^ 1]);
            const float m_tile = ALIBI ? mx : mx * sl2;
            const bool grow = m_tile > m_run + (ALIBI ? 0.f : kRescaleThreshold);
            if (__any_sync(0xffffffffu, grow)) {
                const float alpha = grow ? fast_exp2(m_run - m_tile) : 1.f;
                l_run *= alpha;
                if (j > 0) {
                    // O is written by PV(g-1): wait for it before rescaling (a
                    // wait that gives up is reported at the next pair barrier)
                    const int k = g - 1;
                    o_ok = warp_wait_bounded(bar(Lay::B_ODONE + (k & 1)), (k >> 1) & 1,
                                             p.dev_error, abort);
                }
                if (j > 0 && o_ok) {
                    tc::fence_after_sync();
                    const uint32_t tO = tmem + lane_off + Lay::O_COL + hc * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
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
            const float msub = m_run == kNegInf ? 0.f : m_run;
            const float psc = ALIBI ? 1.f : sl2;
            const uint64_t scale2 = f2_pack(psc, psc), neg2 = f2_pack(-msub, -msub);
            uint64_t ps2[2] = {0ull, 0ull};
            uint32_t pw[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float t0, t1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[i >> 4][(2 * i) & 31]),
                                         __uint_as_float(ra[i >> 4][(2 * i + 1) & 31])),
                                 scale2, neg2),
                          t0, t1);
                const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                ps2[i & 1] = f2_add(ps2[i & 1], f2_pack(p0, p1));
                pw[i] = pack_bf16(p0, p1);
            }
            tc::st_32x32b_x32(tmem + lane_off + s_col(b) + hc * 32, pw);
            float s0, s1, s2, s3;
            f2_unpack(ps2[0], s0, s1);
            f2_unpack(ps2[1], s2, s3);
            l_run += (s0 + s1) + (s2 + s3);
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(bar(Lay::B_PFULL + b));
        }
        // epilogue: combine the halves' sums, normalise (sink in the
        // denominator) and store this warp's 128 output columns
        bool have_o = t.n > 0 && alive;
        if (have_o) {
            // the last PV's commit covers every earlier MMA
            const int k = t.n - 1;
            have_o = warp_wait_bounded(bar(Lay::B_ODONE + (k & 1)), (k >> 1) & 1, p.dev_error,
                                       abort);
            tc::fence_after_sync();
        }
        float *lslot = xl + row * 2;
        lslot[hc] = l_run;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float l_tot = l_run + lslot[hc ^ 1];
        const float M = fmaxf(m_run, sink_l2);
        float oscale = 0.f, lse = kNegInf;
        if (M != kNegInf) {
            const float f = fast_exp2(m_run - M);
            const float Z = l_tot * f + fast_exp2(sink_l2 - M);
            oscale = f / Z;
            lse = (M + log2f(Z)) * kLn2;
        }
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) +
                              ((int64_t)(geo.q_start + tok) * p.num_qo_heads + head) * kD +
                              hc * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t r32[32];
            if (have_o) {  // warp-uniform: every lane takes part in the load
                tc::ld_32x32b_x32(tmem + lane_off + Lay::O_COL + hc * 128 + c * 32, r32);
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
                    dst[i] = make_uint4(
                        pack_bf16(__uint_as_float(r32[e + 0]) * oscale,
                                  __uint_as_float(r32[e + 1]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 2]) * oscale,
                                  __uint_as_float(r32[e + 3]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 4]) * oscale,
                                  __uint_as_float(r32[e + 5]) * oscale),
                        pack_bf16(__uint_as_float(r32[e + 6]) * oscale,
                                  __uint_as_float(r32[e + 7]) * oscale));
                }
            }
        }
        if (row_valid && hc == 0 && p.lse_out)
            p.lse_out[(int64_t)(geo.q_start + tok) * p.num_qo_heads + head] = lse;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        // If a wait of this launch gave up, MMAs this CTA issued may still
        // be running: the issuing thread lets them finish (bounded) before
        // tensor memory is released.
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
    // neither CTA leaves while the other may still commit to its barriers
    cluster_sync();
}

template <typename K>
cudaError_t set_smem_wide(K kernel, int bytes) {
    return ensure_dynamic_smem(reinterpret_cast<const void *>(kernel), bytes);
}

}  // namespace

cudaError_t launch_prefill_wide(const PrefillParams &p, const pkv_cache_desc &cache,
                                bool contiguous, const CUtensorMap *tmap_q,
                                const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                cudaStream_t stream) {
    if (p.max_tiles <= 0) return cudaSuccess;
    if ((int64_t)p.max_tiles * 2 > INT32_MAX) return cudaErrorNotSupported;
    const int grid = 2 * p.max_tiles;  // a cluster of two CTAs per work item
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = set_smem_wide(kern, WideLayout::SMEM);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(WideLayout::THREADS);
        cfg.dynamicSmemBytes = WideLayout::SMEM;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kern, p, *tmap_q, *tmap_k, *tmap_v);
    };
    auto paged = [&](auto alibi_tag) -> cudaError_t {
        constexpr bool AL = decltype(alibi_tag)::value;
        if (cache.block_size == 16)
            return p.hnd ? go(prefill_wide_kernel<16, false, AL, true>)
                         : go(prefill_wide_kernel<16, false, AL, false>);
        if (cache.block_size == 32)
            return p.hnd ? go(prefill_wide_kernel<32, false, AL, true>)
                         : go(prefill_wide_kernel<32, false, AL, false>);
        return cudaErrorNotSupported;
    };
    if (contiguous)
        return p.alibi ? go(prefill_wide_kernel<kTileN, true, true, false>)
                       : go(prefill_wide_kernel<kTileN, true, false, false>);
    return p.alibi ? paged(std::true_type{}) : paged(std::false_type{});
}

}  // namespace pkv
