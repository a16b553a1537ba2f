// prefill_common.cuh -- what the prefill kernels share: the geometry of a work
// item (one request, one kv head, two query tiles of 128 GQA-packed rows) and
// the key tiles its query rows attend.
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace pf {

constexpr int kItemTiles = 2;  // query tiles of 128 rows per work item
constexpr float kNegInf = -INFINITY;

struct Geo {
    int r, t0, g;               // request, first query token, kv head
    int q_start, q_len, kv_len;
};

__device__ __forceinline__ int clip_len(int v, int cap, int32_t *err, bool report) {
    if (v < 0) {
        if (report) flag_error(err, PKV_DEVERR_SEQLEN);
        return 0;
    }
    if (v > cap) {
        if (report) flag_error(err, PKV_DEVERR_SEQLEN);
        return cap;
    }
    return v;
}

// Word 1 of the work list's 256-byte header: the attention launch's abort
// word (mbar_wait_bounded), zeroed by the work-list kernel before each launch.
__device__ __forceinline__ int32_t *abort_word(const PrefillParams &p) { return p.tiles + 1; }

// Word 2: the count of work items drawn beyond the first one of every CTA
// (persistent attention CTAs), zeroed by the work-list kernel.
__device__ __forceinline__ int32_t *item_counter(const PrefillParams &p) { return p.tiles + 2; }

__device__ __forceinline__ int clip_len64(long long v, int cap, int32_t *err, bool report) {
    return clip_len(v < 0 ? -1 : (v > cap ? cap + 1 : (int)v), cap, err, report);
}

// Request r's query rows [q_start, q_start + q_len) of the total_q rows of q,
// out and lse.  cu_seq_lens_q lives on the device, so its entries are checked
// here: an offset outside [0, total_q], a negative length, a length above
// max_seqlen_q or one running past total_q is clipped and flagged
// (PKV_DEVERR_SEQLEN).  No row outside [0, total_q) is ever read or written.
__device__ __forceinline__ void q_rows(const PrefillParams &p, int r, int &q_start, int &q_len,
                                       bool report) {
    const int a = p.cu_q[r], b = p.cu_q[r + 1];
    int s = a;
    if (s < 0 || s > p.total_q) {
        if (report) flag_error(p.dev_error, PKV_DEVERR_SEQLEN);
        s = s < 0 ? 0 : p.total_q;
    }
    int len = clip_len64((long long)b - a, p.max_seqlen_q, p.dev_error, report);
    if (len > p.total_q - s) {
        if (report) flag_error(p.dev_error, PKV_DEVERR_SEQLEN);
        len = p.total_q - s;
    }
    q_start = s;
    q_len = len;
}

// The item's request lengths, clipped to the declared maxima, to the rows of
// q, to the block table's capacity and, for contiguous K/V, to the rows that
// exist.
__device__ __forceinline__ Geo item_geo(const PrefillParams &p, int4 item, int block_size,
                                        bool contiguous, bool report) {
    Geo G;
    G.r = item.x;
    G.t0 = item.y;
    G.g = item.z;
    q_rows(p, G.r, G.q_start, G.q_len, report);
    int cap_k = p.max_seqlen_k;
    const long long cap_blocks = (long long)p.max_blocks_per_seq * block_size;
    if (cap_blocks < cap_k) cap_k = (int)cap_blocks;
    if (contiguous) {  // request r's key rows must lie inside the arrays
        const int k0 = p.cu_k[G.r];
        const long long room = k0 < 0 ? 0 : (long long)p.total_k - k0;
        if (k0 < 0 && report) flag_error(p.dev_error, PKV_DEVERR_SEQLEN);
        if (room < cap_k) cap_k = room > 0 ? (int)room : 0;
    }
    G.kv_len = clip_len64((long long)p.cu_k[G.r + 1] - p.cu_k[G.r], cap_k, p.dev_error, report);
    return G;
}

// Key tiles [kt_lo, kt_lo + n) of `tile` keys that hold every key the query
// tokens [t_begin, t_end) of the request may attend (causal bound, window);
// n = 0 when they attend none.
__device__ __forceinline__ void key_tiles(const PrefillParams &p, const Geo &G, int t_begin,
                                          int t_end, int tile, int &kt_lo, int &n) {
    t_end = min(t_end, G.q_len);
    const int qpos_min = G.kv_len - G.q_len + t_begin;
    const int qpos_max = G.kv_len - G.q_len + t_end - 1;
    const int hi = p.causal ? min(G.kv_len, qpos_max + 1) : G.kv_len;
    int lo = 0;
    if (p.window_left >= 0) lo = max(0, qpos_min - p.window_left);
    if (hi <= lo || t_end <= t_begin) {
        kt_lo = 0;
        n = 0;
    } else {
        kt_lo = lo / tile;
        n = (hi - 1) / tile - kt_lo + 1;
    }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *ptr) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(ptr) + 1023) & ~uintptr_t(1023);
    return reinterpret_cast<uint8_t *>(a);
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

}  // namespace pf
}  // namespace pkv
