// rope_cache.cu -- rotary position embedding fused with the reshape_and_cache
// scatter.
//
// vLLM attention.py, PagedAttentionWithRoPE.forward: before the cache write
// the query and key of every new token are rotated by its position
// (rotary_emb(positions, query, key); head_size, rotary_dim, base,
// is_neox_style and a linear / dynamic rope_scaling factor configure it), and
// the rotated key and the value then go to the paged cache at slot_mapping.
// The rotation is RoFormer's: frequency i in [0, rotary_dim/2) has
// theta_i = base^(-2i/rotary_dim); the pair (x_a, x_b) of frequency i of a
// token at position m turns by m * theta_i (neox style pairs i with
// i + rotary_dim/2, GPT-J style pairs 2i with 2i+1); dimensions past
// rotary_dim are left as they are.
//
// GB300 design.  Two kernels.
//  * rope_table_kernel builds the cos/sin table once per configuration:
//    [max_position][rotary_dim/2] float2 (cos, sin).  The angle m * theta_i
//    reaches 1e5 radians for long contexts, where an fp32 product would be off
//    by several milli-radians, so the table is computed in fp64 and rounded
//    once to fp32.  Scaling variants only change the table (position_scale
//    divides m; a dynamic-NTK caller passes its adjusted base).
//  * rope_reshape_cache_kernel is the per-step op, HBM bound: one flat index
//    space over (token, unit); a unit is one 16-byte vector of a head row, or
//    for neox rotation the two vectors holding a pair's halves.  Per token the
//    units are the q heads' rotated vectors (rotated in place; pass-through
//    vectors of q are not touched at all), the k heads' vectors (rotated in
//    place and written to the cache slot; pass-through ones only copied to
//    the slot) and the v heads' vectors (copied to the slot).  Consecutive
//    threads take consecutive vectors of a row, so every access is a
//    coalesced 16-byte vector; cos/sin come from the table through the
//    read-only path (a few KB per position, mostly L2 hits).
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
rope_table_kernel(float2 *__restrict__ table, int max_position, int rotary_dim, double base,
                  double position_scale) {
    const int half = rotary_dim / 2;
    const int64_t total = (int64_t)max_position * half;
    for (int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * kThreads) {
        const int pos = (int)(idx / half);
        const int i = (int)(idx - (int64_t)pos * half);
        const double theta = pow(base, -2.0 * i / rotary_dim);
        const double angle = ((double)pos / position_scale) * theta;
        double s, c;
        sincos(angle, &s, &c);
        table[idx] = make_float2((float)c, (float)s);
    }
}

template <typename T>
struct Vec;  // one 16-byte vector as floats

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void *p, float (&x)[N]) {
        const float4 v = *static_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static void store(void *p, const float (&x)[N]) {
        *static_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void *p, float (&x)[N]) {
        const uint4 v = *static_cast<const uint4 *>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(void *p, const float (&x)[N]) {
        *static_cast<uint4 *>(p) = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                              pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
    }
};

// x_a' = x_a c - x_b s,  x_b' = x_b c + x_a s  (fp32)
__device__ __forceinline__ void rotate(float &a, float &b, float2 cs) {
    const float a2 = a * cs.x - b * cs.y;
    const float b2 = b * cs.x + a * cs.y;
    a = a2;
    b = b2;
}

// Unit layout per token (V elements per vector, nvec = D / V):
//   [0, Hq*nrot)                 q head h, rotation unit u
//   [.., + Hkv*nk)               k head h, unit u: u < nrot rotates, else copies
//   [.., + Hkv*nvec)             v head h, vector c
// neox: nrot = rd / (2V) units of two vectors (u and u + rd/(2V));
//       nk = nrot + (D - rd) / V.
// GPT-J: nrot = rd / V units of one vector (V/2 pairs); nk = nvec.
enum UnitKind { kQRot = 0, kKRot = 1, kKCopy = 2, kVCopy = 3 };

struct Unit {
    int t;          // token (within this launch)
    int kind;       // UnitKind
    int h;          // head
    int e0, e1;     // first element of the unit's vector(s) in the head row
    int f0;         // first frequency (rotation units)
};

struct Geometry {
    int V, nvec, nrot, nk, half, q_units, k_units, per_token;
};

template <bool NEOX>
__device__ __forceinline__ Geometry geometry(const RopeParams &p, int V) {
    Geometry g;
    g.V = V;
    g.nvec = p.head_dim / V;
    g.nrot = NEOX ? p.rotary_dim / (2 * V) : p.rotary_dim / V;
    g.nk = NEOX ? g.nrot + (p.head_dim - p.rotary_dim) / V : g.nvec;
    g.half = p.rotary_dim / 2;
    g.q_units = p.num_qo_heads * g.nrot;
    g.k_units = p.num_kv_heads * g.nk;
    g.per_token = g.q_units + g.k_units + p.num_kv_heads * g.nvec;
    return g;
}

// idx < 2^31 (the host splits larger launches by tokens)
template <bool NEOX>
__device__ __forceinline__ Unit locate(const RopeParams &p, const Geometry &g, uint32_t idx) {
    Unit w;
    w.t = (int)(idx / (uint32_t)g.per_token);
    int l = (int)(idx - (uint32_t)w.t * (uint32_t)g.per_token);
    int u;
    if (l < g.q_units) {
        w.h = l / g.nrot;
        u = l - w.h * g.nrot;
        w.kind = kQRot;
    } else if (l < g.q_units + g.k_units) {
        l -= g.q_units;
        w.h = l / g.nk;
        u = l - w.h * g.nk;
        w.kind = u < g.nrot ? kKRot : kKCopy;
    } else {
        l -= g.q_units + g.k_units;
        w.h = l / g.nvec;
        u = l - w.h * g.nvec;
        w.kind = kVCopy;
    }
    if (w.kind == kQRot || w.kind == kKRot) {
        w.e0 = u * g.V;
        w.e1 = NEOX ? g.half + u * g.V : w.e0;
        w.f0 = NEOX ? u * g.V : u * g.V / 2;
    } else {
        const int c = (w.kind == kKCopy && NEOX) ? p.rotary_dim / g.V + (u - g.nrot) : u;
        w.e0 = w.e1 = c * g.V;
        w.f0 = 0;
    }
    return w;
}

// Each thread takes kUnits units per pass, spaced one grid apart, and issues
// all their loads (input vectors, position, slot) before it uses any, so
// their HBM round trips overlap.  The cos/sin row of a position is shared by
// every head of the token and is read (from L1, mostly) while rotating.
constexpr int kUnits = 1;

template <typename T, bool NEOX, bool HND>
__global__ void __launch_bounds__(kThreads)
rope_reshape_cache_kernel(RopeParams p) {
    using VT = Vec<T>;
    constexpr int V = VT::N;
    constexpr int64_t ES = sizeof(T);
    const Geometry g = geometry<NEOX>(p, V);
    const uint32_t total = (uint32_t)p.num_tokens * (uint32_t)g.per_token;
    const int64_t row_q = (int64_t)p.num_qo_heads * p.head_dim;  // elements per token
    const int64_t row_kv = (int64_t)p.num_kv_heads * p.head_dim;
    uint8_t *const qb = static_cast<uint8_t *>(p.query);
    uint8_t *const kb = static_cast<uint8_t *>(p.key);
    const uint8_t *const vb = static_cast<const uint8_t *>(p.value);
    uint8_t *const kcb = static_cast<uint8_t *>(p.k_cache);
    uint8_t *const vcb = static_cast<uint8_t *>(p.v_cache);
    const uint32_t stride = gridDim.x * kThreads;

    auto row_of = [&](const Unit &w) -> uint8_t * {
        const uint8_t *r =
            w.kind == kQRot ? qb + ((int64_t)w.t * row_q + (int64_t)w.h * p.head_dim) * ES
            : w.kind == kVCopy ? vb + ((int64_t)w.t * row_kv + (int64_t)w.h * p.head_dim) * ES
                               : kb + ((int64_t)w.t * row_kv + (int64_t)w.h * p.head_dim) * ES;
        return const_cast<uint8_t *>(r);
    };

    for (uint32_t i0 = blockIdx.x * kThreads + threadIdx.x; i0 < total; i0 += kUnits * stride) {
        Unit w[kUnits];
        uint4 a[kUnits], b[kUnits];
        int64_t pos[kUnits], slot[kUnits];
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {  // all loads first
            const uint32_t idx = i0 + k * stride;
            if (idx >= total) continue;
            w[k] = locate<NEOX>(p, g, idx);
            pos[k] = __ldg(p.positions + w[k].t);
            slot[k] = __ldg(p.slot_mapping + w[k].t);
            const uint8_t *row = row_of(w[k]);
            a[k] = *reinterpret_cast<const uint4 *>(row + w[k].e0 * ES);
            if (NEOX && w[k].kind <= kKRot)
                b[k] = *reinterpret_cast<const uint4 *>(row + w[k].e1 * ES);
        }
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
            const uint32_t idx = i0 + k * stride;
            if (idx >= total) continue;
            const Unit &u = w[k];
            const bool first = idx == (uint32_t)u.t * (uint32_t)g.per_token;
            if (pos[k] < 0 || pos[k] >= p.max_position) {  // no table row: left alone
                if (first) flag_error(p.dev_error, PKV_DEVERR_POSITION);
                continue;
            }
            const bool cache_it = slot[k] >= 0 && slot[k] < p.capacity;
            if (slot[k] >= p.capacity && first) flag_error(p.dev_error, PKV_DEVERR_SLOT);
            uint8_t *row = row_of(u);
            // the slot's row of kv head h: NHD slot * row + h * D; HND
            // ((page * Hkv + h) * bs + offset) * D
            const int64_t sl = cache_it ? slot[k] : 0;
            int64_t crow_el;
            if constexpr (HND)
                crow_el = ((sl / p.block_size * p.num_kv_heads + u.h) * p.block_size +
                           sl % p.block_size) * p.head_dim;
            else
                crow_el = sl * row_kv + (int64_t)u.h * p.head_dim;
            uint8_t *crow = (u.kind == kVCopy ? vcb : kcb) + crow_el * ES;
            if (u.kind <= kKRot) {
                const float4 *cs4 =
                    reinterpret_cast<const float4 *>(p.cos_sin + pos[k] * g.half + u.f0);
                float x[V];
                VT::load(&a[k], x);
                if constexpr (NEOX) {
                    float y[V];
                    VT::load(&b[k], y);
#pragma unroll
                    for (int i = 0; i < V / 2; ++i) {
                        const float4 c2 = __ldg(cs4 + i);
                        rotate(x[2 * i], y[2 * i], make_float2(c2.x, c2.y));
                        rotate(x[2 * i + 1], y[2 * i + 1], make_float2(c2.z, c2.w));
                    }
                    VT::store(row + u.e0 * ES, x);
                    VT::store(row + u.e1 * ES, y);
                    if (u.kind == kKRot && cache_it) {
                        VT::store(crow + u.e0 * ES, x);
                        VT::store(crow + u.e1 * ES, y);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < V / 4; ++i) {
                        const float4 c2 = __ldg(cs4 + i);
                        rotate(x[4 * i], x[4 * i + 1], make_float2(c2.x, c2.y));
                        rotate(x[4 * i + 2], x[4 * i + 3], make_float2(c2.z, c2.w));
                    }
                    VT::store(row + u.e0 * ES, x);
                    if (u.kind == kKRot && cache_it) VT::store(crow + u.e0 * ES, x);
                }
            } else if (cache_it) {  // dimensions past rotary_dim of k, and v
                *reinterpret_cast<uint4 *>(crow + u.e0 * ES) = a[k];
            }
        }
    }
}

int grid_for(int64_t total) {
    int64_t blocks = (total + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

// Grid of a grid-stride kernel: every CTA resident at once (SMs x the CTAs
// per SM its registers allow, looked up once per kernel and device), so there
// is no partial last wave; fewer CTAs when the work is small.
template <auto Kernel>
int resident_grid(int64_t total) {
    constexpr int kDevs = 64;
    static std::atomic<int> per_sm_cache[kDevs];
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = (dev >= 0 && dev < kDevs) ? per_sm_cache[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, Kernel, kThreads, 0) !=
                cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        if (dev >= 0 && dev < kDevs) per_sm_cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    int64_t blocks = (total + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(device_sm_count()) * per_sm;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

cudaError_t launch_rope_table(float *table, int max_position, int rotary_dim, double base,
                              double position_scale, cudaStream_t stream) {
    const int64_t total = (int64_t)max_position * (rotary_dim / 2);
    if (total == 0) return cudaSuccess;
    rope_table_kernel<<<grid_for(total), kThreads, 0, stream>>>(
        reinterpret_cast<float2 *>(table), max_position, rotary_dim, base, position_scale);
    return cudaGetLastError();
}

cudaError_t launch_rope_reshape_cache(const RopeParams &p, int dtype, bool neox,
                                      cudaStream_t stream) {
    if (p.num_tokens == 0) return cudaSuccess;
    const int V = dtype == PKV_F32 ? 4 : 8;
    const int esz = dtype == PKV_F32 ? 4 : 2;
    const int nvec = p.head_dim / V;
    const int nrot = neox ? p.rotary_dim / (2 * V) : p.rotary_dim / V;
    const int nk = neox ? nrot + (p.head_dim - p.rotary_dim) / V : nvec;
    const int64_t per_token = (int64_t)p.num_qo_heads * nrot + (int64_t)p.num_kv_heads * (nk + nvec);
    // the kernel indexes units with 32 bits: split the tokens into launches of
    // fewer than 2^31 units
    const int64_t max_tokens = ((int64_t(1) << 31) - 1) / per_token;
    const int64_t row_q = (int64_t)p.num_qo_heads * p.head_dim * esz;
    const int64_t row_kv = (int64_t)p.num_kv_heads * p.head_dim * esz;
    for (int64_t t0 = 0; t0 < p.num_tokens; t0 += max_tokens) {
        RopeParams c = p;
        c.num_tokens = std::min(max_tokens, p.num_tokens - t0);
        c.query = p.query ? static_cast<uint8_t *>(p.query) + t0 * row_q : nullptr;
        c.key = static_cast<uint8_t *>(p.key) + t0 * row_kv;
        c.value = static_cast<const uint8_t *>(p.value) + t0 * row_kv;
        c.positions = p.positions + t0;
        c.slot_mapping = p.slot_mapping + t0;
        const int64_t total = c.num_tokens * per_token;
        auto go = [&](auto tag) -> cudaError_t {
            constexpr auto kern = decltype(tag)::value;
            kern<<<resident_grid<kern>(total), kThreads, 0, stream>>>(c);
            return cudaGetLastError();
        };
        cudaError_t e;
        if (dtype == PKV_F32) {
            if (neox)
                e = p.hnd ? go(std::integral_constant<decltype(&rope_reshape_cache_kernel<float, true, true>),
                                                      &rope_reshape_cache_kernel<float, true, true>>{})
                          : go(std::integral_constant<decltype(&rope_reshape_cache_kernel<float, true, false>),
                                                      &rope_reshape_cache_kernel<float, true, false>>{});
            else
                e = p.hnd ? go(std::integral_constant<decltype(&rope_reshape_cache_kernel<float, false, true>),
                                                      &rope_reshape_cache_kernel<float, false, true>>{})
                          : go(std::integral_constant<decltype(&rope_reshape_cache_kernel<float, false, false>),
                                                      &rope_reshape_cache_kernel<float, false, false>>{});
        } else {
            using B16 = __nv_bfloat16;
            if (neox)
                e = p.hnd ? go(std::integral_constant<decltype(&rope_reshape_cache_kernel<B16, true, true>),
                                                      &rope_reshape_cache_kernel<B16, true, true>>{})
                          : go(std::integral_constant<decltype(&rope_reshape_cache_kernel<B16, true, false>),
                                                      &rope_reshape_cache_kernel<B16, true, false>>{});
            else
                e = p.hnd ? go(std::integral_constant<decltype(&rope_reshape_cache_kernel<B16, false, true>),
                                                      &rope_reshape_cache_kernel<B16, false, true>>{})
                          : go(std::integral_constant<decltype(&rope_reshape_cache_kernel<B16, false, false>),
                                                      &rope_reshape_cache_kernel<B16, false, false>>{});
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pkv
