// Router pieces shared by the small-batch router (route.cu) and the decode
// kernel that runs the router itself (decode_fused.cu), so that both compute
// the same logits and select the same experts with the same weights, bit for
// bit.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
// "MoE block (decode-05)": the router GEMV, topk_softmax with norm_topk_prob
// (a softmax over the k selected logits equals the renormalised full
// softmax), and the top-k key that packs an order-preserving logit above
// (max - expert id), so that one maximum yields value and id and ties go to
// the lower id. The keys here carry the fp32 logit instead of a bf16 one.
#pragma once
#include "common.cuh"

namespace moe {

// Order-preserving map of an fp32 value onto uint32.
__device__ inline uint32_t f32_order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ inline float f32_from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---------------------------------------------------------------------------
// Top-k: keys pack an order key of the fp32 logit above 0xffffffff - id, so
// keys are unique and one maximum gives value and id (ties to the lower id).
// A warp's k largest: every lane sorts its keys, then k rounds of a two-step
// warp max with redux.sync (first the logit half, then the id half among the
// lanes holding that logit); the lane that held the maximum moves to its next
// key. Weights: softmax over the selected logits in fp32.
__device__ inline uint64_t warp_max_key(uint64_t m) {
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(m >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(m >> 32) == hi ? (uint32_t)m : 0u);
    return ((uint64_t)hi << 32) | lo;
}

// Size-generic forms for lanes holding N keys each (N a power of two): sort,
// k rounds of the heads' warp maximum (lane j < k ends with the j-th largest),
// and the softmax over the selected logits with the writes.
template <int N>
__device__ inline void sort_desc_n(uint64_t (&key)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1)
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int l = i ^ stride;
                if (l > i) {
                    const bool up = (i & size) != 0;
                    const uint64_t a = key[i], b = key[l];
                    if (up ? a > b : a < b) {
                        key[i] = b;
                        key[l] = a;
                    }
                }
            }
}

template <int N>
__device__ inline uint64_t warp_topk_n(uint64_t (&key)[N], int k, int lane) {
    sort_desc_n<N>(key);
    uint64_t mine = 0;
    for (int j = 0; j < k; ++j) {
        const uint64_t m = warp_max_key(key[0]);
        if (key[0] == m) {
#pragma unroll
            for (int i = 0; i + 1 < N; ++i) key[i] = key[i + 1];
            key[N - 1] = 0;
        }
        if (lane == j) mine = m;
    }
    return mine;
}

__device__ inline void topk_finish(uint64_t mine, int k, int lane, int32_t *ids_row, float *w_row) {
    const float lmax = f32_from_order_key((uint32_t)(__shfl_sync(0xffffffffu, mine, 0) >> 32));
    const float l = f32_from_order_key((uint32_t)(mine >> 32));
    const float p = lane < k ? expf(l - lmax) : 0.f;
    float z = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane < k) {
        ids_row[lane] = (int32_t)(0xffffffffu - (uint32_t)(mine & 0xffffffffu));
        w_row[lane] = p / z;
    }
}

__device__ inline uint64_t topk_key(float logit, int e) {
    return ((uint64_t)f32_order_key(logit) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
}


__device__ inline float sigmoidf_(float g) { return 1.0f / (1.0f + expf(-g)); }


constexpr int kRouteInlineMaxT = 8;
constexpr int kRouteWarps = 16;
constexpr int kRouteLoads = 3;   // 16-byte loads per lane in flight (a quarter row of H <= 3072 in one pass)
constexpr int kRouteMaxWpt = 4;

// ---- the small-batch router's logits ------------------------------------------
// Four warps per router row, warp q (= warp % 4) taking the quarter
// [q H / 4, (q + 1) H / 4) of it; lane l reads columns c_lo + 256 i + 8 l, 16
// bytes each, kRouteLoads at a time. Rows at or past Eg read row 0 and are
// never stored.
struct RouteQuarter {
    const uint16_t *row;
    bool valid;
    int c_lo, c_hi;
};

__device__ inline RouteQuarter route_quarter(const uint16_t *wr, int e, int Eg, int H, int q) {
    RouteQuarter r;
    r.valid = e < Eg;
    r.row = wr + (size_t)(r.valid ? e : 0) * H;
    r.c_lo = q * (H / 4);
    r.c_hi = r.c_lo + H / 4;
    return r;
}

// The loads of the pass that starts at column c0.
__device__ inline void route_quarter_load(const RouteQuarter &r, int c0, int lane, uint4 (&wv)[kRouteLoads]) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kRouteLoads; ++i) {
        const int c = c0 + 256 * i + 8 * lane;
        wv[i] = r.valid && c < r.c_hi ? ld_nc_v4(r.row + c) : zero;
    }
}

// acc[t] = the quarter's dot product with token t's activations (xs: the T x H
// activations, row-major bf16, in shared memory), summed over the warp, for
// t < T; wv holds the first pass's loads. fp32 FMAs in column order within a
// lane, then a butterfly sum.
__device__ inline void route_quarter_dot(const RouteQuarter &r, const uint4 *xs, int T, int H, int lane,
                                         uint4 (&wv)[kRouteLoads], float (&acc)[kRouteInlineMaxT]) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < kRouteInlineMaxT; ++t) acc[t] = 0.f;
    for (int c0 = r.c_lo; c0 < r.c_hi; c0 += 256 * kRouteLoads) {
        if (c0 != r.c_lo) route_quarter_load(r, c0, lane, wv);
#pragma unroll
        for (int t = 0; t < kRouteInlineMaxT; ++t) {
            if (t >= T) break;
#pragma unroll
            for (int i = 0; i < kRouteLoads; ++i) {
                const int c = c0 + 256 * i + 8 * lane;
                const uint4 xv = c < r.c_hi ? xs[((size_t)t * H + c) / 8] : zero;
                const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[t] = fmaf(__uint_as_float(ww[j] << 16), __uint_as_float(xx[j] << 16), acc[t]);
                    acc[t] = fmaf(__uint_as_float(ww[j] & 0xffff0000u), __uint_as_float(xx[j] & 0xffff0000u), acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kRouteInlineMaxT; ++t) {
        if (t >= T) break;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
}

// Logit of row e (the jj-th of the CTA's four) for token t from the quarter
// sums of its four warps, added in quarter order, plus the bias of a routed row.
__device__ inline float route_logit(const float (*s_part)[kRouteInlineMaxT], int jj, int t, const float *bias,
                                    int e, int E) {
    const float v = ((s_part[4 * jj][t] + s_part[4 * jj + 1][t]) + s_part[4 * jj + 2][t]) + s_part[4 * jj + 3][t];
    return bias && e < E ? v + bias[e] : v;
}

// All n logits into shared memory by every thread of the CTA, eight loads per
// thread in flight (L2, not L1: other CTAs wrote them).
__device__ inline void route_load_logits(float *s_logit, const float *logits, int n) {
    for (int i0 = 0; i0 < n; i0 += 8 * blockDim.x) {
        float lv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x + threadIdx.x;
            lv[u] = i < n ? __ldcg(logits + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * blockDim.x + threadIdx.x;
            if (i < n) s_logit[i] = lv[u];
        }
    }
}

// ---- the small-batch router's selection --------------------------------------
// By all kRouteWarps warps of a CTA (it holds a CTA barrier): the k largest of
// each token's E routed logits (s_logit: T rows of Eg = E + gate f32 values,
// any memory the CTA can read), each token's experts split over wpt warps (4
// for T <= 4, else 2), each warp taking the k largest of its part and one warp
// the k largest of their candidates; then the softmax over the selected logits.
// Row t of ids / w (ldk = k + gate values, any memory) receives the ids in
// order of descending logit and their weights; with a shared expert (gate = 1)
// slot k holds expert E with weight sigmoid(gate logit). s_cand: kRouteWarps
// x 32 keys of scratch in shared memory.
__device__ inline void route_select(const float *s_logit, int T, int E, int k, int gate, uint64_t (*s_cand)[32],
                                    int32_t *ids, float *w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Eg = E + gate;
    const int wpt = T <= kRouteWarps / kRouteMaxWpt ? kRouteMaxWpt : kRouteWarps / kRouteInlineMaxT;
    const int t = warp / wpt, part = warp % wpt;
    const int ep = (E + wpt - 1) / wpt, lo = part * ep, hi = min(E, lo + ep);
    if (t < T) {
        uint64_t mine;
        if (ep <= 128) {
            uint64_t key[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int ee = lo + lane + 32 * i;
                key[i] = ee < hi ? topk_key(s_logit[t * Eg + ee], ee) : 0;
            }
            mine = warp_topk_n<4>(key, k, lane);
        } else if (ep <= 256) {
            uint64_t key[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ee = lo + lane + 32 * i;
                key[i] = ee < hi ? topk_key(s_logit[t * Eg + ee], ee) : 0;
            }
            mine = warp_topk_n<8>(key, k, lane);
        } else {
            uint64_t key[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int ee = lo + lane + 32 * i;
                key[i] = ee < hi ? topk_key(s_logit[t * Eg + ee], ee) : 0;
            }
            mine = warp_topk_n<16>(key, k, lane);
        }
        s_cand[warp][lane] = lane < k ? mine : 0;
    }
    __syncthreads();
    if (t < T && part == 0) {
        uint64_t c[kRouteMaxWpt];
#pragma unroll
        for (int q = 0; q < kRouteMaxWpt; ++q) c[q] = q < wpt ? s_cand[warp + q][lane] : 0;
        const uint64_t mine = warp_topk_n<kRouteMaxWpt>(c, k, lane);
        const int ldk = k + gate;
        topk_finish(mine, k, lane, ids + (size_t)t * ldk, w + (size_t)t * ldk);
        if (gate && lane == 0) {
            ids[(size_t)t * ldk + k] = E;
            w[(size_t)t * ldk + k] = sigmoidf_(s_logit[t * Eg + E]);
        }
    }
}

}  // namespace moe
