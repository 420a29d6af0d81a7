// Router GEMM and the fused softmax / top-k / renormalisation.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
// "MoE block (decode-05)": the router GEMV, topk_softmax, and the two facts
// used here: with norm_topk_prob the full softmax denominator cancels, so a
// softmax over the k selected logits gives the weights; and top-k over keys
// that pack an order-preserving logit above (max - expert id) yields value
// and id in one max, ties going to the lower id. The keys here carry the
// fp32 logit (32 bits) instead of a bf16 one, so that ranking resolves gaps
// far below a bf16 ulp.
#include "common.cuh"
#include "kernels.cuh"
#include "route_dev.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Partial logits: partial[kb][t][e] = sum over K split kb of x[t][:] . Wr[e][:].
//
// One warp computes 16 experts x (8*NT) tokens over H/ksplit of K with
// mma.sync m16n8k16 (router rows as A, tokens as B). Both operands come
// straight from global memory as 16-byte chunks: a chunk of 8 consecutive K
// values of one row feeds two k-steps (values 0-3 to the first, 4-7 to the
// second), the same physical-K assignment being used for A and B, so the dot
// product is unchanged. Grid: (ceil(E/64), ksplit, ceil(T/(8*NT))), 4 warps.
template <int NT>
__device__ __forceinline__ void route_logits_tile(const uint16_t *__restrict__ x, const uint16_t *__restrict__ wr,
                                                  float *__restrict__ partial, int T, int H, int E) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int ksplit = gridDim.y, kb = blockIdx.y;
    const int kpart = H / ksplit;
    const int e0 = blockIdx.x * 64 + warp * 16;
    const int t0 = blockIdx.z * (8 * NT);
    if (e0 >= E) return;

    const int ra = e0 + g, rb = e0 + g + 8;
    const bool va = ra < E, vb = rb < E;
    const uint16_t *pa = wr + (size_t)(va ? ra : 0) * H + kb * kpart + 8 * tig;
    const uint16_t *pb = wr + (size_t)(vb ? rb : 0) * H + kb * kpart + 8 * tig;
    const uint16_t *px[NT];
    bool vx[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = t0 + 8 * nt + g;
        vx[nt] = t < T;
        px[nt] = x + (size_t)(vx[nt] ? t : 0) * H + kb * kpart + 8 * tig;
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 4
    for (int kk = 0; kk < kpart; kk += 32) {
        const uint4 A0 = va ? ld_nc_v4(pa + kk) : zero;
        const uint4 A1 = vb ? ld_nc_v4(pb + kk) : zero;
        uint4 B[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) B[nt] = vx[nt] ? ld_nc_v4(px[nt] + kk) : zero;
        const uint32_t a0[4] = {A0.x, A1.x, A0.y, A1.y};
        const uint32_t a1[4] = {A0.z, A1.z, A0.w, A1.w};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_bf16_16816(acc[nt], a0, B[nt].x, B[nt].y);
            mma_bf16_16816(acc[nt], a1, B[nt].z, B[nt].w);
        }
    }
    float *out = partial + (size_t)kb * T * E;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tc = t0 + 8 * nt + 2 * tig;
        if (tc < T) {
            if (va) out[(size_t)tc * E + ra] = acc[nt][0];
            if (vb) out[(size_t)tc * E + rb] = acc[nt][2];
        }
        if (tc + 1 < T) {
            if (va) out[(size_t)(tc + 1) * E + ra] = acc[nt][1];
            if (vb) out[(size_t)(tc + 1) * E + rb] = acc[nt][3];
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(128) route_logits_kernel(const uint16_t *__restrict__ x,
                                                           const uint16_t *__restrict__ wr,
                                                           float *__restrict__ partial, int T, int H, int E) {
    route_logits_tile<NT>(x, wr, partial, T, H, E);
}

// Top-k for T > 8 tokens: one CTA of four warps per token. Warp w takes the
// experts [w * ep, (w + 1) * ep), ep = ceil(E / 4) <= 256: lane l sums the
// K-split partial logits of experts lo + l, lo + l + 32, ... (all loads of a
// split in flight at once), adds the bias and forms the keys; the warp takes
// the k largest of its part, and warp 0 the k largest of the four parts'
// candidates.
constexpr int kTopkWarps = 4;

template <int N>
__device__ inline uint64_t part_topk(const float *__restrict__ row, size_t split_stride, int ksplit,
                                     const float *__restrict__ bias, int lo, int hi, int k, int lane) {
    float v[N];
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = 0.f;
    for (int s = 0; s < ksplit; ++s) {
        float u[N];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int e = lo + lane + 32 * i;
            u[i] = e < hi ? __ldcg(row + s * split_stride + e) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += u[i];
    }
    uint64_t key[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const int e = lo + lane + 32 * i;
        key[i] = e < hi ? topk_key(bias ? v[i] + bias[e] : v[i], e) : 0;
    }
    return warp_topk_n<N>(key, k, lane);
}

// With a shared expert (wg, the router's row E, not null) the CTA also forms the
// token's gate logit x[t] . wg (fp32) and writes slot k of the token's row of
// k + 1: expert E with weight sigmoid(gate).
__device__ inline float gate_dot_cta(const uint16_t *__restrict__ xrow, const uint16_t *__restrict__ wg, int H,
                                     float *s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc = 0.f;
    for (int c = 8 * threadIdx.x; c < H; c += 8 * blockDim.x) {
        const uint4 a = ld_nc_v4(xrow + c), b = ld_nc_v4(wg + c);
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc = fmaf(__uint_as_float(aa[j] << 16), __uint_as_float(bb[j] << 16), acc);
            acc = fmaf(__uint_as_float(aa[j] & 0xffff0000u), __uint_as_float(bb[j] & 0xffff0000u), acc);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) s_red[warp] = acc;
    __syncthreads();
    float g = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) g += s_red[i];
    return g;
}

__global__ void __launch_bounds__(32 * kTopkWarps) route_topk_kernel(const float *__restrict__ partial, int ksplit,
                                                                     const float *__restrict__ bias, int T, int E,
                                                                     int k, int32_t *__restrict__ ids,
                                                                     float *__restrict__ w,
                                                                     const uint16_t *__restrict__ x,
                                                                     const uint16_t *__restrict__ wg, int H) {
    __shared__ uint64_t s_cand[kTopkWarps][32];
    __shared__ float s_red[kTopkWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    const int ldk = wg ? k + 1 : k;
    if (wg) {
        const float g = gate_dot_cta(x + (size_t)t * H, wg, H, s_red);
        if (threadIdx.x == 0) {
            ids[(size_t)t * ldk + k] = E;
            w[(size_t)t * ldk + k] = sigmoidf_(g);
        }
    }
    const int ep = (E + kTopkWarps - 1) / kTopkWarps, lo = warp * ep, hi = min(E, lo + ep);
    const float *row = partial + (size_t)t * E;
    const size_t ss = (size_t)T * E;
    uint64_t mine;
    if (ep <= 64)
        mine = part_topk<2>(row, ss, ksplit, bias, lo, hi, k, lane);
    else if (ep <= 128)
        mine = part_topk<4>(row, ss, ksplit, bias, lo, hi, k, lane);
    else
        mine = part_topk<8>(row, ss, ksplit, bias, lo, hi, k, lane);
    s_cand[warp][lane] = lane < k ? mine : 0;
    __syncthreads();
    if (warp == 0) {
        uint64_t c[kTopkWarps];
#pragma unroll
        for (int q = 0; q < kTopkWarps; ++q) c[q] = s_cand[q][lane];
        topk_finish(warp_topk_n<kTopkWarps>(c, k, lane), k, lane, ids + (size_t)t * ldk, w + (size_t)t * ldk);
    }
}

// Small batches (T <= 8): logits and top-k in one launch, no K split over
// CTAs. CTA b computes the logits of experts 4b .. 4b + 3 for every token;
// the four warps of expert j (warps 4j .. 4j + 3) take a quarter of its router
// row each. Every lane first issues its 16-byte loads of the row (8 columns
// per load, 256 per pass of the warp, kRouteLoads passes at once); meanwhile
// the CTA copies the T x H activations into shared memory, so that no token
// costs a round trip of its own. Then fp32 FMAs, a warp sum, and the four
// quarter sums added in order. Logits (with the bias) go to partial[0]. Each
// CTA then counts itself on the control block's ticket (release); the CTA
// that completes the count acquires every other CTA's logits, loads all
// T x E of them into shared memory and selects: each token's experts are
// split over wpt warps (4 for T <= 4, else 2), each takes the k largest of
// its part, and one warp takes the k largest of their candidates. The ticket
// is reset for the next launch. The row arithmetic and the selection live in
// route_dev.cuh, shared with the decode kernel that routes itself.

inline size_t route_small_smem(const moe_dims &d) {
    const size_t xb = (size_t)d.T * d.H * 2, lb = (size_t)d.T * (d.E + 1) * 4;
    return xb > lb ? xb : lb;
}

// With a shared expert (gate != 0) the router has E + 1 rows, the last being the
// shared expert's gate: the CTAs compute all E + 1 logits (one GEMV, as on the
// pages), the selection takes the k largest of the first E, and slot k of each
// token's row of k + 1 is expert E with weight sigmoid(gate logit).
__global__ void __launch_bounds__(32 * kRouteWarps) route_small_kernel(const uint16_t *__restrict__ x,
                                                                       const uint16_t *__restrict__ wr,
                                                                       float *__restrict__ logits, int T, int H,
                                                                       int E, const float *__restrict__ bias, int k,
                                                                       int32_t *__restrict__ ids,
                                                                       float *__restrict__ w, Ctrl *ctrl, int gate) {
    // the activations [T][H] bf16; in the last CTA, then, the logits [T][E] f32
    extern __shared__ __align__(16) uint8_t s_raw[];
    __shared__ float s_part[kRouteWarps][kRouteInlineMaxT];
    __shared__ uint64_t s_cand[kRouteWarps][32];
    __shared__ int s_last;
    // the expert kernel behind this one may be launched now (its CTAs wait
    // for this grid's end themselves)
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Eg = E + gate;   // router rows, and the row stride of the logits
    const RouteQuarter rq = route_quarter(wr, blockIdx.x * 4 + (warp >> 2), Eg, H, warp & 3);
    uint4 wv[kRouteLoads];
    route_quarter_load(rq, rq.c_lo, lane, wv);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 *xs = reinterpret_cast<uint4 *>(s_raw);
    const int nx = T * H / 8;
    for (int i0 = threadIdx.x; i0 < nx; i0 += 4 * blockDim.x) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * blockDim.x;
            v[u] = i < nx ? ld_nc_v4(x + 8 * (size_t)i) : zero;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < nx) xs[i] = v[u];
        }
    }
    __syncthreads();
    float acc[kRouteInlineMaxT];
    route_quarter_dot(rq, xs, T, H, lane, wv, acc);
#pragma unroll
    for (int t = 0; t < kRouteInlineMaxT; ++t) {
        if (t >= T) break;
        if (lane == 0) s_part[warp][t] = acc[t];
    }
    __syncthreads();
    if (threadIdx.x < 4 * kRouteInlineMaxT) {
        const int jj = threadIdx.x / kRouteInlineMaxT, t = threadIdx.x % kRouteInlineMaxT;
        const int ee = blockIdx.x * 4 + jj;
        if (t < T && ee < Eg) logits[(size_t)t * Eg + ee] = route_logit(s_part, jj, t, bias, ee, E);
    }
    // the CTA barrier orders the logit stores before thread 0's release
    __syncthreads();
    if (threadIdx.x == 0) s_last = atom_acq_rel_add_u32(&ctrl->route_ticket, 1u) + 1 == gridDim.x;
    __syncthreads();
    if (!s_last) return;
    // the last CTA: all logits at once, then top-k
    float *s_logit = reinterpret_cast<float *>(s_raw);
    route_load_logits(s_logit, logits, T * Eg);
    __syncthreads();
    route_select(s_logit, T, E, k, gate, s_cand, ids, w);
    if (threadIdx.x == 0) ctrl->route_ticket = 0;
}

cudaError_t launch_route(const uint16_t *x, const uint16_t *wr, const float *bias, const moe_dims &d,
                         int32_t *ids, float *w, void *ws, cudaStream_t s, bool gate) {
    const WsLayout L = ws_layout(d);
    float *partial = ws_at<float>(ws, L.partial);
    const int ksplit = L.ksplit;
    // the shared expert's gate row follows the E router rows
    const uint16_t *wg = gate ? wr + (size_t)d.E * d.H : nullptr;
    if (router_tc(d)) {
        cudaError_t err = launch_route_logits_tc(x, wr, d, partial, ksplit, ws_at<Ctrl>(ws, L.ctrl), s);
        if (err != cudaSuccess) return err;
        route_topk_kernel<<<d.T, 32 * kTopkWarps, 0, s>>>(partial, ksplit, bias, d.T, d.E, d.k, ids, w, x, wg, d.H);
        return cudaGetLastError();
    }
    const int tt = d.T <= 64 ? d.T : 64;
    int nt = 1;
    while (8 * nt < tt) nt <<= 1;
    dim3 grid((d.E + 63) / 64, ksplit, (d.T + 8 * nt - 1) / (8 * nt));
    if (d.T <= kRouteInlineMaxT) {
        const size_t smem = route_small_smem(d);
        if (smem > 48 * 1024) {
            const cudaError_t err = set_smem_once(reinterpret_cast<const void *>(route_small_kernel),
                                                  kRouteInlineMaxT * 8192 * 2);
            if (err != cudaSuccess) return err;
        }
        // (a programmatic launch of this kernel behind the expert kernel was
        // measured slower at T = 4: its CTAs then start on the first SMs freed)
        const int rows = d.E + (gate ? 1 : 0);
        route_small_kernel<<<(rows + 3) / 4, 32 * kRouteWarps, smem, s>>>(x, wr, partial, d.T, d.H, d.E, bias, d.k,
                                                                           ids, w, ws_at<Ctrl>(ws, L.ctrl),
                                                                           gate ? 1 : 0);
        return cudaGetLastError();
    }
    switch (nt) {
        case 1: route_logits_kernel<1><<<grid, 128, 0, s>>>(x, wr, partial, d.T, d.H, d.E); break;
        case 2: route_logits_kernel<2><<<grid, 128, 0, s>>>(x, wr, partial, d.T, d.H, d.E); break;
        case 4: route_logits_kernel<4><<<grid, 128, 0, s>>>(x, wr, partial, d.T, d.H, d.E); break;
        default: route_logits_kernel<8><<<grid, 128, 0, s>>>(x, wr, partial, d.T, d.H, d.E); break;
    }
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    route_topk_kernel<<<d.T, 32 * kTopkWarps, 0, s>>>(partial, ksplit, bias, d.T, d.E, d.k, ids, w, x, wg, d.H);
    return cudaGetLastError();
}

}  // namespace moe
