// Decode-shaped expert path: W4A16 skinny GEMMs for a few tokens per expert.
//
// What it computes is the fused Marlin MoE of "Running 125B MoE on Three
// 3090s - vLLM Optimization Edition", section 3.3 "MoE block": per
// assignment g = W1[0:I] x, u = W1[I:2I] x, h = SiLU(g) * u (SiluAndMul),
// y = W2 h, on symmetric INT4 group-128 weights (model card, "What is
// quantized", group A). At decode the layer reads ~2.5 MB of packed weights
// per active expert and does a handful of FLOPs per byte, so the design is a
// byte pump:
//
//  * One persistent CTA per SM, 4 warps. Work is a flat list of tasks of
//    ~20 KB of packed weights each: gate_up tasks (8 gate rows + the matching
//    8 up rows of one expert, full K) first, then down tasks (64 output rows
//    of one expert, full K = I). Warps take tasks round-robin.
//  * Each warp streams its tasks' weights with 1-D bulk copies
//    (cp.async.bulk) into a private ring of shared-memory stages completed on
//    mbarriers, so every SM keeps tens of KB of HBM reads in flight.
//  * Weights are dequantised in registers straight into mma.sync m16n8k16
//    A fragments (bf16 holds q in [-8, 7] exactly); the group scale is applied
//    to each group's fp32 partial sum, so W = q * scale is never rounded.
//    Tokens are the N = 8 side; x is read from L2/L1 and byte-permuted to
//    match the nibble pairing of the A fragments.
//  * A down task of expert e waits (bounded, acquire) until all gate_up tasks
//    of e have published SiLU(g)*u, which they write in bf16 in the order the
//    down task's B fragments need. Gate_up tasks precede all down tasks in
//    every warp's list and all CTAs are co-resident, so the waits end.
//  * The down output of every (token, slot) goes to an fp32 buffer; a
//    separate combine kernel applies the routing weights in a fixed order.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kDecWarps = 4;
constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 227 * 1024;

struct DecodeParams {
    const uint16_t *x;
    const int32_t *w1p;
    const uint16_t *w1s;
    const int32_t *w2p;
    const uint16_t *w2s;
    const int32_t *offsets;
    const int32_t *perm;
    const int32_t *active;
    Ctrl *ctrl;
    uint32_t *done1;
    uint16_t *hbuf;
    float *ybuf;
    int H, I, k;
    int stages;
    uint32_t stage_bytes;
};

// Staged gate_up row stride: a row is H/2 bytes; when that is a multiple of
// 128 bytes, 64 bytes of padding put rows g and g+1 on opposite bank halves.
__host__ __device__ inline uint32_t p1_row_stride(int H) { return H / 2 + ((H / 128) % 2 == 0 ? 64 : 0); }
__host__ __device__ inline uint32_t p1_stage_bytes(int H) { return 16 * p1_row_stride(H) + 16 * (H / 128) * 2; }
__host__ __device__ inline uint32_t p2_stage_bytes(int I) { return 64 * (I / 2) + 64 * (I / 128) * 2; }

inline uint32_t decode_stage_bytes(const moe_dims &d) {
    uint32_t b = p1_stage_bytes(d.H);
    const uint32_t b2 = p2_stage_bytes(d.I);
    if (b2 > b) b = b2;
    return (uint32_t)align_up(b, 128);
}

inline int decode_stages(const moe_dims &d) {
    const uint32_t sb = decode_stage_bytes(d);
    int s = (int)(kSmemBudget / (kDecWarps * (sb + 8)));
    return s > kMaxStages ? kMaxStages : s;
}

bool decode_supported(const moe_dims &d) { return decode_stages(d) >= 1; }

__device__ inline void issue_task(const DecodeParams &p, int task, int total1, int tp1, int tp2, uint8_t *stage,
                                  uint64_t *bar, int lane) {
    if (task < total1) {
        const int a = task / tp1, r = task - a * tp1;
        const int e = p.active[a];
        const int G1 = p.H / 128;
        const uint32_t row_bytes = p.H / 2;
        const uint32_t rs = p1_row_stride(p.H);
        if (lane == 0) mbar_arrive_expect_tx(bar, 16 * row_bytes + 2 * 8 * G1 * 2);
        __syncwarp();
        if (lane < 16) {
            const int n = lane < 8 ? 8 * r + lane : p.I + 8 * r + (lane - 8);
            const char *src = reinterpret_cast<const char *>(p.w1p) + ((size_t)e * 2 * p.I + n) * row_bytes;
            bulk_g2s(stage + lane * rs, src, row_bytes, bar);
        } else if (lane < 18) {
            const int n0 = lane == 16 ? 8 * r : p.I + 8 * r;
            const uint16_t *src = p.w1s + ((size_t)e * 2 * p.I + n0) * G1;
            bulk_g2s(stage + 16 * rs + (lane - 16) * 16 * G1, src, 16 * G1, bar);
        }
    } else {
        const int t2 = task - total1;
        const int a = t2 / tp2, c = t2 - a * tp2;
        const int e = p.active[a];
        const int G2 = p.I / 128;
        const uint32_t rb = p.I / 2;
        if (lane == 0) mbar_arrive_expect_tx(bar, 64 * rb + 128 * G2);
        __syncwarp();
        if (lane == 0)
            bulk_g2s(stage, reinterpret_cast<const char *>(p.w2p) + ((size_t)e * p.H + 64 * c) * rb, 64 * rb, bar);
        else if (lane == 1)
            bulk_g2s(stage + 64 * rb, p.w2s + ((size_t)e * p.H + 64 * c) * G2, 128 * G2, bar);
    }
}

__device__ inline uint32_t word_of(const uint4 &v, int m) {
    return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// gate_up task: 8 gate rows i0..i0+7 (A rows 0-7) and up rows I+i0.. (A rows
// 8-15) against all tokens of the expert, 16 tokens per pass.
//
// Lane (g, tig) holds, for quantisation group q, the four words
// 4*tig..4*tig+3 of A rows g and g+8. Word m covers K = base..base+7 with
// base = 128q + 32tig + 8m; k-step 2m+h uses nibble pairs (2h, 2h+4) for the
// low fragment slots and (2h+1, 2h+5) for the high ones, so the B fragment
// of token g needs (x[base+2h], x[base+2h+4]) and (x[base+2h+1], x[base+2h+5]).
__device__ inline void run_gate_up(const DecodeParams &p, int task, int tp1, const uint8_t *stage, int lane) {
    const int a = task / tp1, r = task - a * tp1;
    const int e = p.active[a];
    const int s0 = p.offsets[e], ne = p.offsets[e + 1] - s0;
    const int g = lane >> 2, tig = lane & 3;
    const int G1 = p.H / 128;
    const uint32_t rs = p1_row_stride(p.H);
    const uint8_t *rg = stage + g * rs + 16 * tig;
    const uint8_t *ru = stage + (8 + g) * rs + 16 * tig;
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(stage + 16 * rs);
    const uint4 zero = make_uint4(0, 0, 0, 0);

    for (int np = 0; np < ne; np += 16) {
        const bool two = ne - np > 8;
        const uint16_t *px[2];
        bool vx[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int j = np + 8 * nt + g;
            vx[nt] = j < ne;
            const int tok = vx[nt] ? p.perm[s0 + j] / p.k : 0;
            px[nt] = p.x + (size_t)tok * p.H + 32 * tig;
        }
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        uint4 bn[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int m = 0; m < 4; ++m) bn[nt][m] = vx[nt] ? ld_nc_v4(px[nt] + 8 * m) : zero;

        for (int q = 0; q < G1; ++q) {
            uint4 bc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) bc[nt][m] = bn[nt][m];
            if (q + 1 < G1) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        bn[nt][m] = vx[nt] ? ld_nc_v4(px[nt] + 128 * (q + 1) + 8 * m) : zero;
            }
            const uint4 wg = lds_v4(rg + 64 * q), wu = lds_v4(ru + 64 * q);
            const float sg = bf16_bits_to_f32(sc[g * G1 + q]);
            const float su = bf16_bits_to_f32(sc[(8 + g) * G1 + q]);
            float c[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t xg = word_of(wg, m), xu = word_of(wu, m);
                const uint32_t a0[4] = {int4_pair(xg, 0), int4_pair(xu, 0), int4_pair(xg, 1), int4_pair(xu, 1)};
                const uint32_t a1[4] = {int4_pair(xg, 2), int4_pair(xu, 2), int4_pair(xg, 3), int4_pair(xu, 3)};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    if (nt == 1 && !two) continue;
                    const uint4 X = bc[nt][m];
                    mma_bf16_16816(c[nt], a0, __byte_perm(X.x, X.z, 0x5410), __byte_perm(X.x, X.z, 0x7632));
                    mma_bf16_16816(c[nt], a1, __byte_perm(X.y, X.w, 0x5410), __byte_perm(X.y, X.w, 0x7632));
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                acc[nt][0] += sg * c[nt][0];
                acc[nt][1] += sg * c[nt][1];
                acc[nt][2] += su * c[nt][2];
                acc[nt][3] += su * c[nt][3];
            }
        }
        // h for intermediate row 8r+g, tokens 2tig and 2tig+1 of each N tile.
        // Stored in chunk r at position 2*(g%4) + g/4: the order in which the
        // down task's fragments consume it.
        const int pos = 2 * (g & 3) + (g >> 2);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int j = np + 8 * nt + 2 * tig + b;
                if (j < ne) {
                    const float hv = silu(acc[nt][b]) * acc[nt][2 + b];
                    const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                    p.hbuf[(size_t)(s0 + j) * p.I + 8 * r + pos] = *reinterpret_cast<const uint16_t *>(&hb);
                }
            }
    }
}

// down task: output rows n0..n0+63 (4 m16 tiles) of expert e against the
// expert's tokens' h, 16 tokens per pass. Returns false if the wait for the
// expert's gate_up tasks gave up.
__device__ inline bool run_down(const DecodeParams &p, int t2, int tp1, int tp2, const uint8_t *stage, int lane) {
    const int a = t2 / tp2, c = t2 - a * tp2;
    const int e = p.active[a];
    const int s0 = p.offsets[e], ne = p.offsets[e + 1] - s0;
    const int g = lane >> 2, tig = lane & 3;
    const int G2 = p.I / 128;
    const uint32_t rb = p.I / 2;
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(stage + 64 * rb);
    const uint4 zero = make_uint4(0, 0, 0, 0);

    uint32_t ok = 1;
    if (lane == 0) {
        uint32_t i = 0;
        while (ld_acquire_u32(&p.done1[a]) < (uint32_t)tp1) {
            if (++i > kSpinLimit) {
                ok = 0;
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) return false;

    for (int np = 0; np < ne; np += 16) {
        const bool two = ne - np > 8;
        const uint16_t *ph[2];
        bool vh[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int j = np + 8 * nt + g;
            vh[nt] = j < ne;
            ph[nt] = p.hbuf + (size_t)(s0 + (vh[nt] ? j : 0)) * p.I + 32 * tig;
        }
        float acc[4][2][4];
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) acc[s][nt][0] = acc[s][nt][1] = acc[s][nt][2] = acc[s][nt][3] = 0.f;

        for (int q = 0; q < G2; ++q) {
            uint4 Y[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) Y[nt][m] = vh[nt] ? ld_cg_v4(ph[nt] + 128 * q + 8 * m) : zero;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int R = 16 * s + g;
                const uint4 w0 = lds_v4(stage + R * rb + 64 * q + 16 * tig);
                const uint4 w1 = lds_v4(stage + (R + 8) * rb + 64 * q + 16 * tig);
                const float s0v = bf16_bits_to_f32(sc[R * G2 + q]);
                const float s1v = bf16_bits_to_f32(sc[(R + 8) * G2 + q]);
                float cc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) cc[nt][0] = cc[nt][1] = cc[nt][2] = cc[nt][3] = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t x0 = word_of(w0, m), x1 = word_of(w1, m);
                    const uint32_t a0[4] = {int4_pair(x0, 0), int4_pair(x1, 0), int4_pair(x0, 1), int4_pair(x1, 1)};
                    const uint32_t a1[4] = {int4_pair(x0, 2), int4_pair(x1, 2), int4_pair(x0, 3), int4_pair(x1, 3)};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        if (nt == 1 && !two) continue;
                        mma_bf16_16816(cc[nt], a0, Y[nt][m].x, Y[nt][m].y);
                        mma_bf16_16816(cc[nt], a1, Y[nt][m].z, Y[nt][m].w);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    acc[s][nt][0] += s0v * cc[nt][0];
                    acc[s][nt][1] += s0v * cc[nt][1];
                    acc[s][nt][2] += s1v * cc[nt][2];
                    acc[s][nt][3] += s1v * cc[nt][3];
                }
            }
        }
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int j = np + 8 * nt + 2 * tig + b;
                    if (j < ne) {
                        float *yr = p.ybuf + (size_t)(s0 + j) * p.H + 64 * c + 16 * s + g;
                        yr[0] = acc[s][nt][b];
                        yr[8] = acc[s][nt][2 + b];
                    }
                }
    }
    return true;
}

__global__ void __launch_bounds__(kDecWarps * 32, 1) decode_experts_kernel(DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages;
    uint8_t *wbase = smem + (size_t)warp * S * p.stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kDecWarps * S * p.stage_bytes) + warp * S;

    const int n_active = (int)p.ctrl->n_active;
    const int tp1 = p.I / 8, tp2 = p.H / 64;
    const int total1 = n_active * tp1;
    const int total = total1 + n_active * tp2;
    const int gw = blockIdx.x * kDecWarps + warp, nw = gridDim.x * kDecWarps;

    if (lane == 0)
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    __syncwarp();

    for (int i = 0; i < S; ++i) {
        const int task = gw + i * nw;
        if (task < total) issue_task(p, task, total1, tp1, tp2, wbase + (size_t)i * p.stage_bytes, &bars[i], lane);
    }

    int li = 0;
    for (int task = gw; task < total; task += nw, ++li) {
        const int st = li % S;
        const uint32_t par = (uint32_t)(li / S) & 1u;
        uint8_t *stage = wbase + (size_t)st * p.stage_bytes;
        if (!mbar_wait(&bars[st], par)) {
            // A copy did not land in time: record it, give the outstanding
            // copies one more bounded wait, and stop.
            if (lane == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
            for (int i = 0; i < S; ++i) {
                const int lj = li + i;
                if (gw + lj * nw < total) mbar_wait(&bars[lj % S], (uint32_t)(lj / S) & 1u);
            }
            return;
        }
        if (task < total1) {
            run_gate_up(p, task, tp1, stage, lane);
            __threadfence();
            __syncwarp();
            if (lane == 0) red_release_add_u32(&p.done1[task / tp1], 1u);
        } else {
            run_down(p, task - total1, tp1, tp2, stage, lane);
        }
        __syncwarp();
        const int nxt = task + S * nw;
        if (nxt < total) {
            fence_proxy_async_smem();
            issue_task(p, nxt, total1, tp1, tp2, stage, &bars[st], lane);
        }
    }
}

cudaError_t launch_decode_experts(const ExpertArgs &a, const moe_dims &d, void *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(d);
    DecodeParams p;
    p.x = a.x;
    p.w1p = a.w1p;
    p.w1s = a.w1s;
    p.w2p = a.w2p;
    p.w2s = a.w2s;
    p.offsets = ws_at<int32_t>(ws, L.offsets);
    p.perm = ws_at<int32_t>(ws, L.perm);
    p.active = ws_at<int32_t>(ws, L.active);
    p.ctrl = ws_at<Ctrl>(ws, L.ctrl);
    p.done1 = ws_at<uint32_t>(ws, L.done1);
    p.hbuf = ws_at<uint16_t>(ws, L.hbuf);
    p.ybuf = ws_at<float>(ws, L.ybuf);
    p.H = d.H;
    p.I = d.I;
    p.k = d.k;
    p.stages = decode_stages(d);
    p.stage_bytes = decode_stage_bytes(d);
    if (p.stages < 1) return cudaErrorInvalidValue;
    const size_t smem = (size_t)kDecWarps * p.stages * (p.stage_bytes + 8);
    cudaError_t err = set_smem_once(reinterpret_cast<const void *>(decode_experts_kernel), kSmemBudget);
    if (err != cudaSuccess) return err;

    // Upper bound on the task count: active experts <= min(E, T*k).
    const long long max_active = (long long)d.T * d.k < d.E ? (long long)d.T * d.k : d.E;
    const long long max_tasks = max_active * (d.I / 8 + d.H / 64);
    long long grid = (max_tasks + kDecWarps - 1) / kDecWarps;
    if (grid > sm_count()) grid = sm_count();
    if (grid < 1) grid = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_experts_kernel, p);
}

}  // namespace moe
