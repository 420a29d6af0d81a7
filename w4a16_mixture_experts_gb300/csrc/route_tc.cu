// Router logits for large batches on the tcgen05 tensor core.
//
// The router GEMM of "Running 125B MoE on Three 3090s - vLLM Optimization
// Edition", section 3.3 "MoE block (decode-05)" (the router stays BF16, model
// card "What is quantized"): partial[s][t][e] = sum over K split s of
// x[t][:] . Wr[e][:], read back and summed by route_topk_kernel.
//
// One CTA per (128 experts, 128 tokens, K split). Warp 0 lane 0 streams 64-wide
// K slices of both operands with 2-D TMA (128-byte swizzle, K-major) into a
// 4-stage ring; warp 1 issues tcgen05.mma (M=128 experts, N=128 tokens, K=16,
// both operands from shared memory) into a 128-column fp32 TMEM accumulator
// from one elected lane; then all four warps read their 32 TMEM lanes (32
// experts) and store the logits of every valid token column. Tokens past T
// read as zero (TMA out-of-bounds fill) and are not stored.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kRtStages = 4;
constexpr uint32_t kRtTile = 128 * 128;      // bytes of one 128 x 64 bf16 operand slice
constexpr uint32_t kRtSmem = kRtStages * 2 * kRtTile + 1024 + 256;

struct RouteTcParams {
    CUtensorMap tm_w;   // bf16 [E][H], box (64, 128), 128-byte swizzle
    CUtensorMap tm_x;   // bf16 [T][H], box (64, 128), 128-byte swizzle
    float *partial;     // f32 [ksplit][T][E]
    Ctrl *ctrl;
    int T, E, ksteps;   // ksteps: 64-wide K steps per split
    int ktot;           // 64-wide K steps in H
};

__device__ inline bool rt_elect() {
    uint32_t pred;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
    return pred != 0;
}

__global__ void __launch_bounds__(128, 1) route_logits_tc_kernel(const __grid_constant__ RouteTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                              // [stage] router rows
    uint8_t *sB = smem + kRtStages * kRtTile;        // [stage] token rows
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + 2 * kRtStages * kRtTile);
    uint64_t *empty = full + kRtStages;
    uint64_t *done = empty + kRtStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128, n0 = blockIdx.y * 128;
    const int k0 = blockIdx.z * p.ksteps;
    const int nk = min(p.ksteps, p.ktot - k0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRtStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_w) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_x) : "memory");
    }
    if (warp == 0) {
        tc::alloc(tmem_slot, 128);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            int i = 0;
            for (; i < nk; ++i) {
                const int s = i % kRtStages;
                if (!mbar_wait(&empty[s], ((i / kRtStages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], 2 * kRtTile);
                tma_load_2d(sA + s * kRtTile, &p.tm_w, (k0 + i) * 64, m0, &full[s]);
                tma_load_2d(sB + s * kRtTile, &p.tm_x, (k0 + i) * 64, n0, &full[s]);
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                for (int j = i > kRtStages ? i - kRtStages : 0; j < i; ++j)
                    mbar_wait(&full[j % kRtStages], (j / kRtStages) & 1);
            }
        }
        // the other lanes wait here, not in the spin on the accumulator below:
        // spinning beside the producing lane of their own warp held it back
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = tc::idesc_bf16(128, 128);
        for (int i = 0; i < nk; ++i) {
            const int s = i % kRtStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kRtStages) & 1))) {
                ok = false;
                break;
            }
            tc::fence_after();
            if (rt_elect()) {
                const uint64_t ad = tc::sdesc_sw128(sA + s * kRtTile), bd = tc::sdesc_sw128(sB + s * kRtTile);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ss(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (i | kk) != 0);
                tc::commit(&empty[s]);
            }
            __syncwarp();
        }
        if (ok && rt_elect()) tc::commit(done);
        __syncwarp();
        if (!ok && lane == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
    }

    // epilogue: TMEM lane = expert row of the tile, column = token (a split with no
    // K steps left, possible when ksplit does not divide the steps, stores zeros)
    const bool ready = nk <= 0 || mbar_wait(done, 0);
    if (ready) {
        tc::fence_after();
        const int e = m0 + 32 * warp + lane;
        float *dst = p.partial + (size_t)blockIdx.z * p.T * p.E + e;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
            if (nk > 0) {
                tc::ld_32x32b_x32(tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) v[u] = 0.f;
            }
            const int nu = min(32, p.T - (n0 + c0));
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (u < nu) dst[(size_t)(n0 + c0 + u) * p.E] = v[u];
        }
    } else if (threadIdx.x == 0) {
        set_error(p.ctrl, MOE_ERR_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::dealloc(tmem, 128);
}

}  // namespace

cudaError_t launch_route_logits_tc(const uint16_t *x, const uint16_t *wr, const moe_dims &d, float *partial,
                                   int ksplit, Ctrl *ctrl, cudaStream_t s) {
    RouteTcParams p;
    cudaError_t err = encode_tmap_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wr, (uint64_t)d.H, (uint64_t)d.E,
                                     (uint64_t)d.H * 2, 64u, 128u, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    err = encode_tmap_2d(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)d.H, (uint64_t)d.T,
                         (uint64_t)d.H * 2, 64u, 128u, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    if ((err = set_smem_once(reinterpret_cast<const void *>(route_logits_tc_kernel), (int)kRtSmem)) != cudaSuccess)
        return err;
    p.partial = partial;
    p.ctrl = ctrl;
    p.T = d.T;
    p.E = d.E;
    p.ktot = d.H / 64;
    p.ksteps = (p.ktot + ksplit - 1) / ksplit;
    dim3 grid(d.E / 128, (d.T + 127) / 128, ksplit);
    route_logits_tc_kernel<<<grid, 128, kRtSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
