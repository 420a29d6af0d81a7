// Token-to-expert permutation: histogram, prefix sum, stable scatter.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
// "MoE block": moe_align_block_size groups the (token, slot) assignments by
// expert for the expert GEMMs. Here no block padding is needed (the expert
// kernels take ragged counts), and the order inside an expert is made
// canonical: increasing assignment index a = t*k + j. That makes the slot
// of every assignment a pure function of topk_ids (a stable counting sort),
// so the result can be compared bit for bit.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Per-chunk histogram: chunk c covers assignments [c*kPermChunk, (c+1)*kPermChunk).
__global__ void __launch_bounds__(256) permute_hist_kernel(const int32_t *__restrict__ ids, int n, int E,
                                                           int32_t *__restrict__ chunk, Ctrl *ctrl) {
    __shared__ int32_t hist[kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int a0 = blockIdx.x * kPermChunk;
    for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
        const int a = a0 + i;
        if (a < n) {
            const int e = ids[a];
            if (e >= 0 && e < E)
                atomicAdd(&hist[e], 1);
            else
                set_error(ctrl, MOE_ERR_DEVICE);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk[(size_t)blockIdx.x * E + e] = hist[e];
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024);
// the block total goes to *total (a __shared__ variable).
__device__ inline int block_exclusive_scan(int v, int *total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int s = warp_sums[lane];
        int si = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, si, off);
            if (lane >= off) si += o;
        }
        warp_sums[lane] = si - s;
        if (lane == 31) *total = si;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

// One CTA of 1024 threads: per-expert totals and per-chunk bases, the
// expert offsets, the list of active experts, and the per-expert completion
// counters of the expert kernel cleared.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t *__restrict__ chunk, int nchunk, int E,
                                                            int32_t *__restrict__ counts,
                                                            int32_t *__restrict__ offsets,
                                                            int32_t *__restrict__ active,
                                                            uint32_t *__restrict__ done1, Ctrl *ctrl) {
    __shared__ int tot_all, tot_active;
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) {
        for (int c = 0; c < nchunk; ++c) {
            const int v = chunk[(size_t)c * E + e];
            chunk[(size_t)c * E + e] = total;
            total += v;
        }
    }
    const int off = block_exclusive_scan(e < E ? total : 0, &tot_all);
    const int act = block_exclusive_scan((e < E && total > 0) ? 1 : 0, &tot_active);
    if (e < E) {
        counts[e] = total;
        offsets[e] = off;
        for (int c = 0; c < nchunk; ++c) chunk[(size_t)c * E + e] += off;
        if (total > 0) active[act] = e;
        done1[(size_t)e * kCtrStride] = 0;
    }
    __syncthreads();
    if (e == 0) {
        offsets[E] = tot_all;
        ctrl->n_active = (uint32_t)tot_active;
    }
}

// Stable scatter: within a chunk, the rank of an assignment among earlier
// ones of the same expert = (same-expert entries in earlier warps) + (same-
// expert lanes below it in its warp, from __match_any_sync).
__global__ void __launch_bounds__(1024) permute_scatter_kernel(const int32_t *__restrict__ ids, int n, int E,
                                                               const int32_t *__restrict__ chunk,
                                                               int32_t *__restrict__ perm,
                                                               int32_t *__restrict__ inv) {
    extern __shared__ uint16_t wc[];   // [32 warps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wc[i] = 0;
    __syncthreads();
    const int a = blockIdx.x * kPermChunk + threadIdx.x;
    int e = -1;
    if (a < n) {
        e = ids[a];
        if (e < 0 || e >= E) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wc[warp * E + e] = (uint16_t)__popc(same);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        uint16_t run = 0;
        for (int w = 0; w < 32; ++w) {
            const uint16_t v = wc[w * E + x];
            wc[w * E + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (a < n) {
        if (e >= 0) {
            const int slot = chunk[(size_t)blockIdx.x * E + e] + wc[warp * E + e] + rank;
            perm[slot] = a;
            inv[a] = slot;
        } else {
            inv[a] = -1;
        }
    }
}

cudaError_t launch_permute(const int32_t *ids, const moe_dims &d, void *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(d);
    Ctrl *ctrl = ws_at<Ctrl>(ws, L.ctrl);
    const int n = d.T * d.k;
    int32_t *chunk = ws_at<int32_t>(ws, L.chunk);
    if (n > 0) {
        permute_hist_kernel<<<L.nchunk, 256, 0, s>>>(ids, n, d.E, chunk, ctrl);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    permute_scan_kernel<<<1, 1024, 0, s>>>(chunk, n > 0 ? L.nchunk : 0, d.E, ws_at<int32_t>(ws, L.counts),
                                           ws_at<int32_t>(ws, L.offsets), ws_at<int32_t>(ws, L.active),
                                           ws_at<uint32_t>(ws, L.done1), ctrl);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || n == 0) return err;
    const size_t smem = (size_t)32 * d.E * sizeof(uint16_t);
    err = set_smem_once(reinterpret_cast<const void *>(permute_scatter_kernel), 32 * kMaxE * (int)sizeof(uint16_t));
    if (err != cudaSuccess) return err;
    permute_scatter_kernel<<<L.nchunk, kPermChunk, smem, s>>>(ids, n, d.E, chunk, ws_at<int32_t>(ws, L.perm),
                                                              ws_at<int32_t>(ws, L.inv));
    return cudaGetLastError();
}

}  // namespace moe
