// Weighted combine of the per-slot expert outputs, and the stack epilogue.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
// "MoE block": moe_sum adds the k weighted expert outputs of each token.
// Here the weights are applied in slot order j = 0..k-1 in fp32, so the
// result does not depend on how the expert kernels were scheduled, and the
// bf16 rounding happens once. The stack variant adds the residual and
// rescales each row to unit RMS (no learned weight) before rounding.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

__device__ inline float4 weighted_sum4(const float *__restrict__ ybuf, const int32_t *__restrict__ inv,
                                       const float *__restrict__ topk_w, int t, int n, int H, int k) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int slot = inv[(size_t)t * k + j];
        if (slot < 0) continue;
        const float w = topk_w[(size_t)t * k + j];
        const float4 y = *reinterpret_cast<const float4 *>(ybuf + (size_t)slot * H + n);
        acc.x += w * y.x;
        acc.y += w * y.y;
        acc.z += w * y.z;
        acc.w += w * y.w;
    }
    return acc;
}

__device__ inline void store_bf16x4(uint16_t *dst, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(dst) = u;
}

// grid (ceil(H / 1024), T), 256 threads, 4 outputs per thread.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ ybuf,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ topk_w, int H, int k,
                                                      uint16_t *__restrict__ out) {
    const int t = blockIdx.y;
    const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (n >= H) return;
    store_bf16x4(out + (size_t)t * H + n, weighted_sum4(ybuf, inv, topk_w, t, n, H, k));
}

constexpr int kRmsMaxPer = 8;   // float4s per thread: H <= 256 * 4 * 8

// grid T, 256 threads: r = x + moe, next = bf16(r / sqrt(mean(r^2) + eps)).
__global__ void __launch_bounds__(256) combine_rms_kernel(const float *__restrict__ ybuf,
                                                          const int32_t *__restrict__ inv,
                                                          const float *__restrict__ topk_w,
                                                          const uint16_t *__restrict__ x, int H, int k,
                                                          float eps, uint16_t *__restrict__ next) {
    __shared__ float red[8];
    const int t = blockIdx.x;
    float4 r[kRmsMaxPer];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kRmsMaxPer; ++i) {
        const int n = (threadIdx.x + 256 * i) * 4;
        r[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n < H) {
            float4 v = weighted_sum4(ybuf, inv, topk_w, t, n, H, k);
            const uint2 xb = *reinterpret_cast<const uint2 *>(x + (size_t)t * H + n);
            v.x += __uint_as_float(xb.x << 16);
            v.y += __uint_as_float(xb.x & 0xffff0000u);
            v.z += __uint_as_float(xb.y << 16);
            v.w += __uint_as_float(xb.y & 0xffff0000u);
            r[i] = v;
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float scale = rsqrtf(tot / (float)H + eps);
#pragma unroll
    for (int i = 0; i < kRmsMaxPer; ++i) {
        const int n = (threadIdx.x + 256 * i) * 4;
        if (n < H) {
            float4 v = r[i];
            v.x *= scale;
            v.y *= scale;
            v.z *= scale;
            v.w *= scale;
            store_bf16x4(next + (size_t)t * H + n, v);
        }
    }
}

cudaError_t launch_combine(const ExpertArgs &a, const moe_dims &d, void *ws, uint16_t *out, uint16_t *next,
                           float eps, cudaStream_t s) {
    if (d.T == 0) return cudaSuccess;
    const WsLayout L = ws_layout(d);
    const float *ybuf = ws_at<float>(ws, L.ybuf);
    const int32_t *inv = ws_at<int32_t>(ws, L.inv);
    if (next) {
        combine_rms_kernel<<<d.T, 256, 0, s>>>(ybuf, inv, a.topk_w, a.x, d.H, d.k, eps, next);
    } else {
        dim3 grid((d.H + 1023) / 1024, d.T);
        combine_kernel<<<grid, 256, 0, s>>>(ybuf, inv, a.topk_w, d.H, d.k, out);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// INT4 packing (model card, "What is quantized": pack-quantized storage):
// word w of a row holds q[8w+i] + 8 in bits [4i, 4i+4).
__global__ void pack_int4_kernel(const int8_t *__restrict__ q, int64_t nwords, int32_t *__restrict__ packed,
                                 int32_t *__restrict__ bad) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nwords) return;
    const uint2 v = *reinterpret_cast<const uint2 *>(q + 8 * i);
    uint32_t word = 0;
    int nbad = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        int x = (int)(int8_t)((b < 4 ? v.x >> (8 * b) : v.y >> (8 * (b - 4))) & 0xffu);
        if (x < -8) { x = -8; ++nbad; }
        if (x > 7) { x = 7; ++nbad; }
        word |= (uint32_t)(x + 8) << (4 * b);
    }
    packed[i] = (int32_t)word;
    if (nbad && bad) atomicAdd(bad, nbad);
}

cudaError_t launch_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed, int32_t *bad,
                             cudaStream_t s) {
    const int64_t nwords = N * (K / 8);
    if (nwords == 0) return cudaSuccess;
    const int64_t blocks = (nwords + 255) / 256;
    pack_int4_kernel<<<(unsigned)blocks, 256, 0, s>>>(q, nwords, packed, bad);
    return cudaGetLastError();
}

}  // namespace moe
