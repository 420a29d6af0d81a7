// On-device INT4 quantiser: BF16 weights -> the packed storage of the experts.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 7
// "Putting MTP on the GPU": the MTP experts are quantised to INT4 by round to
// nearest, group size 128, symmetric, with a per-group search for the clip
// that minimises the squared error. The output is the format of the routed
// experts (model card, "What is quantized", group A): eight values q + 8 per
// int32 word, lowest nibble first, one bf16 scale per 128 values of a row.
//
// Per group of 128 values with amax = max |w| and clip c_j = (100 - j) / 100,
// j = 0 .. nclip - 1:
//   s_j   = bf16(c_j * amax / 7)            fp32 multiply, fp32 divide, bf16 RNE
//   q_i   = clamp(rint(w_i / s_j), -8, 7)   fp32 divide (IEEE), ties to even
//   err_j = sum_i (w_i - q_i * s_j)^2
// and the group keeps the j with the smallest err_j (the lowest j on a tie).
// These scale and code decisions are exact fp32 operations, so any
// implementation that performs them in fp32 reaches the same codes for a given
// j; only the choice of j can differ between implementations, by the rounding
// of the error sums. Here the sums are formed in fp32 in units of amax^2:
// err_j / amax^2 = (s_j / amax)^2 * sum_i (w_i / s_j - q_i)^2, the same ranking,
// which neither underflows for tiny weights nor overflows for large ones.
//
// One warp per group: lane l holds values 4l .. 4l + 3 (one 8-byte load), the
// warp forms amax, the lanes prepare one candidate scale each (32 at a time),
// then for each candidate the lanes' partial errors are summed by shuffles. The work is arithmetic (nclip quotients per value): the kernel is
// bound by the ALU, not by HBM. Lanes 2m and 2m + 1 together fill word m.
//
// The quotient w / s of the search is formed as w * RN(1 / s): within 2^-23
// relative of the correctly rounded division, i.e. within 2e-6 for the
// quotients here (|w / s| <= 7 / 0.01). rint of the two can differ only when
// the quotient lies that close to a half-integer, where either code leaves
// |w / s - q| within 2e-6 of 0.5: the group's error moves by less than 1e-5 of
// one value's share, far below the fp32 rounding of the sum, so the search
// ranks the candidates as the division would. The stored codes are computed
// with the division, bit for bit.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kQWarps = 8;

__device__ inline float bf16_round_f32(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ inline float clip_scale_dev(float amax, int j) {
    const float c = __fdiv_rn((float)(100 - j), 100.0f);
    const float t = __fmul_rn(c, amax);
    return bf16_round_f32(__fdiv_rn(t, 7.0f));
}

__device__ inline int quant_code(float w, float s) {
    if (s == 0.0f) return 0;
    const float q = rintf(__fdiv_rn(w, s));
    return (int)fminf(fmaxf(q, -8.0f), 7.0f);
}

__global__ void __launch_bounds__(kQWarps * 32) quantize_int4_kernel(const uint16_t *__restrict__ w, int64_t ngroups,
                                                                    int nclip, int32_t *__restrict__ packed,
                                                                    uint16_t *__restrict__ scales,
                                                                    int32_t *__restrict__ choice) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kQWarps;
    for (int64_t grp = (int64_t)blockIdx.x * kQWarps + (threadIdx.x >> 5); grp < ngroups; grp += nw) {
        // group grp = row n, group g: its 128 values are contiguous (K = 128 G per row)
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(w + grp * 128) + lane);
        const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        int best = 0;
        float best_err = 0.f;
        for (int jb = 0; jb < nclip; jb += 32) {
            // lane l prepares candidate jb + l (its scale, the reciprocal and (s / amax)^2,
            // the same for every lane), and the candidates are taken from their lanes in
            // turn: half of a candidate's instructions were these warp-uniform divisions
            const int jl = jb + lane;
            float ls = 0.f, linv = 0.f, lr2 = 0.f;
            if (jl < nclip) {
                ls = clip_scale_dev(amax, jl);
                if (ls != 0.0f) {
                    linv = __frcp_rn(ls);
                    const float ratio = __fdiv_rn(ls, amax);
                    lr2 = ratio * ratio;
                }
            }
            const int jn = nclip - jb < 32 ? nclip - jb : 32;
            for (int jj = 0; jj < jn; ++jj) {
                const int j = jb + jj;
                const float s = __shfl_sync(0xffffffffu, ls, jj);
                const float inv = __shfl_sync(0xffffffffu, linv, jj);
                const float r2 = __shfl_sync(0xffffffffu, lr2, jj);
                float e = 0.f;
                if (s != 0.0f) {
                    // in units of s: d = w/s - q, then scaled by (s / amax)^2
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float r = v[i] * inv;
                        const float d = r - fminf(fmaxf(rintf(r), -8.0f), 7.0f);
                        e = fmaf(d, d, e);
                    }
                    e *= r2;
                } else if (amax != 0.0f) {
                    // a scale that underflowed: every code is 0, the error is the group itself
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float d = __fdiv_rn(v[i], amax);
                        e = fmaf(d, d, e);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
                if (j == 0 || e < best_err) {
                    best = j;
                    best_err = e;
                }
            }
        }
        const float s = clip_scale_dev(amax, best);
        uint32_t half = 0;   // nibbles of this lane's 4 values
#pragma unroll
        for (int i = 0; i < 4; ++i) half |= (uint32_t)(quant_code(v[i], s) + 8) << (4 * i);
        const uint32_t hi = __shfl_down_sync(0xffffffffu, half, 1);
        if ((lane & 1) == 0) packed[grp * 16 + (lane >> 1)] = (int32_t)(half | (hi << 16));
        if (lane == 0) {
            const __nv_bfloat16 sb = __float2bfloat16_rn(s);
            scales[grp] = *reinterpret_cast<const uint16_t *>(&sb);
            if (choice) choice[grp] = best;
        }
    }
}

cudaError_t launch_quantize_int4(const uint16_t *w, int64_t N, int64_t K, int nclip, int32_t *packed,
                                 uint16_t *scales, int32_t *choice, cudaStream_t s) {
    const int64_t ngroups = N * (K / 128);
    if (ngroups == 0) return cudaSuccess;
    int64_t grid = (ngroups + kQWarps - 1) / kQWarps;
    const int64_t cap = 8LL * sm_count();   // a few waves of 8-warp CTAs; warps loop over groups
    if (grid > cap) grid = cap;
    quantize_int4_kernel<<<(unsigned)grid, kQWarps * 32, 0, s>>>(w, ngroups, nclip, packed, scales, choice);
    return cudaGetLastError();
}

}  // namespace moe
