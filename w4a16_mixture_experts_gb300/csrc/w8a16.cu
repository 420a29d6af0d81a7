// W8A16 linear layers: y = x . W^T with INT8 pack-quantized weights.
//
// "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
// "Hyper-connection (decode-04)": compressed-tensors INT8 pack-quantized puts
// four values in each int32 word, least significant byte first, each stored
// as q + 128, so the words are read as they are stored (no repacking). The
// pages serve decode with INT8 GEMVs and batches over 4 tokens with a W8A16
// GEMM. Groups (model card, "What is quantized"): C = INT8 gs64
// (hyper-connection mixers), D = INT8 gs128 (lm_head and others).
//
// Dequantisation, exact in bf16 and in natural K order: prmt places bytes
// (b0, b1) (or (b2, b3)) in the two 16-bit halves of a register; then
//   lo = (v & 0x007F007F) | 0x43004300   -> bf16 128 + (b & 127)
//   hi = (v & 0x00800080) ^ 0xC380C380   -> bf16 -256, or -128 if b >= 128
// and one bf16x2 add gives b - 128 = q exactly (all values are integers of
// magnitude <= 256). Eight instructions per word of four weights.
//
// Decode (T <= 8): a GEMV that streams the weights from HBM. A warp owns 16
// rows; per step every lane loads 16 bytes (64 values) of two rows, g and
// g + 8, a step ahead of use; the rows are the M = 16 side of
// mma.sync m16n8k16 and the tokens the N = 8 side; each group's fp32 partial
// product is scaled by the group's bf16 scale. x is staged once per CTA in
// shared memory. Layers with few rows (the hyper-connection mixer [320, 10240]
// has 20 blocks of 16 rows) split K: the 16 warps of a CTA take 16 / S blocks,
// S warps each on consecutive ranges of whole scale groups, and the S partial
// results of a block are summed in shared memory in a fixed order.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kW8Warps = 16;
constexpr int kW8Ahead = 1;          // 16-byte weight loads per row issued ahead of use per lane

// Weight loads: read once (non-coherent path), each asking L2 to fetch the
// 256-byte run around it, so that the next loads of the row hit L2. Measured on
// the lm_head [248320, 2560]: with one load ahead and this hint 5.2 TB/s;
// with four loads ahead (spilling at the register budget of two CTAs a SM) and
// no hint 3.8 TB/s.
__device__ __forceinline__ uint4 ld_w8(const void *p) {
    uint4 v;
    asm("ld.global.nc.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
constexpr int kW8MaxSmem = 196608;   // bytes of staged x (T x K bf16)

// Bytes (b_lo, b_hi) of w -> bf16x2 of (b - 128) each. sel picks the bytes
// (0x4140: bytes 0, 1; 0x4342: bytes 2, 3).
__device__ __forceinline__ uint32_t int8_pair(uint32_t w, uint32_t sel) {
    const uint32_t v = __byte_perm(w, 0u, sel);
    uint32_t lo, hi;
    asm("lop3.b32 %0, %1, 0x007F007F, %2, 0xEA;" : "=r"(lo) : "r"(v), "r"(0x43004300u));   // (a & b) | c
    asm("lop3.b32 %0, %1, 0x00800080, %2, 0x6A;" : "=r"(hi) : "r"(v), "r"(0xC380C380u));   // (a & b) ^ c
    __nv_bfloat162 r = __hadd2(*reinterpret_cast<__nv_bfloat162 *>(&lo), *reinterpret_cast<__nv_bfloat162 *>(&hi));
    return *reinterpret_cast<uint32_t *>(&r);
}

struct W8Params {
    const uint16_t *x;      // bf16 [T][K]
    const uint32_t *w;      // int32 [N][K/4]
    const uint16_t *s;      // bf16 [N][K/gs]
    uint16_t *y;            // bf16 [T][N]
    int T, N, K, gs;
    int split;              // warps per 16-row block (a power of two <= kW8Warps)
};

// One warp per 16-row block (grid-stride over blocks). In each 64-wide K step,
// lane (g, tig) loads 16 bytes of rows g and g + 8: words 4 tig .. 4 tig + 3 of
// the step, K = 64 st + 16 tig + 4 m + 0..3 for word m. Word m feeds k-step m:
// A slots (2 tig, 2 tig + 1) <- its values 0, 1 and (2 tig + 8, 2 tig + 9) <-
// values 2, 3; the B fragment of token g is x[g] at the same four K in the
// same order, one 8-byte shared load. (The four lanes of a row cover each
// k-step's 16 K values once; A and B agree, so the products are the dot
// product's.) x rows are staged with a stride of K + 8, so that the eight
// tokens' loads fall in different banks.
__global__ void __launch_bounds__(kW8Warps * 32, 2) w8a16_gemv_kernel(const __grid_constant__ W8Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tig = lane & 3;
    // x staged once per CTA: [T][K + 8] bf16, 16-byte chunks
    const int kp = p.K + 8;
    {
        const int cpr = p.K / 8, nch = p.T * cpr;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        for (int i = threadIdx.x; i < nch; i += blockDim.x) {
            const int t = i / cpr, c = i - t * cpr;
            dst[t * (kp / 8) + c] = __ldg(src + i);
        }
    }
    __syncthreads();
    const uint16_t *xs = reinterpret_cast<const uint16_t *>(smem);
    float4 *part = reinterpret_cast<float4 *>(smem + (size_t)p.T * kp * 2);   // [kW8Warps][32] partial sums
    const int tok = g < p.T ? g : 0;   // columns past T read token 0 and are not stored
    const int steps_per_group = p.gs / 64;
    const int G = p.K / p.gs;
    const int nblocks = (p.N + 15) / 16;
    const int S = p.split, bpc = kW8Warps / S;    // warps per block, blocks per CTA pass
    const int piece = warp % S;
    // this warp's K range: scale groups [G piece / S, G (piece + 1) / S)
    const int st_lo = (G * piece / S) * steps_per_group, st_hi = (G * (piece + 1) / S) * steps_per_group;
    const uint4 zero4 = make_uint4(0, 0, 0, 0);
    const int npass = (nblocks + bpc - 1) / bpc;
    for (int pass = blockIdx.x; pass < npass; pass += gridDim.x) {
        const int blk = pass * bpc + warp / S;
        const int r0 = blk * 16 + g, r1 = r0 + 8;
        const bool v0 = r0 < p.N, v1 = r1 < p.N;
        const uint4 *w0 = reinterpret_cast<const uint4 *>(p.w + (size_t)(v0 ? r0 : 0) * (p.K / 4)) + tig;
        const uint4 *w1 = reinterpret_cast<const uint4 *>(p.w + (size_t)(v1 ? r1 : 0) * (p.K / 4)) + tig;
        uint4 ring0[kW8Ahead], ring1[kW8Ahead];
#pragma unroll
        for (int a = 0; a < kW8Ahead; ++a) {
            ring0[a] = st_lo + a < st_hi && v0 ? ld_w8(w0 + 4 * (st_lo + a)) : zero4;
            ring1[a] = st_lo + a < st_hi && v1 ? ld_w8(w1 + 4 * (st_lo + a)) : zero4;
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float cc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int st0 = st_lo; st0 < st_hi; st0 += kW8Ahead) {
#pragma unroll
            for (int a = 0; a < kW8Ahead; ++a) {
                const int st = st0 + a;
                if (st < st_hi) {
                    const uint4 q0 = ring0[a], q1 = ring1[a];
                    if (st + kW8Ahead < st_hi) {
                        ring0[a] = v0 ? ld_w8(w0 + 4 * (st + kW8Ahead)) : zero4;
                        ring1[a] = v1 ? ld_w8(w1 + 4 * (st + kW8Ahead)) : zero4;
                    }
                    const uint32_t wa[4] = {q0.x, q0.y, q0.z, q0.w}, wb[4] = {q1.x, q1.y, q1.z, q1.w};
                    const uint16_t *xr = xs + (size_t)tok * kp + 64 * st + 16 * tig;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint2 xv = *reinterpret_cast<const uint2 *>(xr + 4 * m);
                        const uint32_t af[4] = {int8_pair(wa[m], 0x4140), int8_pair(wb[m], 0x4140),
                                                int8_pair(wa[m], 0x4342), int8_pair(wb[m], 0x4342)};
                        mma_bf16_16816(cc, af, xv.x, xv.y);
                    }
                    // the group ends: scale its partial products into the accumulator
                    if ((st + 1) % steps_per_group == 0) {
                        const int grp = st / steps_per_group;
                        const float s0 = v0 ? bf16_bits_to_f32(__ldg(p.s + (size_t)r0 * G + grp)) : 0.f;
                        const float s1 = v1 ? bf16_bits_to_f32(__ldg(p.s + (size_t)r1 * G + grp)) : 0.f;
                        acc[0] = fmaf(s0, cc[0], acc[0]);
                        acc[1] = fmaf(s0, cc[1], acc[1]);
                        acc[2] = fmaf(s1, cc[2], acc[2]);
                        acc[3] = fmaf(s1, cc[3], acc[3]);
                        cc[0] = cc[1] = cc[2] = cc[3] = 0.f;
                    }
                }
            }
        }
        // the block's S partial results, summed in piece order by the warp of piece 0
        if (S > 1) {
            part[warp * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            __syncthreads();
            if (piece == 0) {
#pragma unroll 1
                for (int j = 1; j < S; ++j) {
                    const float4 o = part[(warp + j) * 32 + lane];
                    acc[0] += o.x, acc[1] += o.y, acc[2] += o.z, acc[3] += o.w;
                }
            }
            __syncthreads();
            if (piece != 0) continue;
        }
        // acc: (row g, tokens 2 tig, 2 tig + 1), (row g + 8, same tokens)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int t = 2 * tig + b;
            if (t < p.T) {
                if (v0) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(acc[b]);
                    p.y[(size_t)t * p.N + r0] = *reinterpret_cast<const uint16_t *>(&h);
                }
                if (v1) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(acc[2 + b]);
                    p.y[(size_t)t * p.N + r1] = *reinterpret_cast<const uint16_t *>(&h);
                }
            }
        }
    }
}

bool w8a16_gemv_supported(int T, int K) { return T >= 1 && T <= 8 && (size_t)T * (K + 8) * 2 <= kW8MaxSmem; }

// Warps per 16-row block: enough blocks x warps to give every SM's warps work,
// never more pieces than scale groups.
static int w8a16_split(int N, int K, int gs) {
    const int nblocks = (N + 15) / 16, G = K / gs;
    int S = 1;
    while (S < kW8Warps && (long long)nblocks * S < 2LL * kW8Warps * sm_count() && 2 * S <= G) S *= 2;
    return S;
}

cudaError_t launch_w8a16(const uint16_t *x, const int32_t *w, const uint16_t *s, int gs, uint16_t *y, int T, int N,
                         int K, cudaStream_t st) {
    if (T == 0 || N == 0) return cudaSuccess;
    if (!w8a16_gemv_supported(T, K)) return cudaErrorInvalidValue;
    const int S = w8a16_split(N, K, gs);
    W8Params p{x, reinterpret_cast<const uint32_t *>(w), s, y, T, N, K, gs, S};
    const int smem = T * (K + 8) * 2 + kW8Warps * 32 * 16;
    cudaError_t err = set_smem_once(reinterpret_cast<const void *>(w8a16_gemv_kernel), kW8MaxSmem + kW8Warps * 32 * 16);
    if (err != cudaSuccess) return err;
    const int nblocks = (N + 15) / 16, bpc = kW8Warps / S;
    // two CTAs of 16 warps per SM (registers capped for it: measured 12% faster than one
    // CTA per SM on lm_head), no more than the blocks need
    long long grid = (nblocks + bpc - 1) / bpc;
    const long long cap = 2LL * sm_count();
    if (grid > cap) grid = cap;
    w8a16_gemv_kernel<<<(unsigned)grid, kW8Warps * 32, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
