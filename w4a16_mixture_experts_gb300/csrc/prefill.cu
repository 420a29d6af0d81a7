// Expert path for batches of 8 tokens and more: W4A16 grouped GEMMs on the
// tcgen05 tensor core.
//
// Same computation as the fused Marlin MoE of "Running 125B MoE on Three
// 3090s - vLLM Optimization Edition", section 3.3 "MoE block" (gate_up,
// SiluAndMul, down, weighted sum), for batches where each expert sees many
// tokens. Section 3.3's W8A16 lesson (decode tiles do not carry over to
// prefill) is why this is a separate kernel. Two launches of one
// warp-specialised persistent kernel:
//
//   gate_up: tile = (expert, 64 intermediate rows i0.., up to 128 tokens).
//            A = 128 weight rows: gate row i0+i in TMEM lane 2i, the
//            matching up row in lane 2i+1; K = H.
//            Epilogue: h = topk_w * SiLU(g) * u (lane pairs meet by one
//            shuffle), rounded to bf16 and stored per slot. The routing weight
//            is applied here because the down projection is linear in h.
//   down:    tile = (expert, 128 output rows, up to 128 tokens), K = I.
//            Epilogue: out_acc[t] += y (fp32 reductions in L2).
//
// One pipeline stage is one quantisation group (128 of K):
//   * warp 12 lane 0 loads the stage's packed INT4 (128 rows x 64 bytes) with
//     two 2-D TMA copies in the 64-byte swizzle, which spreads the dequant
//     threads' 16-byte shared loads over the banks (consecutive rows of one
//     box are conflict-free; gate_up's paired lanes read two boxes and meet
//     2-way);
//   * warp 13 lane 0 loads the stage's activation rows (128 bf16 per slot)
//     with 2-D TMA copies in the 128-byte swizzle, as two K-major blocks: the
//     layout the MMA's shared-memory descriptor reads. The activations are in
//     slot order in global memory (x is gathered per slot before gate_up; h
//     is written per slot by it), so every tile's rows are contiguous;
//   * 128 dequant threads (one per weight row; two groups take alternate
//     stages) turn 128 nibbles into bf16 q*scale in registers and write them
//     straight into tensor memory as the A operand (tcgen05.st);
//   * the MMA warp issues 8 tcgen05.mma (M=128, N=tokens, K=16) from one
//     elected lane into an fp32 TMEM accumulator; one tcgen05.commit frees
//     the stage's A slot and activation buffer.
// Issuing the MMAs from a tight, unrolled, warp-uniform sequence matters: a
// 128x128x16 MMA takes about 64 SM cycles, so per-instruction issue overhead
// of the same order halves the tensor rate. The accumulator is double-buffered
// in TMEM so 256 epilogue threads drain one tile while the next accumulates.
//
// The same kernel, instantiated for INT8 (kW8), is the W8A16 linear layer for
// batches ("vLLM Optimization Edition", section 3.3 "Hyper-connection": the
// W8A16 GEMM over 4 tokens; model card groups C and D): one dense GEMM with the
// weight rows as M and the tokens as N, tiles of (128 rows, up to 128 tokens).
// The INT8 rows arrive by TMA (128 x 128 bytes a stage, 128-byte swizzle) and
// are dequantised exactly into bf16 in natural K order, so the activation rows
// are the caller's x as they are (no gather); each thread loads its row's
// scale(s) for the stage itself; the epilogue stores bf16 y.
//
// Weights enter A as W = bf16(q * scale) (one rounding per weight). Nibble
// pairs (j, j+4) of each word fill one 32-bit TMEM column, so the
// activations are kept in the matching order within each 8-element chunk
// (0,4,1,5,2,6,3,7): x is written in that order when it is gathered per
// slot, and the gate_up epilogue stores h in it directly.
#include <cuda.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace moe {

constexpr int kKS = 128;             // K per pipeline stage: one quantisation group
constexpr int kRR = 8;               // packed-INT4 stages (HBM stream)
constexpr int kRS = 4;               // A slots in TMEM = activation stages in smem (freed together)
constexpr int kPN = 128;             // max tokens per tile (columns of one TMEM accumulator)
constexpr int kWEpi = 8, kWRaw = 12, kWAct = 13, kWMma = 14, kWEpi2 = 15;
constexpr int kPThreads = 19 * 32;   // warps 0-7 dequant (two groups), 8-11 and 15-18 epilogue, 12 INT4 TMA,
                                     // 13 activation TMA, 14 MMA
constexpr int kNEpi = 256;           // epilogue threads: two per accumulator row
constexpr int kNBoxMaps = 4;         // activation TMA boxes of 16, 32, 64 and 128 token rows
static_assert((16 << (kNBoxMaps - 1)) == 128, "box sizes cover any multiple of 16 up to 128 rows");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAStage0 = 2 * kPN;          // TMEM columns: 2 accumulators, then the A slots
constexpr uint32_t kACols = kKS / 2;            // 64 columns (bf16 pairs) per A slot
constexpr uint32_t kBKBlock = kPN * 128;        // 128 token rows x 64 bf16: one 128-byte-swizzle K block
constexpr uint32_t kBBytes = 2 * kBKBlock;      // one activation stage: two K blocks
constexpr uint32_t kRawHalf = 64 * 64;          // 64 weight rows x 16 words
constexpr uint32_t kRawBytes = 2 * kRawHalf;    // one packed-INT4 stage
constexpr int kRR8 = 4;                         // INT8 stages: 128 rows x 128 bytes each
constexpr uint32_t kRawBytes8 = 128 * 128;
static_assert(kRR8 * kRawBytes8 == kRR * kRawBytes, "one raw ring size for both weight widths");
constexpr uint32_t kPrefillSmemMax = 232448 - 1024;   // dynamic; the static part is a few bytes
static_assert(kAStage0 + kRS * kACols <= kTmemCols, "tensor memory budget");

// A tile's scales (128 rows x G) go to one of nsc buffers: 2 at least, up to
// kMaxSC where shared memory allows. With 2, the scale copy of a tile waited
// for the dequantisation of the tile two before it, which held back the
// weight stream of short tiles (down: 5 stages a tile; measured at T = 64: the
// weight copies waited 24% of the kernel for a free scale buffer).
constexpr int kMaxSC = 4;
struct PrefillLayout {   // shared-memory offsets from the 1024-aligned base; scales sized by K
    uint32_t b, raw, sc, sc_bytes, cols, bars, tmem_slot, total;
    int nsc;
};
constexpr int kNBars = 2 * kRR + 3 * kRS + 4 + 2 * kMaxSC;

__host__ __device__ inline PrefillLayout prefill_layout_n(int G, int nsc) {
    PrefillLayout L;
    L.b = 0;
    L.raw = L.b + kRS * kBBytes;
    L.sc = L.raw + kRR * kRawBytes;
    L.sc_bytes = (uint32_t)(128 * G * 2 + 127) / 128 * 128;
    L.nsc = nsc;
    L.cols = L.sc + nsc * L.sc_bytes;         // per token column: f32 weight, i32 token
    L.bars = L.cols + 2 * 4 * kPN;
    L.tmem_slot = L.bars + kNBars * 8;
    L.total = L.tmem_slot + 16 + 1024;   // + alignment slack
    return L;
}

__host__ __device__ inline PrefillLayout prefill_layout(int G) {
    for (int n = kMaxSC; n > 2; --n) {
        const PrefillLayout L = prefill_layout_n(G, n);
        if (L.total <= kPrefillSmemMax) return L;
    }
    return prefill_layout_n(G, 2);
}

struct PrefillParams {
    CUtensorMap tm_w;          // int32 [rows][K/8], box (16 words, 64 rows; 128 for down), 64-byte swizzle
    CUtensorMap tm_b[4];       // bf16 [T*k][K] activations per slot, boxes (64, 16 << i rows), 128-byte swizzle
    const uint16_t *scales;    // bf16 [rows][K/128]
    const int32_t *offsets;    // [E+1] slot offsets per expert
    const int32_t *active;     // active experts, increasing
    const int32_t *n_chunks;   // [1] chunks in chunk_info
    const int4 *chunk_info;    // per chunk of at most 128 tokens: expert, first slot, tokens
    const int32_t *perm;       // slot -> assignment t*k+j
    const float *topk_w;
    const Ctrl *ctrl;
    Ctrl *ctrl_rw;
    uint16_t *hbuf;            // gate_up output, bf16 [T*k][I] fragment order
    const uint16_t *xs;        // gate_up input, bf16 [T*k][H] fragment order
    float *out_acc;            // down output, f32 [T][H]
    uint16_t *y;               // W8A16 output, bf16 [T][N]
    float *part;               // W8A16 split over K: f32 [ksplit][T][N] partial results
    int N, gs, dense_chunks;   // W8A16: output features, scale group, token chunks of 128
    int ksplit;                // W8A16: splits of K (1: the tile covers all of K)
    int T, H, E, k, I;
    int K;                     // reduction length: H (gate_up) or I (down)
    int mb;                    // row blocks per expert: I/64 (gate_up) or H/128 (down)
    int down;                  // 0: gate_up, 1: down
    PrefillLayout L;
};

struct Tile {
    int e, s0, nv, n16, m;
};

// Tile t = (chunk t / mb, row block t % mb): chunks of each expert are
// consecutive, and the row blocks of one chunk are consecutive tiles. The
// dense (W8A16) GEMM has one "expert" and chunks of 128 consecutive tokens.
template <bool kW8>
__device__ inline int4 chunk_of(const PrefillParams &p, int t) {
    if constexpr (kW8) {
        const int c = (t / p.mb) % p.dense_chunks;
        return make_int4(0, c * kPN, min(kPN, p.T - c * kPN), 0);
    } else {
        return __ldg(p.chunk_info + t / p.mb);
    }
}

// Stages [ks0, ks1) of tile t: all of K, or, for the dense GEMM split over K
// (tiles t = split * (row blocks * chunks) + chunk * row blocks + row block),
// the split's share.
template <bool kW8>
__device__ inline void tile_kspan(const PrefillParams &p, int t, int G, int &ks0, int &ks1) {
    if constexpr (kW8) {
        const int s = t / (p.mb * p.dense_chunks);
        ks0 = G * s / p.ksplit;
        ks1 = G * (s + 1) / p.ksplit;
    } else {
        ks0 = 0;
        ks1 = G;
    }
}

__device__ inline Tile make_tile(int4 ci, int m) {
    Tile r;
    r.e = ci.x;
    r.s0 = ci.y;
    r.nv = ci.z;
    r.n16 = (r.nv + 15) & ~15;
    r.m = m;
    return r;
}

// One lane of the (converged) warp returns true.
__device__ inline bool elect_one() {
    uint32_t pred;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
    return pred != 0;
}

// Bounded wait that also gives up when another role has aborted.
__device__ inline bool pwait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort_flag) return false;
    }
    return false;
}

// Named barrier 1 over the epilogue threads, returning the AND of `v`.
__device__ inline bool bar_and_epi(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kNEpi)
        : "memory");
    return r != 0;
}

__device__ inline void fail(const PrefillParams &p, volatile int *abort_flag) {
    *abort_flag = 1;
    set_error(p.ctrl_rw, MOE_ERR_TIMEOUT);
}

// 8 words (64 nibbles) of one weight row -> 32 TMEM columns: the bf16 pairs
// (j, j+4) of each word, times the group scale.
__device__ inline void dequant8(const uint4 &a, const uint4 &b, __nv_bfloat162 s2, uint32_t (&v)[32]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t q = int4_pair(w[m], j);
            __nv_bfloat162 qv = *reinterpret_cast<__nv_bfloat162 *>(&q);
            qv = __hmul2(qv, s2);
            v[4 * m + j] = *reinterpret_cast<uint32_t *>(&qv);
        }
}

// Bytes (b_lo, b_hi) of an INT8 pack-quantized word -> bf16x2 of (b - 128)
// each, exactly: prmt places the bytes in the two halves; 128 + (b & 127)
// and -256 (or -128 when b >= 128) are formed bitwise and added (sel 0x4140:
// bytes 0, 1; 0x4342: bytes 2, 3).
__device__ __forceinline__ uint32_t int8_pair(uint32_t w, uint32_t sel) {
    const uint32_t v = __byte_perm(w, 0u, sel);
    uint32_t lo, hi;
    asm("lop3.b32 %0, %1, 0x007F007F, %2, 0xEA;" : "=r"(lo) : "r"(v), "r"(0x43004300u));
    asm("lop3.b32 %0, %1, 0x00800080, %2, 0x6A;" : "=r"(hi) : "r"(v), "r"(0xC380C380u));
    __nv_bfloat162 r = __hadd2(*reinterpret_cast<__nv_bfloat162 *>(&lo), *reinterpret_cast<__nv_bfloat162 *>(&hi));
    return *reinterpret_cast<uint32_t *>(&r);
}

// 16 words (64 INT8 values) of one weight row -> 32 TMEM columns in natural K
// order (column j: values 2j, 2j + 1), times the scale.
__device__ inline void dequant8_w8(const uint4 &a, const uint4 &b, const uint4 &c, const uint4 &d,
                                   __nv_bfloat162 s2, uint32_t (&v)[32]) {
    const uint32_t w[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        uint32_t lo = int8_pair(w[m], 0x4140), hi = int8_pair(w[m], 0x4342);
        __nv_bfloat162 l2 = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&lo), s2);
        __nv_bfloat162 h2 = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&hi), s2);
        v[2 * m] = *reinterpret_cast<uint32_t *>(&l2);
        v[2 * m + 1] = *reinterpret_cast<uint32_t *>(&h2);
    }
}

template <bool kW8, bool kRed4>
__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int kRing = kW8 ? kRR8 : kRR;                       // raw weight stages
    constexpr uint32_t kStageBytes = kW8 ? kRawBytes8 : kRawBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PrefillLayout &L = p.L;
    uint8_t *sB = smem + L.b;
    uint8_t *sRaw = smem + L.raw;
    uint16_t *sSc = reinterpret_cast<uint16_t *>(smem + L.sc);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *raw_full = bars;              // [kRR] INT4 TMA (+tx)
    uint64_t *raw_empty = raw_full + kRR;   // [kRR] the 128 dequant threads of the stage's group
    uint64_t *b_full = raw_empty + kRR;     // [kRS] activation TMA (+tx)
    uint64_t *a_full = b_full + kRS;        // [kRS] 128 dequant threads (tcgen05.st done)
    uint64_t *ab_empty = a_full + kRS;      // [kRS] MMA commit: A slot and activation stage are free
    uint64_t *acc_full = ab_empty + kRS;    // [2] MMA commit
    uint64_t *acc_empty = acc_full + 2;     // [2] the epilogue threads
    uint64_t *sc_full = acc_empty + 2;      // [nsc] scale copy (+tx)
    uint64_t *sc_empty = sc_full + kMaxSC;  // [nsc] the 256 dequant threads
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    float *col_w = reinterpret_cast<float *>(smem + L.cols);     // epilogue (gate_up): routing weight
    uint32_t *col_off = reinterpret_cast<uint32_t *>(col_w + kPN);   // epilogue (down): token * H (< 2^32)
    __shared__ int abort_s;
    volatile int *abort_flag = &abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 128);
        }
        for (int i = 0; i < kRS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&a_full[i], 128);
            mbar_init(&ab_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kNEpi);
        }
        for (int b = 0; b < kMaxSC; ++b) {
            mbar_init(&sc_full[b], 1);
            mbar_init(&sc_empty[b], 256);
        }
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_w) : "memory");
        for (int i = 0; i < kNBoxMaps; ++i) asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_b[i]) : "memory");
    }
    if (warp == kWMma) {
        tc::alloc(tmem_slot, kTmemCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    const int ntiles = kW8 ? p.ksplit * p.dense_chunks * p.mb : *p.n_chunks * p.mb;
    const int G = (p.K + kKS - 1) / kKS;   // stages per tile (the dense GEMM's last one may be half)

    if (kW8 && warp < kWEpi) {
        // ------------------------------------------------ INT8 dequant: one weight row per thread
        // (rows in order); group 0 takes the even stages, group 1 the odd ones. The row's scales
        // for a stage (one per 128 values for gs 128, two for gs 64) come from global memory,
        // requested before the stage's weights are waited for.
        const int grp = warp >> 2;
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int sw = r & 7;              // 128-byte swizzle: 16-byte chunk c of row r sits at c ^ (r & 7)
        const int nG = p.K / p.gs;          // scale groups per row
        uint32_t g = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int n = (t % p.mb) * 128 + r;   // this thread's weight row (output feature)
            const uint16_t *srow = p.scales + (size_t)(n < p.N ? n : 0) * nG;
            bool ok = true;
            int ks0, ks1;
            tile_kspan<kW8>(p, t, G, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g) {
                if ((int)(g & 1) != grp) continue;
                const int sr = g % kRing, sa = g % kRS;
                const int q0 = ks * kKS / p.gs, q1 = p.gs == kKS ? q0 : q0 + 1;
                const uint32_t sb0 = n < p.N && q0 < nG ? (uint32_t)__ldg(srow + q0) : 0u;
                const uint32_t sb1 = n < p.N && q1 < nG ? (uint32_t)__ldg(srow + q1) : 0u;
                if (!pwait(&raw_full[sr], (g / kRing) & 1, abort_flag)) { ok = false; break; }
                const uint8_t *rr = sRaw + sr * kStageBytes + r * 128;
                uint4 c[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) c[i] = lds_v4(rr + 16 * (i ^ sw));
                const uint32_t s2a = sb0 | (sb0 << 16), s2b = sb1 | (sb1 << 16);
                uint32_t v0[32], v1[32];
                dequant8_w8(c[0], c[1], c[2], c[3], *reinterpret_cast<const __nv_bfloat162 *>(&s2a), v0);
                dequant8_w8(c[4], c[5], c[6], c[7], *reinterpret_cast<const __nv_bfloat162 *>(&s2b), v1);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&raw_empty[sr]);
                if (!pwait(&ab_empty[sa], ((g / kRS) & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc::fence_after();
                const uint32_t ta = tmem + lane_base + kAStage0 + sa * kACols;
                tc::st_32x32b_x32(ta, v0);
                tc::st_32x32b_x32(ta + 32, v1);
                tc::wait_st();
                tc::fence_before();
                mbar_arrive(&a_full[sa]);
            }
            if (!ok) { fail(p, abort_flag); break; }
        }
    } else if (warp < kWEpi) {
        // ------------------------------------------------ dequant: one weight row per thread; group
        // 0 (warps 0-3) takes the even stages, group 1 (warps 4-7) the odd ones
        const int grp = warp >> 2;
        const int r = threadIdx.x & 127;   // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;   // the warp's TMEM lane quarter
        // TMA box (half of the stage) and row within it: gate_up puts gate row i in lane 2i and
        // up row i in lane 2i+1, so the epilogue pairs them with one shuffle; down is in order
        const int half = p.down ? r >> 6 : r & 1;
        const int br = p.down ? r & 63 : r >> 1;
        const int rbase = half * (int)kRawHalf + br * 64;
        const int rot = (br >> 1) & 3;     // 64-byte swizzle: 16-byte chunk c sits at c ^ rot
        uint32_t g = 0;
        int lt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            const int tb = lt % L.nsc;
            if (!pwait(&sc_full[tb], (lt / L.nsc) & 1, abort_flag)) { fail(p, abort_flag); break; }
            const uint16_t *sc = sSc + tb * (L.sc_bytes / 2) + (half * 64 + br) * G;
            bool ok = true;
            int ks0, ks1;
            tile_kspan<kW8>(p, t, G, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g) {
                if ((int)(g & 1) != grp) continue;
                const int sr = g % kRR, sa = g % kRS;
                if (!pwait(&raw_full[sr], (g / kRR) & 1, abort_flag)) { ok = false; break; }
                const uint8_t *rr = sRaw + sr * kRawBytes + rbase;
                const uint4 c0 = lds_v4(rr + 16 * (0 ^ rot)), c1 = lds_v4(rr + 16 * (1 ^ rot));
                const uint4 c2 = lds_v4(rr + 16 * (2 ^ rot)), c3 = lds_v4(rr + 16 * (3 ^ rot));
                const uint32_t sb = sc[ks];
                const uint32_t s2u = sb | (sb << 16);
                const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162 *>(&s2u);
                uint32_t v0[32], v1[32];
                dequant8(c0, c1, s2, v0);
                dequant8(c2, c3, s2, v1);
                // The words are consumed (v depends on them), so the loads have landed;
                // order them before the TMA that will refill the stage.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&raw_empty[sr]);
                // the MMA must have finished reading this tensor-memory slot
                if (!pwait(&ab_empty[sa], ((g / kRS) & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc::fence_after();
                const uint32_t ta = tmem + lane_base + kAStage0 + sa * kACols;
                tc::st_32x32b_x32(ta, v0);
                tc::st_32x32b_x32(ta + 32, v1);
                tc::wait_st();
                tc::fence_before();
                mbar_arrive(&a_full[sa]);
            }
            if (!ok) { fail(p, abort_flag); break; }
            mbar_arrive(&sc_empty[tb]);
        }
    } else if (warp < kWRaw || warp >= kWEpi2) {
        // ------------------------------------------------ epilogue: two threads per accumulator row
        // (one in warps 8-11, one in warps 15-18) taking alternate column chunks, written
        // straight to global memory (h as bf16 stores, down as fp32 reductions in L2)
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int eh = warp >= kWEpi2;             // which of the row's two threads
        const int et = 32 * q + lane;              // 0..127 = TMEM lane = tile row
        // gate_up: this lane pair's intermediate row and its fragment-order position
        const int il = et >> 1;
        const int pl = 8 * (il >> 3) + 2 * (il & 3) + ((il >> 2) & 1);
        int lt = 0;
        int4 ci = blockIdx.x < (unsigned)ntiles ? chunk_of<kW8>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            const Tile T = make_tile(ci, t % p.mb);
            if (t + (int)gridDim.x < ntiles) ci = chunk_of<kW8>(p, t + gridDim.x);   // lands during this tile
            const int b = lt & 1;
            // the epilogue threads share named barrier 1: they give up together
            if (!bar_and_epi(pwait(&acc_full[b], (lt >> 1) & 1, abort_flag))) { fail(p, abort_flag); break; }
            tc::fence_after();
            const uint32_t dbase = tmem + ((uint32_t)(32 * q) << 16) + b * kPN;
            // per column of the tile: gate_up needs the slot's routing weight, down the
            // token's output row (the previous tile's readers passed the barrier above)
            if (!kW8 && !eh && et < T.nv) {
                const int a = p.perm[T.s0 + et];
                if (p.down) col_off[et] = (uint32_t)(a / p.k) * (uint32_t)p.H;
                else col_w[et] = p.topk_w[a];
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kNEpi) : "memory");
            if (kW8) {
                // y[token][n] (or, split over K, this split's f32 part): for each column the 32
                // lanes of a warp store 32 consecutive n
                const int n = T.m * 128 + et;
                const int split = t / (p.mb * p.dense_chunks);
                for (int c0 = 32 * eh; c0 < T.nv; c0 += 64) {
                    float v[32];
                    tc::ld_32x32b_x32(dbase + c0, v);
                    tc::wait_ld();
                    const int nu = min(32, T.nv - c0);
                    if (n < p.N) {
                        if (p.ksplit > 1) {
                            float *prow = p.part + ((size_t)split * p.T + T.s0 + c0) * p.N + n;
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                if (u < nu) prow[(size_t)u * p.N] = v[u];
                        } else {
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                if (u < nu) {
                                    const __nv_bfloat16 hb = __float2bfloat16_rn(v[u]);
                                    p.y[(size_t)(T.s0 + c0 + u) * p.N + n] = *reinterpret_cast<const uint16_t *>(&hb);
                                }
                        }
                    }
                }
            } else if (p.down) {
                // one reduction per (row, token): the 32 lanes of a warp cover 128 consecutive
                // bytes of the token's output row; the routing weight is already in h
                float *orow = p.out_acc + T.m * 128 + et;
                // with kRed4, one 16-byte reduction per (4 rows, token): the 4 lanes of a row
                // quad swap values in two butterfly stages, so that lane r of the quad holds
                // rows 4j .. 4j + 3 of token 4i + r. A quarter of the reduction requests at
                // the cost of the swaps: measured 5% faster for a 4096-token layer, where the
                // reductions (105 M a layer) bind, and 2-3% slower for 64 to 2048 tokens.
                float *obase = p.out_acc + T.m * 128 + 32 * q + (lane & ~3);
                const int r = lane & 3;
                const bool b1 = (r & 2) != 0, b0 = (r & 1) != 0;
                (void)orow, (void)obase, (void)b1, (void)b0;
                for (int c0 = 32 * eh; c0 < T.nv; c0 += 64) {
                    float v[32];
                    tc::ld_32x32b_x32(dbase + c0, v);
                    tc::wait_ld();
                    const int nu = min(32, T.nv - c0);
                    if constexpr (!kRed4) {
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            if (u < nu) atomicAdd(orow + (size_t)col_off[c0 + u], v[u]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (4 * i < nu) {
                                const float a0 = v[4 * i], a1 = v[4 * i + 1], a2 = v[4 * i + 2], a3 = v[4 * i + 3];
                                // stage 1 (lanes r, r ^ 2): keep columns 2 b1, 2 b1 + 1 of rows r, r ^ 2
                                const float k0 = b1 ? a2 : a0, k1 = b1 ? a3 : a1;
                                const float g0 = __shfl_xor_sync(0xffffffffu, b1 ? a0 : a2, 2);
                                const float g1 = __shfl_xor_sync(0xffffffffu, b1 ? a1 : a3, 2);
                                // stage 2 (lanes r, r ^ 1): keep column r of all four rows
                                const float kr = b0 ? k1 : k0, kq = b0 ? g1 : g0;
                                const float h1 = __shfl_xor_sync(0xffffffffu, b0 ? k0 : k1, 1);
                                const float h3 = __shfl_xor_sync(0xffffffffu, b0 ? g0 : g1, 1);
                                // row k of token 4i + r is [kr, h1, kq, h3][k ^ r]
                                float4 o;
                                o.x = b1 ? (b0 ? h3 : kq) : (b0 ? h1 : kr);
                                o.y = b1 ? (b0 ? kq : h3) : (b0 ? kr : h1);
                                o.z = b1 ? (b0 ? h1 : kr) : (b0 ? h3 : kq);
                                o.w = b1 ? (b0 ? kr : h1) : (b0 ? kq : h3);
                                if (4 * i + r < nu)
                                    atomicAdd(reinterpret_cast<float4 *>(obase + (size_t)col_off[c0 + 4 * i + r]), o);
                            }
                        }
                    }
                }
            } else {
                uint16_t *hrow = p.hbuf + (size_t)T.s0 * p.I + T.m * 64 + pl;
                for (int c0 = 16 * eh; c0 < T.nv; c0 += 32) {
                    float v[16];
                    tc::ld_32x32b_x16(dbase + c0, v);
                    tc::wait_ld();
                    const int nu = min(16, T.nv - c0);
                    // the gate lane finishes columns 0-7 of the chunk, the up lane columns 8-15
                    const bool odd = et & 1;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[j + 8], 1);
                        const float gv = odd ? recv : v[j], uv = odd ? v[j + 8] : recv;
                        const int u = odd ? j + 8 : j;
                        if (u < nu) {
                            const __nv_bfloat16 hb = __float2bfloat16_rn(silu(gv) * uv * col_w[c0 + u]);
                            hrow[(size_t)(c0 + u) * p.I] = *reinterpret_cast<const uint16_t *>(&hb);
                        }
                    }
                }
            }
            tc::fence_before();
            mbar_arrive(&acc_empty[b]);
        }
    } else if (warp == kWRaw) {
        // ------------------------------------------------ INT4 stages and scales: one TMA thread
        // (the weights are read once: they go through L2 at evict-first priority, so that
        // the activations, which every row block of a chunk re-reads, stay resident)
        if (lane == 0) {
            const uint64_t wpol = l2_evict_first();
            uint32_t g = 0;
            int lt = 0;
            int4 ci = blockIdx.x < (unsigned)ntiles ? chunk_of<kW8>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
                const Tile T = make_tile(ci, t % p.mb);
                if (t + (int)gridDim.x < ntiles) ci = chunk_of<kW8>(p, t + gridDim.x);
                const int tb = lt % L.nsc;
                // weight rows of TMEM lanes 0-63 and 64-127
                const int row_a = kW8 ? T.m * 128 : p.down ? T.e * p.H + T.m * 128 : T.e * 2 * p.I + T.m * 64;
                const int row_b = row_a + (p.down ? 64 : p.I);
                if (!kW8) {
                    if (!pwait(&sc_empty[tb], ((lt / L.nsc) & 1) ^ 1, abort_flag)) { fail(p, abort_flag); break; }
                    uint16_t *dst = sSc + tb * (L.sc_bytes / 2);
                    mbar_arrive_expect_tx(&sc_full[tb], 128 * G * 2);
                    bulk_g2s(dst, p.scales + (size_t)row_a * G, 64 * G * 2, &sc_full[tb]);
                    bulk_g2s(dst + 64 * G, p.scales + (size_t)row_b * G, 64 * G * 2, &sc_full[tb]);
                }
                bool ok = true;
                int ks0, ks1;
            tile_kspan<kW8>(p, t, G, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g) {
                    const int sr = g % kRing;
                    if (!pwait(&raw_empty[sr], ((g / kRing) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&raw_full[sr], kStageBytes);
                    uint8_t *rdst = sRaw + sr * kStageBytes;
                    if (kW8) {
                        // 128 INT8 rows x 128 values (32 words); rows past N and words past K read as zero
                        tma_load_2d_hint(rdst, &p.tm_w, ks * 32, row_a, &raw_full[sr], wpol);
                    } else {
                        // down's 128 rows are consecutive: one box (gate_up: gate and up boxes)
                        tma_load_2d_hint(rdst, &p.tm_w, ks * 16, row_a, &raw_full[sr], wpol);
                        if (!p.down) tma_load_2d_hint(rdst + kRawHalf, &p.tm_w, ks * 16, row_b, &raw_full[sr], wpol);
                    }
                }
                if (!ok) { fail(p, abort_flag); break; }
            }
            // the consumers waited on every issued weight stage, except after an abort:
            // then give the outstanding ones a bounded wait before the CTA exits
            if (*abort_flag)
                for (uint32_t gg = g > (uint32_t)kRing ? g - kRing : 0; gg < g; ++gg)
                    mbar_wait(&raw_full[gg % kRing], (gg / kRing) & 1);
        }
    } else if (warp == kWAct) {
        // ------------------------------------------------ activation stages: one TMA thread
        if (lane == 0) {
            uint32_t g = 0;
            const int grid = (int)gridDim.x;
            int4 ci = blockIdx.x < (unsigned)ntiles ? chunk_of<kW8>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
            int4 ci2 = blockIdx.x + grid < ntiles ? chunk_of<kW8>(p, blockIdx.x + grid) : make_int4(0, 0, 0, 0);
            for (int t = blockIdx.x; t < ntiles; t += grid) {
                const Tile T = make_tile(ci, t % p.mb);
                ci = ci2;
                const int t2 = t + 2 * grid;   // the tile after next
                if (t2 < ntiles) ci2 = chunk_of<kW8>(p, t2);
                bool ok = true;
                int ks0, ks1;
            tile_kspan<kW8>(p, t, G, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g) {
                    const int sb = g % kRS;
                    if (!pwait(&ab_empty[sb], ((g / kRS) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&b_full[sb], 2u * T.n16 * 128u);
                    // n16 rows as few, large boxes (TMA moves big boxes much faster); rows past
                    // the tile's tokens belong to other slots (or lie past the tensor and read as
                    // zero): they only feed columns the epilogue skips
                    for (int kb = 0; kb < 2; ++kb)
                        for (int i = kNBoxMaps - 1, r0 = 0; i >= 0; --i)
                            if (T.n16 & (16 << i)) {
                                tma_load_2d(sB + sb * kBBytes + kb * kBKBlock + r0 * 128, &p.tm_b[i],
                                            ks * kKS + kb * 64, T.s0 + r0, &b_full[sb]);
                                r0 += 16 << i;
                            }
                }
                if (!ok) { fail(p, abort_flag); break; }
                // gate_up's x rows of a chunk are first read from HBM by the chunk's row-block
                // tiles all at once; the CTA that will start a chunk pulls its rows into L2
                // about one tile ahead
                if (!p.down && t2 < ntiles && t2 % p.mb == 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.xs + (size_t)ci2.y * p.H),
                                 "r"((uint32_t)ci2.z * (uint32_t)p.H * 2u)
                                 : "memory");
            }
            // after an abort, give the stages still in flight a bounded wait before the CTA exits
            if (*abort_flag)
                for (uint32_t gg = g > (uint32_t)kRS ? g - kRS : 0; gg < g; ++gg)
                    mbar_wait(&b_full[gg % kRS], (gg / kRS) & 1);
        }
    } else {
        // ------------------------------------------------ MMA issuer: the whole warp waits, one
        // elected lane issues the stage's 8 MMAs and the commit
        uint32_t g = 0;
        int lt = 0;
        int4 ci = blockIdx.x < (unsigned)ntiles ? chunk_of<kW8>(p, blockIdx.x) : make_int4(0, 0, 0, 0);
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            const Tile T = make_tile(ci, t % p.mb);
            if (t + (int)gridDim.x < ntiles) ci = chunk_of<kW8>(p, t + gridDim.x);
            const int b = lt & 1;
            if (!__all_sync(0xffffffffu, pwait(&acc_empty[b], ((lt >> 1) & 1) ^ 1, abort_flag))) {
                fail(p, abort_flag);
                break;
            }
            tc::fence_after();
            const uint32_t d = tmem + b * kPN;
            const uint32_t idesc = tc::idesc_bf16(128, T.n16);
            bool ok = true;
            int ks0, ks1;
            tile_kspan<kW8>(p, t, G, ks0, ks1);
            for (int ks = ks0; ks < ks1; ++ks, ++g) {
                const int s = g % kRS;
                const uint32_t par = (g / kRS) & 1;
                const bool ready = pwait(&a_full[s], par, abort_flag) && pwait(&b_full[s], par, abort_flag);
                if (!__all_sync(0xffffffffu, ready)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                if (elect_one()) {
                    const uint64_t bd0 = tc::sdesc_sw128(sB + s * kBBytes);
                    const uint64_t bd1 = tc::sdesc_sw128(sB + s * kBBytes + kBKBlock);
                    const uint32_t a0 = tmem + kAStage0 + s * kACols;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(d, a0 + kk * 8, (kk < 4 ? bd0 : bd1) + (uint64_t)((kk & 3) * 2), idesc,
                                   ks != ks0 || kk != 0);
                    tc::commit(&ab_empty[s]);   // one commit: A slot and activation stage share the index
                }
                __syncwarp();
            }
            if (!ok) { fail(p, abort_flag); break; }
            if (elect_one()) tc::commit(&acc_full[b]);
            __syncwarp();
        }
    }

    // all tensor-core work of this CTA has been consumed by the epilogue (or the
    // CTA aborted); free the tensor memory
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == kWMma) tc::dealloc(tmem, kTmemCols);
}
// Batches from which the down epilogue reduces 4 rows at a time (measured:
// slower at 2048 tokens, faster at 4096).
constexpr int kRed4MinT = 4096;

// ---------------------------------------------------------------------------
// xs[slot] = x[token of slot] in fragment order within each 8-element chunk
// (0,4,1,5,2,6,3,7), for the offsets[E] slots that hold a valid assignment.
// A warp copies whole rows: the row's token is read once (the next row's is
// fetched while this one moves), then up to kXgLoads 16-byte chunks per lane
// are in flight at once. The same warps then clear the T rows of the down
// kernel's fp32 accumulator.
constexpr int kXgThreads = 256;
constexpr int kXgLoads = 10;   // a 2560-wide row in one pass

__global__ void __launch_bounds__(kXgThreads) xgather_kernel(const uint16_t *__restrict__ x,
                                                             const int32_t *__restrict__ perm,
                                                             const int32_t *__restrict__ offsets, int E, int H, int k,
                                                             uint16_t *__restrict__ xs, float *__restrict__ out_acc,
                                                             int T) {
    const int nslots = offsets[E];
    const int cpr = H / 8;   // 16-byte chunks per row
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (kXgThreads / 32);
    int slot = blockIdx.x * (kXgThreads / 32) + (threadIdx.x >> 5);
    int tok = slot < nslots ? perm[slot] / k : 0;
    for (; slot < nslots; slot += nw) {
        const int nxt = slot + nw < nslots ? perm[slot + nw] / k : 0;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)tok * H);
        uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)slot * H);
        for (int c0 = lane; c0 < cpr; c0 += 32 * kXgLoads) {
            uint4 v[kXgLoads];
#pragma unroll
            for (int u = 0; u < kXgLoads; ++u) {
                const int c = c0 + 32 * u;
                v[u] = c < cpr ? ld_nc_v4(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kXgLoads; ++u) {
                const int c = c0 + 32 * u;
                if (c < cpr)
                    dst[c] = make_uint4(__byte_perm(v[u].x, v[u].z, 0x5410), __byte_perm(v[u].x, v[u].z, 0x7632),
                                        __byte_perm(v[u].y, v[u].w, 0x5410), __byte_perm(v[u].y, v[u].w, 0x7632));
            }
        }
        tok = nxt;
    }
    // the down kernel's accumulator starts at zero: the warps clear its T rows
    // (so that nothing depends on what an earlier call left in the workspace)
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = blockIdx.x * (kXgThreads / 32) + (threadIdx.x >> 5); t < T; t += nw) {
        float4 *row = reinterpret_cast<float4 *>(out_acc + (size_t)t * H);
        for (int c = lane; c < H / 4; c += 32) row[c] = z4;
    }
}

// The chunk table of the two persistent launches, in one CTA. Each active
// expert's slots are split into c = ceil(count / 128) chunks of near-equal
// size (the first count % c of them one token larger); the experts are
// ordered by that size, largest first (by 16-token band, ties in expert
// order), with each expert's chunks adjacent. The kernels deal tiles
// round-robin in this order, so every CTA gets a tile of each size band and
// the launch ends with the small ones, while an expert's chunks still run side
// by side (its weights come from HBM once, the other chunks find them in L2).
// chunk_info[i] = (expert, first slot, tokens); *n_chunks = their number.
constexpr int kNBands = kPN / 16;

__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *__restrict__ counts,
                                                           const int32_t *__restrict__ offsets, int E,
                                                           int32_t *__restrict__ n_chunks,
                                                           int4 *__restrict__ chunk_info) {
    __shared__ int s_warp[32][kNBands];   // chunks of each band in each warp, then the exclusive prefix
    __shared__ int s_band[kNBands];       // first chunk of each band
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    const int cnt = e < E ? counts[e] : 0;
    const int c = (cnt + kPN - 1) / kPN;
    const int band = c ? kNBands - ((cnt + c - 1) / c + 15) / 16 : -1;
    int before = 0;   // chunks of e's band held by lower experts of this warp
#pragma unroll
    for (int b = 0; b < kNBands; ++b) {
        const int v = band == b ? c : 0;
        int iv = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, iv, off);
            if (lane >= off) iv += o;
        }
        if (band == b) before = iv - v;
        if (lane == 31) s_warp[w][b] = iv;
    }
    __syncthreads();
    if (e < kNBands) {   // exclusive prefix over the warps, band e
        int run = 0;
        for (int ww = 0; ww < 32; ++ww) {
            const int v = s_warp[ww][e];
            s_warp[ww][e] = run;
            run += v;
        }
        s_band[e] = run;
    }
    __syncthreads();
    if (e == 0) {
        int run = 0;
        for (int b = 0; b < kNBands; ++b) {
            const int v = s_band[b];
            s_band[b] = run;
            run += v;
        }
        *n_chunks = run;
    }
    __syncthreads();
    if (c > 0) {
        const int first = s_band[band] + s_warp[w][band] + before;
        const int base = cnt / c, rem = cnt % c;
        for (int j = 0; j < c; ++j)
            chunk_info[first + j] = make_int4(e, offsets[e] + j * base + min(j, rem), base + (j < rem), 0);
    }
}

// out[t][n] = bf16(out_acc[t][n]) (or the stack epilogue); out_acc was
// cleared by the gather kernel at the start of the call.
// One CTA per token, 16-byte accesses; the stack variant keeps the token's
// row in registers between the sum of squares and the rescale.
constexpr int kConvThreads = 256;
constexpr int kConvPer = 8192 / 4 / kConvThreads;   // float4s of a row per thread (H <= 8192)

__device__ inline uint2 bf16x4(float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    return u;
}

__global__ void __launch_bounds__(kConvThreads) acc_convert_kernel(float *__restrict__ acc, const uint16_t *__restrict__ x,
                                                                   int H, float eps, uint16_t *__restrict__ out,
                                                                   uint16_t *__restrict__ next) {
    __shared__ float red[kConvThreads / 32];
    const int t = blockIdx.x;
    float4 *row = reinterpret_cast<float4 *>(acc + (size_t)t * H);
    const int n4 = H / 4;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    // the whole row in flight at once (and, for the stack, the residual row)
    float4 r[kConvPer];
    uint2 xv[kConvPer];
    const uint2 *xr = reinterpret_cast<const uint2 *>(x + (size_t)t * H);
#pragma unroll
    for (int j = 0; j < kConvPer; ++j) {
        const int i = threadIdx.x + kConvThreads * j;
        r[j] = i < n4 ? row[i] : zero;
        xv[j] = next && i < n4 ? xr[i] : make_uint2(0u, 0u);
    }
    if (!next) {
        uint2 *o = reinterpret_cast<uint2 *>(out + (size_t)t * H);
#pragma unroll
        for (int j = 0; j < kConvPer; ++j) {
            const int i = threadIdx.x + kConvThreads * j;
            if (i < n4) o[i] = bf16x4(r[j].x, r[j].y, r[j].z, r[j].w);
        }
        return;
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kConvPer; ++j) {
        r[j] = make_float4(r[j].x + __uint_as_float(xv[j].x << 16), r[j].y + __uint_as_float(xv[j].x & 0xffff0000u),
                           r[j].z + __uint_as_float(xv[j].y << 16), r[j].w + __uint_as_float(xv[j].y & 0xffff0000u));
        ss += r[j].x * r[j].x + r[j].y * r[j].y + r[j].z * r[j].z + r[j].w * r[j].w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConvThreads / 32; ++w) tot += red[w];
    const float scale = rsqrtf(tot / (float)H + eps);
    uint2 *o = reinterpret_cast<uint2 *>(next + (size_t)t * H);
#pragma unroll
    for (int j = 0; j < kConvPer; ++j) {
        const int i = threadIdx.x + kConvThreads * j;
        if (i < n4) o[i] = bf16x4(r[j].x * scale, r[j].y * scale, r[j].z * scale, r[j].w * scale);
    }
}

bool prefill_supported(const moe_dims &d) {
    const int gmax = d.H > d.I ? d.H / 128 : d.I / 128;
    return d.H % 128 == 0 && d.I % 128 == 0 && prefill_layout(gmax).total <= kPrefillSmemMax;
}

cudaError_t launch_prefill(const ExpertArgs &a, const moe_dims &d, void *ws, uint16_t *out, uint16_t *next, float eps,
                           cudaEvent_t ev_before, cudaEvent_t ev_after, cudaStream_t s) {
    const WsLayout W = ws_layout(d);
    uint16_t *xperm = ws_at<uint16_t>(ws, W.xperm);
    float *out_acc = ws_at<float>(ws, W.out_acc);
    int32_t *n_chunks = ws_at<int32_t>(ws, W.n_chunks);
    // the down launch of a large batch takes the instantiation with 16-byte reductions
    const bool red4 = d.T >= kRed4MinT;
    cudaError_t err = set_smem_once(reinterpret_cast<const void *>(prefill_kernel<false, false>), (int)kPrefillSmemMax);
    if (err == cudaSuccess && red4)
        err = set_smem_once(reinterpret_cast<const void *>(prefill_kernel<false, true>), (int)kPrefillSmemMax);
    if (err != cudaSuccess) return err;

    {
        // a warp per row, at most 8 CTAs of 8 warps per SM
        const long long rows = (long long)d.T * d.k, per_cta = kXgThreads / 32;
        long long grid = (rows + per_cta - 1) / per_cta;
        if (grid > 8LL * sm_count()) grid = 8LL * sm_count();
        if (grid < 1) grid = 1;
        xgather_kernel<<<(unsigned)grid, kXgThreads, 0, s>>>(a.x, ws_at<int32_t>(ws, W.perm),
                                                             ws_at<int32_t>(ws, W.offsets), d.E, d.H, d.k, xperm,
                                                             out_acc, d.T);
    }
    int4 *chunk_info = ws_at<int4>(ws, W.chunk_info);
    chunk_table_kernel<<<1, 1024, 0, s>>>(ws_at<int32_t>(ws, W.counts), ws_at<int32_t>(ws, W.offsets), d.E, n_chunks,
                                          chunk_info);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    PrefillParams p;
    p.offsets = ws_at<int32_t>(ws, W.offsets);
    p.active = ws_at<int32_t>(ws, W.active);
    p.n_chunks = n_chunks;
    p.chunk_info = chunk_info;
    p.perm = ws_at<int32_t>(ws, W.perm);
    p.topk_w = a.topk_w;
    p.ctrl = ws_at<Ctrl>(ws, W.ctrl);
    p.ctrl_rw = ws_at<Ctrl>(ws, W.ctrl);
    p.hbuf = ws_at<uint16_t>(ws, W.hbuf);
    p.out_acc = out_acc;
    p.T = d.T;
    p.H = d.H;
    p.E = d.E;
    p.k = d.k;
    p.I = d.I;
    const unsigned grid = (unsigned)sm_count();

    // gate_up: K = H, 64 intermediate rows (x2 for gate and up) per tile
    err = encode_tmap_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, a.w1p, (uint64_t)d.H / 8, (uint64_t)d.E * 2 * d.I,
                         (uint64_t)d.H / 2, 16u, 64u, CU_TENSOR_MAP_SWIZZLE_64B);
    if (err != cudaSuccess) return err;
    if ((err = record_profile_event(ev_before, s)) != cudaSuccess) return err;
    p.xs = xperm;
    for (int i = 0; i < kNBoxMaps && err == cudaSuccess; ++i)
        err = encode_tmap_2d(&p.tm_b[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xperm, (uint64_t)d.H,
                             (uint64_t)d.T * d.k, (uint64_t)d.H * 2, 64u, 16u << i, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    p.scales = a.w1s;
    p.K = d.H;
    p.mb = d.I / 64;
    p.down = 0;
    p.L = prefill_layout(p.K / kKS);
    prefill_kernel<false, false><<<grid, kPThreads, p.L.total, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    // down: K = I, 128 output rows per tile
    err = encode_tmap_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, a.w2p, (uint64_t)d.I / 8, (uint64_t)d.E * d.H,
                         (uint64_t)d.I / 2, 16u, 128u, CU_TENSOR_MAP_SWIZZLE_64B);
    if (err != cudaSuccess) return err;
    for (int i = 0; i < kNBoxMaps && err == cudaSuccess; ++i)
        err = encode_tmap_2d(&p.tm_b[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.hbuf, (uint64_t)d.I,
                             (uint64_t)d.T * d.k, (uint64_t)d.I * 2, 64u, 16u << i, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    p.scales = a.w2s;
    p.K = d.I;
    p.mb = d.H / 128;
    p.down = 1;
    p.L = prefill_layout(p.K / kKS);
    if (red4) prefill_kernel<false, true><<<grid, kPThreads, p.L.total, s>>>(p);
    else prefill_kernel<false, false><<<grid, kPThreads, p.L.total, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if ((err = record_profile_event(ev_after, s)) != cudaSuccess) return err;

    acc_convert_kernel<<<d.T, kConvThreads, 0, s>>>(out_acc, a.x, d.H, eps, next ? nullptr : out, next);
    return cudaGetLastError();
}

// The W8A16 linear layer for batches: the dense INT8 instantiation, x and y the
// caller's (token chunks of 128 consecutive tokens, row blocks of 128 weight rows).
// A layer with fewer tiles than SMs (the hyper-connection mixer [320, 10240] at
// 512 tokens has 12) splits K so that about one wave of CTAs runs, each split at
// least kMinSplitStages stages long; the splits' f32 results are summed in split
// order (deterministic) by w8a16_reduce_kernel.
constexpr int kMinSplitStages = 4;
// The split aims at one wave of CTAs on a 152-SM GB300; it is fixed rather than
// read from the device so that the workspace size does not depend on it.
constexpr int kSplitWave = 148;

int w8a16_gemm_splits(int T, int N, int K) {
    const long long tiles = (long long)((N + 127) / 128) * ((T + kPN - 1) / kPN);
    const int G = (K + kKS - 1) / kKS;
    long long s = kSplitWave / (tiles > 0 ? tiles : 1);
    if (s > G / kMinSplitStages) s = G / kMinSplitStages;
    return s < 1 ? 1 : (int)s;
}

__global__ void __launch_bounds__(256) w8a16_reduce_kernel(const float *__restrict__ part, int S, size_t n,
                                                          uint16_t *__restrict__ y) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int j = 0; j < S; ++j) s += __ldcg(part + (size_t)j * n + i);
        const __nv_bfloat16 h = __float2bfloat16_rn(s);
        y[i] = *reinterpret_cast<const uint16_t *>(&h);
    }
}

cudaError_t launch_w8a16_gemm(const uint16_t *x, const int32_t *w, const uint16_t *s, int gs, uint16_t *y, int T, int N,
                              int K, Ctrl *ctrl, float *part, cudaStream_t st) {
    cudaError_t err = set_smem_once(reinterpret_cast<const void *>(prefill_kernel<true, false>), (int)kPrefillSmemMax);
    if (err != cudaSuccess) return err;
    PrefillParams p{};
    err = encode_tmap_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, w, (uint64_t)K / 4, (uint64_t)N, (uint64_t)K, 32u,
                         128u, CU_TENSOR_MAP_SWIZZLE_128B);
    for (int i = 0; i < kNBoxMaps && err == cudaSuccess; ++i)
        err = encode_tmap_2d(&p.tm_b[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, (uint64_t)K, (uint64_t)T,
                             (uint64_t)K * 2, 64u, 16u << i, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    p.scales = s;
    p.y = y;
    p.part = part;
    p.N = N;
    p.gs = gs;
    p.T = T;
    p.K = K;
    p.mb = (N + 127) / 128;
    p.dense_chunks = (T + kPN - 1) / kPN;
    p.ksplit = w8a16_gemm_splits(T, N, K);
    p.down = 1;
    p.ctrl = ctrl;
    p.ctrl_rw = ctrl;
    p.L = prefill_layout(0);
    const long long tiles = (long long)p.ksplit * p.mb * p.dense_chunks;
    const unsigned grid = (unsigned)(tiles < sm_count() ? tiles : sm_count());
    prefill_kernel<true, false><<<grid, kPThreads, p.L.total, st>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (p.ksplit > 1) {
        const size_t n = (size_t)T * N;
        const long long blocks = (long long)((n + 255) / 256);
        w8a16_reduce_kernel<<<(unsigned)(blocks < 8LL * sm_count() ? blocks : 8LL * sm_count()), 256, 0, st>>>(
            part, p.ksplit, n, y);
        err = cudaGetLastError();
    }
    return err;
}

}  // namespace moe
