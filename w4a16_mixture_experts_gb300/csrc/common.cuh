// Device helpers shared by the kernels of libw4a16moe (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "w4a16moe.h"

namespace moe {

constexpr int kGroup = 128;           // quantisation group along K
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr uint32_t kSpinLimit = 1u << 22;   // polls before a wait gives up (~0.5 s)

// ---- workspace layout -------------------------------------------------------
// A fixed control block followed by 256-byte aligned regions; offsets depend
// only on the dims, so host and device agree without storing them.
// Per-expert completion counters sit one 128-byte line apart, so that the
// pollers and the increments of different experts do not share a line.
constexpr int kCtrStride = 32;
constexpr int kRowssMax = 8;   // tokens of the decode stack step's per-token sums

struct Ctrl {
    uint32_t error;          // first MOE_ERR_DEVICE / MOE_ERR_TIMEOUT seen
    uint32_t route_ticket;   // router CTAs done with their logits (small batches; the last resets it)
    uint32_t n_active;       // experts with at least one assignment
    uint32_t bar_arrive;     // grid barrier of the decode stack step: CTAs arrived
    uint32_t bar_depart;     // ... and CTAs done with the rows after it (the last resets both)
    uint32_t exit_count;     // decode CTAs finished (the last resets the per-expert counters)
    uint32_t route_arrive;   // grid barrier of the decode kernel that routes itself: CTAs with their logits stored
    uint32_t pad1[57];
};
static_assert(sizeof(Ctrl) == 256, "control block");

struct WsLayout {
    size_t ctrl;         // Ctrl
    size_t partial;      // f32 [ksplit][T][E (+1)] router partial logits
    size_t counts;       // i32 [E]        per-expert assignment counts
    size_t offsets;      // i32 [E+1]
    size_t active;       // i32 [E]        active expert ids, increasing
    size_t done1;        // u32 [E][kCtrStride] per expert (one 128-byte line each): finished gate_up tasks
    size_t rowss;        // f32 [T]        per token: sum of r^2 (stack epilogue, decode path)
    size_t rbuf;         // f32 [T][H]     residual sums (stack epilogue)
    size_t chunk;        // i32 [nchunk][E] per-chunk counts -> per-chunk bases
    size_t perm;         // i32 [T*k]      slot -> assignment
    size_t inv;          // i32 [T*k]      assignment -> slot (-1: dropped)
    size_t hbuf;         // bf16 [T*k][I]  SiLU(g)*u per slot (fragment order)
    size_t xperm;        // bf16 [T*k][H]  activations per slot, fragment order (prefill path)
    size_t out_acc;      // f32 [T][H]     weighted output accumulator (prefill path)
    size_t n_chunks;     // i32 [1]        chunks in chunk_info (prefill path)
    size_t chunk_info;   // i32x4 [T*k/128+E+1] per chunk of at most 128 tokens: expert, first slot, tokens (prefill path)
    size_t total;
    int ksplit;
    int nchunk;
};

constexpr int kPermChunk = 1024;      // assignments per permute CTA

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Router K split: small batches split K across CTAs so that enough SMs pull
// the router weight; each split must be a whole number of 32-wide K blocks.
// Large batches (the tensor-core router, E a multiple of 128) split K until
// the 128x128 tiles times the splits fill about one wave of 148 CTAs, keeping
// at least four 64-wide K steps per split.
inline bool router_tc(const moe_dims &d) { return d.T > 64 && d.E % 128 == 0; }
inline int router_ksplit(const moe_dims &d) {   // at most 16
    if (router_tc(d)) {
        const int tiles = (d.E / 128) * ((d.T + 127) / 128);
        int s = 1;
        while (s < 8 && tiles * s * 2 <= 148 && d.H / 64 / (s * 2) >= 4) s *= 2;
        return s;
    }
    if (d.T > 64) return 1;
    for (int s = 16; s > 1; s >>= 1)
        if (d.H % (32 * s) == 0 && s <= d.H / 128) return s;
    return 1;
}

// True when the forward calls take the fused decode kernel (T <= 8 and its
// shared-memory layout fits); otherwise they take the prefill pipeline. The
// workspace holds the regions of the path that will run.
bool fused_supported(const moe_dims &d);

inline WsLayout ws_layout(const moe_dims &d) {
    WsLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    const size_t T = (size_t)d.T, E = (size_t)d.E, k = (size_t)d.k;
    const size_t H = (size_t)d.H, I = (size_t)d.I;
    L.ksplit = router_ksplit(d);
    L.nchunk = (int)((T * k + kPermChunk - 1) / kPermChunk);
    // the regions that must be zero when a call starts (each call leaves them
    // so) come first, with sizes and offsets that depend on no dimension, so
    // that calls of different dims can share one workspace (a router call of
    // dims (E, k) and the forward of its layer with a shared expert, dims
    // (E + 1, k + 1), among them)
    L.ctrl = take(sizeof(Ctrl));
    L.rowss = take(kRowssMax * 4);
    L.done1 = take((size_t)kMaxE * kCtrStride * 4);   // every expert id a call can have
    L.partial = take((size_t)L.ksplit * T * (E + 1) * 4);   // (+1: a shared expert's gate row)
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.active = take(E * 4);
    const bool small = fused_supported(d);
    L.rbuf = take(small ? T * H * 4 : 0);
    L.chunk = take((size_t)(L.nchunk > 0 ? L.nchunk : 1) * E * 4);
    L.perm = take(T * k * 4);
    L.inv = take(T * k * 4);
    L.hbuf = take(T * k * I * 2);
    L.xperm = take(small ? 0 : T * k * H * 2);
    L.out_acc = take(small ? 0 : T * H * 4);
    L.n_chunks = take(4);
    L.chunk_info = take(small ? 0 : (T * k / 128 + E + 1) * 16);
    L.total = o;
    return L;
}

template <typename P>
__host__ __device__ inline P *ws_at(void *ws, size_t off) {
    return reinterpret_cast<P *>(reinterpret_cast<char *>(ws) + off);
}

// ---- error word -------------------------------------------------------------
__device__ inline void set_error(Ctrl *c, uint32_t code) { atomicCAS(&c->error, 0u, code); }

// ---- small PTX wrappers -----------------------------------------------------
__device__ inline uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase. Returns false if it gave up.
__device__ inline bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completing `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ inline void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA load of the box at (c0 = inner element, c1 = row), completing on `bar`.
// c0 * element size must be a multiple of 16 bytes.
__device__ inline void tma_load_2d(void *dst, const void *tmap, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Same as tma_load_2d, with an L2 eviction-priority policy (from l2_evict_first()).
__device__ inline void tma_load_2d_hint(void *dst, const void *tmap, int c0, int c1, uint64_t *bar,
                                        uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read once (streamed weights): evict it before other lines.
__device__ inline uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ inline uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ inline void red_release_add_u32(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ inline uint32_t atom_acq_rel_add_u32(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch. A kernel launched with the programmatic
// stream-serialisation attribute may start while the kernel ahead of it in the
// stream is still running; pdl_wait() returns once that kernel has completed
// and its writes are visible (at once for a kernel launched without the
// attribute). Nothing written by an earlier kernel may be read, and nothing an
// earlier kernel reads may be written, before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream, if launched with the attribute, start
// once every CTA of this grid has executed this (or exited).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ inline uint4 ld_cg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only (for the whole kernel) global load through the non-coherent path:
// not volatile, so the compiler may hoist and batch these loads.
__device__ inline uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte shared-memory load. A plain C++ load, so that the compiler may
// schedule it around arithmetic (and software-pipeline loops), while it still
// stays after the mbarrier waits, whose asm carries a memory clobber.
__device__ inline uint4 lds_v4(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

// D = A * B + C, m16n8k16, bf16 inputs, fp32 accumulate.
// A pure register operation: not volatile, so loads of the next step can be
// scheduled ahead of it.
__device__ inline void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- INT4 -> bf16x2 ---------------------------------------------------------
// Word w holds nibbles n0..n7 (low first), each = q + 8. Pair j (0..3) is
// (n_j, n_{j+4}) as bf16x2 with n_j in the low half, converted to q exactly:
// OR-ing a nibble into the mantissa of 128.0 (0x4300) gives 128 + n, and
// subtracting 136 leaves n - 8, both exact in bf16.
// The mask and the bias go into one lop3 ((a & b) | c, table 0xEA) with the
// bias in a register: written as plain C the pair costs a third instruction,
// and the dequantisation loops are bound by the integer pipe.
__device__ inline uint32_t int4_pair_bias(uint32_t w, int j) {
    const uint32_t s = w >> (4 * j);
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(d) : "r"(s), "r"(0x43004300u));
    return d;
}

__device__ inline uint32_t bf16x2_sub136(uint32_t v) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&v);
    const __nv_bfloat162 c = __floats2bfloat162_rn(136.0f, 136.0f);
    __nv_bfloat162 r = __hsub2(a, c);
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ inline uint32_t int4_pair(uint32_t w, int j) { return bf16x2_sub136(int4_pair_bias(w, j)); }

__device__ inline float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ inline float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace moe
