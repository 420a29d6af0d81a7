// Fused decode forward: permute, W4A16 expert GEMMs and combine in one launch.
//
// Computes the fused Marlin MoE of "Running 125B MoE on Three 3090s - vLLM
// Optimization Edition", section 3.3 "MoE block" (moe_align_block_size,
// gate_up, SiluAndMul, down, moe_sum) for decode batches (T <= 8), on
// symmetric INT4 group-128 weights (model card, "What is quantized", group A).
// At decode the layer streams ~2.5 MB of packed weights per active expert
// and does a few FLOPs per byte, so everything here serves the byte stream:
//
//  * One persistent CTA per SM, launched cooperatively (the CTAs wait on one
//    another, so all must be resident) and programmatically behind the
//    router, so that the launch is under way while the router finishes (and
//    the kernel lets the next one launch at its own entry: the next layer's
//    CTAs take the SMs this one frees and prefetch their inputs). Or
//    the kernel runs the router itself (moe_layer_forward): each CTA computes
//    a few router rows, the CTAs meet at a grid-wide barrier, and each selects
//    the top-k from all logits (see f_route); this removes the router's own
//    launch, its last-CTA hand-over and the wait between the kernels. Each CTA
//    first derives the whole token-to-expert permutation from topk_ids in
//    shared memory (every CTA computes the same result), so no separate
//    permute launch sits on the critical path. Each assignment is ranked by
//    comparison (slot = #assignments with a lower expert + #earlier ones with
//    the same expert): a batch holds at most kDecodeMaxT * kMaxK of them.
//  * Work: gate_up tasks (8 gate rows and the matching 8 up rows of one
//    expert, all of K, in chunks of kGC quantisation groups) and output
//    blocks (16 rows of H). A CTA owns whole output blocks: for each of them
//    it runs one down chunk per active expert (the block's 16 rows of that
//    expert's W2, all of K = I), so the sum over experts never leaves the
//    CTA. The gate_up tasks are shared out so that every CTA streams about
//    the same number of bytes. A CTA runs its work as one sequence of
//    chunks: all its gate_up chunks first, then its down chunks. From two
//    rounds of work on, the tasks are dealt in a stride order and each CTA
//    takes them expert by expert, so that experts complete one after another
//    (see task_stride).
//  * One producer warp issues the copies of the sequence (two 2-D TMA boxes
//    per gate_up chunk, one bulk copy per down chunk) into a ring of kNS
//    shared-memory stages completed on mbarriers; its lanes issue side by
//    side. The copy instructions themselves are the limit of this stream (a
//    few tens of ns each per SM, measured), so the small scale rows do not
//    take copies of their own: the producer prefetches them into L2, and
//    each consumer loads its chunk's scales with plain loads before it waits
//    for the chunk's data. The kCons consumer warps take chunks in sequence
//    order by a shared ticket and hand each stage back as soon as they are
//    done with it, so up to kNS copies are in flight per SM.
//  * Weights are dequantised in registers into mma.sync m16n8k16 A fragments
//    (bf16 holds 128 + n exactly, and one lop3 makes a pair); each group's
//    fp32 partial sum is corrected by 136 * sum(x) over the group and scaled
//    by its bf16 scale, so W = q * scale is never rounded. Tokens are the
//    N = 8 side. Activations for small T are staged once per CTA in shared
//    memory, already in fragment order.
//  * A gate_up chunk leaves its partial sums in a shared buffer of its task;
//    the chunk that completes the task sums them in chunk order
//    (deterministic), stores h = SiLU(g) * u (bf16, fragment order) and
//    counts the task in its expert's counter (release).
//  * A down chunk of expert e waits (bounded, acquire, with back-off) until
//    all gate_up tasks of e are counted, then loads h from L2 into registers.
//  * The combine is fused and stays in the CTA: a down chunk writes its fp32
//    outputs per slot into a shared buffer of its block, and the chunk that
//    completes the block's count sums each token's slots in slot order
//    (deterministic) and writes the bf16 output (in the stack variant: the
//    residual sum and its share of sum(r^2); the RMS rescale follows a grid
//    barrier). All counters reset themselves.
#include "common.cuh"
#include "kernels.cuh"
#include "route_dev.cuh"

namespace moe {

constexpr int kFW = 16;              // warps per CTA: kCons consumers, then the producer
constexpr int kCons = 15;            // warps that compute
constexpr int kProd = kCons;         // the warp that issues every weight copy
constexpr int kGC = 5;               // quantisation groups per gate_up chunk
constexpr int kGCMin = 4;            // ... where kGC's stages leave no room to stage the activations
constexpr int kNS = 29;              // stages of the CTA's chunk ring
constexpr int kRedMax = 20480;       // bytes for the gate_up partial-sum buffers
constexpr int kMaxNB = 8;            // partial-sum buffers (gate_up tasks in flight)
constexpr int kP2Rows = 16;          // output rows per down item
// Batches of up to 8 tokens (route + forward at T = 8: 88.6 us here against
// 96.9 us on the tensor-core grouped GEMM of prefill.cu, measured). Beyond, an
// expert can hold more than one 8-token MMA tile, which the gate_up reduction
// slots do not provide for, and the tensor-core path grows more slowly.
constexpr int kDecodeMaxT = 8;
static_assert(kDecodeMaxT <= kRowssMax, "the stack step's per-token sums fit their region");
constexpr int kMaxNT = (kDecodeMaxT + 7) / 8;   // token tiles of 8 per expert
static_assert(kMaxNT == 1, "the gate_up reduction slots hold one token tile");
constexpr int kFastN = 256;          // assignments ranked by comparison: one thread each
static_assert(kDecodeMaxT * kMaxK <= kFastN && kFastN <= kFW * 32, "every assignment has a thread");
constexpr int kFusedSmem = 232448 - 512;   // per-block opt-in limit, less static shared memory

struct FusedParams {
    CUtensorMap tm_w1;   // int32 [E*2I][H/8], box (gcw words, 8 rows)
    const uint16_t *x;
    const int32_t *ids;
    const float *topk_w;
    const uint16_t *w1s;
    const int32_t *w2p;
    const uint16_t *w2s;
    uint16_t *out;       // bf16 [T][H], or nullptr in the stack variant
    uint16_t *next;      // bf16 [T][H] stack variant output
    float eps;
    Ctrl *ctrl;
    uint32_t *done1;     // [E][kCtrStride] finished gate_up tasks (reset by the last CTA to exit)
    float *rowss;        // [T] sum of r^2 per token (stack variant)
    uint16_t *hbuf;      // bf16 [T*k][I], fragment order
    float *rbuf;         // f32 [T][H] residual sums (stack variant)
    int T, H, E, k, I;
    int gcw;             // words per gate_up chunk row (groups per chunk * 16)
    int nkc;             // chunks per gate_up task
    uint32_t stage_bytes;
    uint32_t red_off;    // offset of the gate_up partial sums and counters
    int nb;              // partial-sum buffers
    int nyb;             // output-block buffers
    uint32_t red_area;   // bytes of the partial-sum area: the larger of the partial sums and one block buffer
    uint32_t pro_off;    // offset of the permutation arrays
    uint32_t xs_off;     // offset of the staged activations (0: not staged)
    uint32_t ys_off;     // offset of the output-block buffers (0: in the partial-sum area)
    // the router, when the kernel runs it (E, k above count the shared expert)
    const uint16_t *wr;  // bf16 [E][H] router rows (row E - 1 the shared gate if rgate)
    const float *rbias;  // f32 [E - rgate] or null
    float *logits;       // f32 [T][E] (workspace)
    int32_t *ids_out;    // int32 [T][k] selection (output)
    float *w_out;        // f32 [T][k]
    int rgate;           // 1: a shared expert (slot k - 1 of each token, expert E - 1)
    // the work split's constants per unit of active experts, for the down
    // weights w = 1 and w = kSpreadDownWeight (see fused_split)
    long long sx0[2], sx1[2];
    float sr[2];         // 1 / (the sum of all capacities), or 0: an even split
};

struct FusedLayout {
    uint32_t stage_bytes, red_off, red_area, pro_off, xs_off, ys_off, total;
    int gcw, nkc, nb, nyb;
    bool ok;
};

// At most min(E, T*k) experts are active.
inline int fused_max_active(const moe_dims &d) { return d.E < d.T * d.k ? d.E : d.T * d.k; }

inline uint32_t fused_pro_bytes(const moe_dims &d) {
    const size_t n = (size_t)d.T * d.k;
    const size_t na = (size_t)(fused_max_active(d) > 0 ? fused_max_active(d) : 1);
    return (uint32_t)(align_up(n * 2, 16) * 3 + align_up(kFastN * 4, 16) + align_up(na * 2, 16) * 3 +
                      align_up(d.T * 2, 16) + 4 * kFW * 8 + 16 + align_up(n * 4, 16));
}

// Gate_up partial results: nb buffers of [chunk][lane][4] f32 (a task's
// chunks each leave one), then per buffer a count of finished chunks and of
// finalised tasks, the consumers' chunk ticket, per ring stage the chunk last
// issued into it and the chunk it may take next, the CTA's count of finalised
// gate_up tasks, and per output-block buffer a count of finished down chunks
// and of combined blocks. The nyb output-block buffers of [T*k slots][16 rows]
// f32 have a region of their own where shared memory allows; otherwise they lie
// in the partial-sum area, which holds them once every gate_up task of the CTA
// is finalised.
constexpr int kRingWordsExtra = 5;
inline uint32_t fused_red_bytes(uint32_t area, int nb) {
    return area + (uint32_t)(2 * nb * 4 + 4 + 2 * kNS * 4 + 4 * kRingWordsExtra);
}
struct RingWords {
    int *cnt, *ticket, *dcnt;
    volatile int *fin, *issued, *next, *gu_done, *dfin;
};
__device__ inline RingWords ring_words(uint8_t *smem, const FusedParams &p) {
    int *w = reinterpret_cast<int *>(smem + p.red_off + p.red_area);
    RingWords r;
    r.cnt = w;
    r.fin = w + p.nb;
    r.ticket = w + 2 * p.nb;
    r.issued = w + 2 * p.nb + 1;
    r.next = w + 2 * p.nb + 1 + kNS;
    r.gu_done = w + 2 * p.nb + 1 + 2 * kNS;
    r.dcnt = w + 2 * p.nb + 2 + 2 * kNS;
    r.dfin = w + 2 * p.nb + 4 + 2 * kNS;
    return r;
}

// Shared memory: the CTA's ring of kNS stages | partial sums | permutation
// arrays | staged activations (if they fit) | two output-block buffers (if
// they fit). gc_max: groups per gate_up chunk.
inline FusedLayout fused_layout_gc(const moe_dims &d, int gc_max) {
    FusedLayout L{};
    const int G1 = d.H / 128;
    const int gc = G1 < gc_max ? G1 : gc_max;
    L.gcw = gc * 16;
    L.nkc = (G1 + gc - 1) / gc;
    const uint32_t p1 = 2u * 8 * L.gcw * 4;
    const uint32_t p2 = (uint32_t)kP2Rows * (d.I / 2);
    L.stage_bytes = (uint32_t)align_up(p1 > p2 ? p1 : p2, 128);
    L.nb = kRedMax / (L.nkc * 512);
    L.nb = L.nb < 1 ? 1 : L.nb > kMaxNB ? kMaxNB : L.nb;
    // output-block buffers in the partial-sum area: one or two (the area holds at least one)
    const uint32_t yb = (uint32_t)d.T * d.k * kP2Rows * 4;
    const uint32_t pa = (uint32_t)(L.nb * L.nkc * 512);
    L.red_area = pa > yb ? pa : yb;
    L.nyb = yb ? (int)(L.red_area / yb) : 0;
    L.nyb = L.nyb > 2 ? 2 : L.nyb;
    L.red_off = kNS * L.stage_bytes;
    L.pro_off = L.red_off + (uint32_t)align_up(fused_red_bytes(L.red_area, L.nb), 128);
    // staged activations, then their sum over each 128-wide group (f32 [T][H/128])
    const uint32_t xs_bytes = (uint32_t)d.T * d.H * 2 + (uint32_t)align_up((size_t)d.T * G1 * 4, 16);
    const uint32_t base = L.pro_off + (uint32_t)align_up(fused_pro_bytes(d), 128);
    L.xs_off = base + xs_bytes <= (uint32_t)kFusedSmem ? base : 0;
    L.total = L.xs_off ? base + xs_bytes : base;
    // the output-block buffers in a region of their own, so that a CTA's down
    // chunks need not wait for its last gate_up task (measured at T = 1: the
    // wait held each down chunk about 1 us after its expert was complete)
    const uint32_t ys_start = (uint32_t)align_up(L.total, 128);
    if (yb && ys_start + 2 * yb <= (uint32_t)kFusedSmem) {
        L.ys_off = ys_start;
        L.nyb = 2;
        L.total = ys_start + 2 * yb;
    }
    L.ok = L.total <= (uint32_t)kFusedSmem && d.T <= kDecodeMaxT && d.k <= kMaxK && d.I <= 1280 && L.gcw <= 256 &&
           (L.nyb >= 1 || d.T == 0);
    return L;
}

// kGC groups per chunk (fewer chunks, each task's partial sums in fewer
// slots: measured faster at T = 1 and 4), unless its larger stages leave no
// room to stage the activations or do not fit at all; then kGCMin.
inline FusedLayout fused_layout(const moe_dims &d) {
    const FusedLayout a = fused_layout_gc(d, kGC);
    if (a.ok && a.xs_off) return a;
    const FusedLayout b = fused_layout_gc(d, kGCMin);
    return b.ok && (b.xs_off || !a.ok) ? b : a;
}

bool fused_supported(const moe_dims &d) { return fused_layout(d).ok; }

// Scratch of the router phase at the start of the ring (free until the first
// weight copy): candidate keys, quarter sums, the selection, the logits.
constexpr uint32_t kRtCand = 0;       // uint64 [kRouteWarps][32]
constexpr uint32_t kRtPart = 4096;    // f32 [kRouteWarps][kRouteInlineMaxT]
constexpr uint32_t kRtIds = 4608;     // int32 [T * k] <= kFastN
constexpr uint32_t kRtW = 5632;       // f32 [T * k]
constexpr uint32_t kRtLogit = 6656;   // f32 [T][E]
static_assert(kRtPart >= kRouteWarps * 32 * 8 && kRtIds - kRtPart >= kRouteWarps * kRouteInlineMaxT * 4 &&
                  kRtW - kRtIds >= kFastN * 4 && kRtLogit - kRtW >= kFastN * 4,
              "router scratch");
static_assert(kFW == kRouteWarps, "the router selection runs on the kernel's warps");

// The kernel runs the router itself for batches of up to kRouteFusedMaxT
// tokens. Measured (route + forward in one graph of 10 layers, H 2560, E 512,
// k 10, I 640; separate calls -> one kernel): T = 1 29.91 -> 29.42 us, T = 2
// 36.92 -> 36.63, T = 4 54.75 -> 54.88, T = 7 81.19 -> 82.09, T = 8 88.76 ->
// 89.60. Each CTA reads all T x E logits after the barrier (the same lines,
// from every SM) and selects for every token, which outweighs the saved
// hand-over from 4 tokens on.
constexpr int kRouteFusedMaxT = 2;

bool fused_route_supported(const moe_dims &d) {
    const FusedLayout L = fused_layout(d);
    return L.ok && L.xs_off && d.T <= kRouteFusedMaxT && (size_t)d.T * d.k <= kFastN &&
           kRtLogit + (size_t)d.T * d.E * 4 <= L.red_off;
}

int fused_plan(const moe_dims &d) {
    const FusedLayout L = fused_layout(d);
    if (!L.ok) return 0;
    return (L.xs_off ? 1 : 2) | ((L.gcw / 16) << 4) | (L.ys_off ? 256 : 0) | (fused_route_supported(d) ? 512 : 0);
}

struct Pro {   // permutation arrays in shared memory
    int16_t *ids, *perm, *inv;
    float *wv;      // per assignment: its routing weight
    int32_t *cnt;   // per assignment: 1 if it is its expert's first
    int16_t *act, *aoff, *acnt, *kv;
    uint64_t *bar;
    int *nact;
};

__device__ inline Pro pro_views(uint8_t *smem, const FusedParams &p) {
    Pro v;
    const int n = p.T * p.k;
    uint8_t *q = smem + p.pro_off;
    auto take = [&](size_t bytes) { uint8_t *r = q; q += (bytes + 15) / 16 * 16; return r; };
    v.ids = reinterpret_cast<int16_t *>(take(n * 2));
    v.perm = reinterpret_cast<int16_t *>(take(n * 2));
    v.inv = reinterpret_cast<int16_t *>(take(n * 2));
    v.cnt = reinterpret_cast<int32_t *>(take(kFastN * 4));
    const int na = p.E < n ? p.E : n;
    v.act = reinterpret_cast<int16_t *>(take((na > 0 ? na : 1) * 2));
    v.aoff = reinterpret_cast<int16_t *>(take((na > 0 ? na : 1) * 2));
    v.acnt = reinterpret_cast<int16_t *>(take((na > 0 ? na : 1) * 2));
    v.kv = reinterpret_cast<int16_t *>(take(p.T * 2));
    v.bar = reinterpret_cast<uint64_t *>(take(4 * kFW * 8));
    v.nact = reinterpret_cast<int *>(take(16));
    v.wv = reinterpret_cast<float *>(take(n * 4));
    return v;
}

// mbarriers in v.bar: per ring stage "full" (the producer's copies landed),
// then the activations' bulk copy. A stage changes hands through two shared
// words (RingWords): the producer writes issued[q] = i just before it copies
// chunk i into stage q, which it may do only once next[q] == i; the consumer
// of chunk i waits for issued[q] == i before it waits on the barrier, so the
// barrier's phase is then exactly chunk i's (a parity alone cannot tell chunk
// i from chunk i - 2 * kNS), and sets next[q] = i + kNS when done with it.
static_assert(kNS + 1 <= 4 * kFW, "mbarrier slots");
__device__ inline uint64_t *full_bar(const Pro &v, int q) { return v.bar + q; }
__device__ inline uint64_t *x_bar(const Pro &v) { return v.bar + kNS; }

// The ring's shared words and full barriers, set by the CTA's threads before
// the barrier that ends either prologue.
__device__ __forceinline__ void fused_ring_init(const FusedParams &p, uint8_t *smem, const Pro &v, int tid) {
    const RingWords rw = ring_words(smem, p);
    if (tid < 2 * p.nb + 1) rw.cnt[tid] = 0;   // chunks done, tasks finalised, the ticket
    if (tid < kRingWordsExtra) rw.gu_done[tid] = 0;   // tasks finalised, block counts
    if (tid < kNS) {
        rw.issued[tid] = -1;
        rw.next[tid] = tid;
    }
    // the ring's full barriers (one arrival: the producer's expect_tx)
    if (tid < kNS) {
        mbar_init(v.bar + tid, 1);
        fence_mbar_init();
    }
}

// The stable permutation, in every CTA: the slot of assignment a is
// #{valid a' with a lower expert} + #{a' < a with the same expert}. Thread a
// ranks assignment a (id_reg: its id, already loaded by the caller); the
// first assignment of each expert also places the expert in the active list.
__device__ __forceinline__ void fused_prologue(const FusedParams &p, uint8_t *smem, const Pro &v, int id_reg,
                                               float w_reg) {
    __shared__ int nact_s;
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int n = p.T * p.k, E = p.E;

    bool bad = false;
    if (tid < n) {
        if (id_reg < 0 || id_reg >= E) {
            id_reg = -1;
            bad = true;
        }
        v.ids[tid] = (int16_t)id_reg;
        v.wv[tid] = w_reg;
    }
    if (bad && blockIdx.x == 0) set_error(p.ctrl, MOE_ERR_DEVICE);
    if (tid == 0) nact_s = 0;
    __syncthreads();
    for (int t = tid; t < p.T; t += nthr) {
        int c = 0;
        for (int j = 0; j < p.k; ++j) c += v.ids[t * p.k + j] >= 0;
        v.kv[t] = (int16_t)c;
    }

    int32_t *is_lead = v.cnt;
    const int a = tid;
    int e = -1, cl = 0, rk = 0, ct = 0;
    if (a < n) {
        e = v.ids[a];
        is_lead[a] = 0;
        if (e < 0) {
            v.inv[a] = -1;
        } else {
            for (int a2 = 0; a2 < n; ++a2) {
                const int e2 = v.ids[a2];
                cl += (e2 >= 0) & (e2 < e);
                ct += e2 == e;
                rk += (e2 == e) & (a2 < a);
            }
            const int slot = cl + rk;
            v.perm[slot] = (int16_t)a;
            v.inv[a] = (int16_t)slot;
            if (rk == 0) {
                is_lead[a] = 1;
                atomicAdd(&nact_s, 1);
            }
        }
    }
    __syncthreads();
    if (a < n && e >= 0 && rk == 0) {
        int ai = 0;
        for (int a2 = 0; a2 < n; ++a2) ai += is_lead[a2] & (v.ids[a2] < e);
        v.act[ai] = (int16_t)e;
        v.aoff[ai] = (int16_t)cl;
        v.acnt[ai] = (int16_t)ct;
    }
    if (tid == 0) *v.nact = nact_s;
    fused_ring_init(p, smem, v, tid);
    __syncthreads();
}

// The permutation for the kernel's own selection (f_route) when it has at most
// 32 assignments: every id is valid, so warp 0 sorts the keys (expert << 5 |
// assignment) across its lanes with a bitonic network of shuffles and reads
// the slots, the active-expert list, the first slots and the counts off the
// sorted order: the arrays of fused_prologue, without its three CTA barriers
// (the other warps set up the ring meanwhile). Ties of the expert go by the
// assignment, as there.
__device__ __forceinline__ void f_route_prologue(const FusedParams &p, uint8_t *smem, const Pro &v) {
    const int tid = threadIdx.x;
    const int n = p.T * p.k;   // <= 32
    if (tid < 32) {
        const int lane = tid;
        const int32_t *s_ids = reinterpret_cast<const int32_t *>(smem + kRtIds);
        const float *s_w = reinterpret_cast<const float *>(smem + kRtW);
        int key = 0x7fffffff;   // lanes past n sort last
        if (lane < n) {
            const int e = s_ids[lane];
            v.ids[lane] = (int16_t)e;
            v.wv[lane] = s_w[lane];
            key = (e << 5) | lane;
        }
#pragma unroll
        for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
            for (int j = kk >> 1; j > 0; j >>= 1) {
                const int o = __shfl_xor_sync(0xffffffffu, key, j);
                const bool up = (lane & kk) == 0, low = (lane & j) == 0;
                key = low == up ? min(key, o) : max(key, o);
            }
        const int e = key >> 5, a = key & 31;
        const int eprev = __shfl_up_sync(0xffffffffu, e, 1);
        const bool valid = lane < n;
        const bool start = valid && (lane == 0 || eprev != e);   // the first slot of an expert
        const unsigned starts = __ballot_sync(0xffffffffu, start);
        if (valid) {
            v.perm[lane] = (int16_t)a;
            v.inv[a] = (int16_t)lane;
        }
        if (start) {
            const int ai = __popc(starts & ((1u << lane) - 1u));
            const unsigned later = starts & ~((2u << lane) - 1u);
            v.act[ai] = (int16_t)e;
            v.aoff[ai] = (int16_t)lane;
            v.acnt[ai] = (int16_t)((later ? __ffs(later) - 1 : n) - lane);
        }
        if (lane < p.T) v.kv[lane] = (int16_t)p.k;   // every slot valid
        if (lane == 0) *v.nact = __popc(starts);
    }
    fused_ring_init(p, smem, v, tid);
    __syncthreads();
}

// After the permutation: the activations in fragment order and their
// per-group sums (if staged). Run by the consumer warps only; ends on a named
// barrier among them.
__device__ __noinline__ void fused_stage(const FusedParams &p, uint8_t *smem, const Pro &v) {
    const int tid = threadIdx.x, nthr = kCons * 32;
    const int lane = tid & 31;
    if (p.xs_off) {
        // x arrived row-major (a bulk copy issued at kernel entry); each 16-byte
        // chunk is rewritten in place in fragment order, and per token the sum
        // of each 128-wide group is formed (the gate_up MMAs run on the biased
        // nibbles 128 + n, see f_gate_up_chunk). A row holds H/8 chunks, a
        // multiple of 16, so the 16 chunks of a group sit in 16 consecutive
        // lanes; every lane runs every pass (the count is rounded up to whole
        // warps) so that the shuffles see the full warp.
        if (!mbar_wait(x_bar(v), 0) && tid == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
        uint4 *xs = reinterpret_cast<uint4 *>(smem + p.xs_off);
        float *xsum = reinterpret_cast<float *>(smem + p.xs_off + (size_t)p.T * p.H * 2);
        const int nch = p.T * p.H / 8;
        const int nch32 = (nch + 31) & ~31;
        for (int i = tid; i < nch32; i += nthr) {
            float sum = 0.f;
            if (i < nch) {
                const uint4 c = xs[i];
                xs[i] = make_uint4(__byte_perm(c.x, c.z, 0x5410), __byte_perm(c.x, c.z, 0x7632),
                                   __byte_perm(c.y, c.w, 0x5410), __byte_perm(c.y, c.w, 0x7632));
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    sum += __uint_as_float(w[m] << 16) + __uint_as_float(w[m] & 0xffff0000u);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (i < nch && (lane & 15) == 0) xsum[i / 16] = sum;   // i / 16 = token * (H/128) + group
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kCons * 32) : "memory");
}

__device__ inline uint32_t fw_word(const uint4 &v, int m) {
    return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// ---- the CTA's chunk sequence -----------------------------------------------
// Chunk i of the CTA: for i < m1 * nkc, K chunk i % nkc of the CTA's gate_up
// task u = i / nkc (tab[u], or b1 + u when tab is null; see task_stride);
// after them the down chunks of its nblk output blocks from cb0: block by block
// (each block's chunk for every active expert a), or, with the spread task
// order when every block has a buffer of its own (nblk <= nyb, emaj), expert
// by expert (each expert's chunk for every block), so that a CTA with two
// blocks runs both blocks' chunks of an expert as soon as the expert is
// complete.
// Task ids: gate_up tasks 0..n1-1; the down chunk of output block c and active
// expert a is n1 + c * nact + a, and a CTA's down chunks cover whole blocks.
// The producer issues the chunks in this order and the consumers take them in
// this order.
struct ChunkRef {
    int task, chunk, u;   // u: the CTA's gate_up task index
};

__device__ inline ChunkRef chunk_at(int i, int b1, int m1, int cb0, int nblk, int nact, int n1, int nkc,
                                    const uint16_t *tab, bool emaj) {
    ChunkRef r;
    if (i < m1 * nkc) {
        const int u = i / nkc;
        r.task = tab ? (int)tab[u] : b1 + u;
        r.chunk = i - u * nkc;
        r.u = u;
    } else {
        const int d = i - m1 * nkc;
        const int c = emaj ? cb0 + d % nblk : cb0 + d / nact, a = emaj ? d / nblk : d % nact;
        r.task = n1 + c * nact + a;
        r.chunk = 0;
        r.u = 0;
    }
    return r;
}

__device__ __noinline__ void f_issue(const FusedParams &p, const Pro &v, int task, int chunk, int n1, uint8_t *stage,
                               uint64_t *bar, int lane) {
    if (lane != 0) return;
    const int tp1 = p.I / 8;
    if (task < n1) {
        const int a = task / tp1, r = task - a * tp1;
        const int e = v.act[a];
        const uint32_t box = 8u * p.gcw * 4;
        const int row = e * 2 * p.I + 8 * r;
        mbar_arrive_expect_tx(bar, 2 * box);
        tma_load_2d(stage, &p.tm_w1, chunk * p.gcw, row, bar);
        tma_load_2d(stage + box, &p.tm_w1, chunk * p.gcw, row + p.I, bar);
        if (chunk == 0) {
            // the task's scale rows (8 contiguous rows of G1 bf16 each, gate and up) go to L2
            // now, so that the consumers' loads of them find them there (measured 1-2% at T = 4, 7)
            const int G1 = p.H / 128;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w1s + (size_t)row * G1), "r"((uint32_t)(16 * G1)) : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w1s + (size_t)(row + p.I) * G1), "r"((uint32_t)(16 * G1)) : "memory");
        }
    } else {
        const int t2 = task - n1, nact = *v.nact;
        const int c = t2 / nact, a = t2 - c * nact;   // output block c, active expert a
        const int e = v.act[a];
        const uint32_t rb = p.I / 2;
        mbar_arrive_expect_tx(bar, kP2Rows * rb);
        bulk_g2s(stage, reinterpret_cast<const char *>(p.w2p) + ((size_t)e * p.H + kP2Rows * c) * rb, kP2Rows * rb,
                 bar);
        // the block's scale rows to L2 as well
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w2s + ((size_t)e * p.H + kP2Rows * c) * (p.I / 128)),
                     "r"((uint32_t)(kP2Rows * (p.I / 128) * 2))
                     : "memory");
    }
}

// ---- scales -------------------------------------------------------------------
// A chunk's scales, loaded by its consumer from global memory (L2) before it
// waits for the chunk's weights, held as bf16 pairs: sk[0..4] for the lane's
// first row (gate row g of a gate_up chunk, row g of a down chunk), sk[5..9]
// for its second row (up row g, row g + 8), group q in half q & 1 of word q / 2.
// Indexed by runtime group numbers through selects, never through local memory.
constexpr int kScW = 5;   // words per row: up to 10 groups (I <= 1280, kGC <= 10)
static_assert(kGC <= 2 * kScW, "gate_up chunk scales fit");

__device__ __forceinline__ float scale_of(const uint32_t (&sk)[2 * kScW], int half, int q) {
    const int i = q >> 1;
    uint32_t w = sk[half * kScW];
#pragma unroll
    for (int j = 1; j < kScW; ++j) w = i == j ? sk[half * kScW + j] : w;
    return __uint_as_float((q & 1) ? (w & 0xffff0000u) : (w << 16));
}

// n consecutive scales from row pointer s (2-byte aligned) into half `half` of sk.
__device__ __forceinline__ void load_scales(const uint16_t *s, int n, int half, uint32_t (&sk)[2 * kScW]) {
#pragma unroll
    for (int j = 0; j < kScW; ++j) {
        const uint32_t lo = 2 * j < n ? (uint32_t)__ldg(s + 2 * j) : 0u;
        const uint32_t hi = 2 * j + 1 < n ? (uint32_t)__ldg(s + 2 * j + 1) : 0u;
        sk[half * kScW + j] = lo | (hi << 16);
    }
}

// Scales of chunk `chunk` of gate_up task `task`: its groups q0 .. q0 + qn - 1
// of gate row 8r + g and up row I + 8r + g of the task's expert.
__device__ __forceinline__ void gate_up_scales(const FusedParams &p, const Pro &v, int task, int chunk, int lane,
                                               uint32_t (&sk)[2 * kScW]) {
    const int tp1 = p.I / 8, G1 = p.H / 128, gc = p.gcw / 16;
    const int a = task / tp1, r = task - a * tp1;
    const int q0 = chunk * gc, qn = G1 - q0 < gc ? G1 - q0 : gc;
    const size_t row = (size_t)v.act[a] * 2 * p.I + 8 * r + (lane >> 2);
    load_scales(p.w1s + row * G1 + q0, qn, 0, sk);
    load_scales(p.w1s + (row + p.I) * G1 + q0, qn, 1, sk);
}

// Scales of down chunk t2 (output block c, active expert a): all groups of
// rows 16c + g and 16c + g + 8 of the expert's W2.
__device__ __forceinline__ void down_scales(const FusedParams &p, const Pro &v, int t2, int lane,
                                            uint32_t (&sk)[2 * kScW]) {
    const int nact = *v.nact, G2 = p.I / 128;
    const int c = t2 / nact, a = t2 - c * nact;
    const size_t row = (size_t)v.act[a] * p.H + kP2Rows * c + (lane >> 2);
    load_scales(p.w2s + row * G2, G2, 0, sk);
    load_scales(p.w2s + (row + 8) * G2, G2, 1, sk);
}

// ---- gate_up ----------------------------------------------------------------
// Lane (g, tig) holds, for group q, words 4*tig..4*tig+3 of A rows g (gate)
// and g+8 (up). Word m covers K = base..base+7, base = 128q + 32tig + 8m;
// k-step 2m+h takes nibble pairs (2h, 2h+4) for the low fragment slots and
// (2h+1, 2h+5) for the high ones, so the B fragment of token g is the
// activation chunk base..base+7 in the order (0,4),(1,5),(2,6),(3,7).
template <bool kStaged>
__device__ inline void f_gate_up_chunk(const FusedParams &p, const Pro &v, int task, int chunk, bool first,
                                       const uint8_t *stage, const uint8_t *smem, int lane,
                                       const uint32_t (&sk)[2 * kScW], float (&acc)[kMaxNT][4]) {
    const int tp1 = p.I / 8;
    const int a = task / tp1;
    const int s0 = v.aoff[a], ne = v.acnt[a];
    const int nt_n = (ne + 7) >> 3;
    const int g = lane >> 2, tig = lane & 3;
    const int G1 = p.H / 128;
    const int gc = p.gcw / 16;
    const int q0 = chunk * gc;
    const int qn = G1 - q0 < gc ? G1 - q0 : gc;
    const uint32_t rowb = p.gcw * 4;
    const uint8_t *rg = stage + g * rowb + 16 * tig;
    const uint8_t *ru = stage + 8 * rowb + g * rowb + 16 * tig;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (first) {
#pragma unroll
        for (int nt = 0; nt < kMaxNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
    // staged x: the MMAs take the biased nibble values 128 + n (exact in bf16, no
    // subtraction per weight) and each group's sum is corrected by 136 * sum(x)
    // over the group: sum (n - 8) x = sum (128 + n) x - 136 sum x, in fp32
    const float *xsum = reinterpret_cast<const float *>(smem + p.xs_off + (size_t)p.T * p.H * 2);
    for (int nt = 0; nt < nt_n; ++nt) {
        // activation row of the token in column g of this N tile; columns past
        // ne read the first column's token (always valid) and are never stored
        const int j = 8 * nt + g;
        const int tok = v.perm[s0 + (j < ne ? j : 8 * nt)] / p.k;
        // group sums of the tokens of the output columns 2tig and 2tig+1 (0 past ne)
        const int j0 = 8 * nt + 2 * tig, j1 = j0 + 1;
        const float *xs0 = j0 < ne ? xsum + (size_t)(v.perm[s0 + j0] / p.k) * G1 : nullptr;
        const float *xs1 = j1 < ne ? xsum + (size_t)(v.perm[s0 + j1] / p.k) * G1 : nullptr;
        const uint4 *xb;
        if (kStaged)
            xb = reinterpret_cast<const uint4 *>(smem + p.xs_off) + (size_t)tok * (p.H / 8) + 4 * tig;
        else
            xb = reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.H + 32 * tig);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        // two groups per pass: their load -> dequant -> mma chains overlap
#pragma unroll 2
        for (int qq = 0; qq < qn; ++qq) {
            const int q = q0 + qq;
            const uint4 wg = lds_v4(rg + 64 * qq), wu = lds_v4(ru + 64 * qq);
            const float sg = scale_of(sk, 0, qq);
            const float su = scale_of(sk, 1, qq);
            uint4 X[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                X[m] = kStaged ? xb[16 * q + m] : ld_nc_v4(xb + 16 * q + m);
                if (!kStaged)
                    X[m] = make_uint4(__byte_perm(X[m].x, X[m].z, 0x5410), __byte_perm(X[m].x, X[m].z, 0x7632),
                                      __byte_perm(X[m].y, X[m].w, 0x5410), __byte_perm(X[m].y, X[m].w, 0x7632));
            }
            // the group's 8 MMAs accumulate in one fragment (fewer adds than a
            // fragment per word; the two groups in flight keep the pipe busy)
            float cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t xg = fw_word(wg, m), xu = fw_word(wu, m);
                uint32_t f0[4], f1[4];
                if (kStaged) {
                    f0[0] = int4_pair_bias(xg, 0), f0[1] = int4_pair_bias(xu, 0);
                    f0[2] = int4_pair_bias(xg, 1), f0[3] = int4_pair_bias(xu, 1);
                    f1[0] = int4_pair_bias(xg, 2), f1[1] = int4_pair_bias(xu, 2);
                    f1[2] = int4_pair_bias(xg, 3), f1[3] = int4_pair_bias(xu, 3);
                } else {
                    f0[0] = int4_pair(xg, 0), f0[1] = int4_pair(xu, 0), f0[2] = int4_pair(xg, 1), f0[3] = int4_pair(xu, 1);
                    f1[0] = int4_pair(xg, 2), f1[1] = int4_pair(xu, 2), f1[2] = int4_pair(xg, 3), f1[3] = int4_pair(xu, 3);
                }
                mma_bf16_16816(cc, f0, X[m].x, X[m].y);
                mma_bf16_16816(cc, f1, X[m].z, X[m].w);
            }
            float b0 = 0.f, b1 = 0.f;
            if (kStaged) {
                b0 = xs0 ? 136.f * xs0[q] : 0.f;
                b1 = xs1 ? 136.f * xs1[q] : 0.f;
            }
            a0 += sg * (cc[0] - b0);
            a1 += sg * (cc[1] - b1);
            a2 += su * (cc[2] - b0);
            a3 += su * (cc[3] - b1);
        }
#pragma unroll
        for (int i = 0; i < kMaxNT; ++i)
            if (i == nt) {
                acc[i][0] += a0;
                acc[i][1] += a1;
                acc[i][2] += a2;
                acc[i][3] += a3;
            }
    }
}

// h for intermediate row 8r+g, tokens 8nt+2tig(+1): chunk r, position 2*(g%4) + g/4.
__device__ inline void f_gate_up_store(const FusedParams &p, const Pro &v, int task, int lane,
                                       const float (&acc)[kMaxNT][4]) {
    const int tp1 = p.I / 8;
    const int a = task / tp1, r = task - a * tp1;
    const int s0 = v.aoff[a], ne = v.acnt[a];
    const int g = lane >> 2, tig = lane & 3;
    const int pos = 2 * (g & 3) + (g >> 2);
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int j = 8 * nt + 2 * tig + b;
            if (j < ne) {
                const float hv = silu(acc[nt][b]) * acc[nt][2 + b];
                const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                p.hbuf[(size_t)(s0 + j) * p.I + 8 * r + pos] = *reinterpret_cast<const uint16_t *>(&hb);
            }
        }
}

// The warp has computed K chunk c of gate_up task `task`, the CTA's u-th
// task. Its partial sums go to slot c of buffer u % nb; the warp that
// completes the count of the task's nkc chunks adds the slots in chunk order,
// publishes h and releases the expert's done1 counter. A buffer is written for
// task u only once task u - nb, its previous user, is finalised (its slots
// read): a bounded wait on the buffer's count of finalised tasks. Returns
// false if it gave up.
__device__ inline bool f_gu_reduce(const FusedParams &p, const Pro &v, uint8_t *smem, int task, int u, int c,
                                   int lane, const float (&acc)[kMaxNT][4]) {
    const int b = u % p.nb;
    float4 *slots = reinterpret_cast<float4 *>(smem + p.red_off) + b * p.nkc * 32;
    const RingWords rw = ring_words(smem, p);
    int *cnt = rw.cnt + b;
    volatile int *fin = rw.fin + b;
    uint32_t ok = 1;
    if (lane == 0) {
        uint32_t i = 0;
        while (*fin < u / p.nb)
            if (++i > kSpinLimit) {
                ok = 0;
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    __threadfence_block();
    slots[c * 32 + lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(cnt, 1) + 1 == p.nkc;
        if (last) *cnt = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return true;
    __threadfence_block();
    float sum[kMaxNT][4];
    float4 a = slots[lane];
    sum[0][0] = a.x, sum[0][1] = a.y, sum[0][2] = a.z, sum[0][3] = a.w;
    for (int q = 1; q < p.nkc; ++q) {
        a = slots[q * 32 + lane];
        sum[0][0] += a.x, sum[0][1] += a.y, sum[0][2] += a.z, sum[0][3] += a.w;
    }
    f_gate_up_store(p, v, task, lane, sum);
    // the warp's h stores are ordered before lane 0's release by the warp barrier
    __syncwarp();
    if (lane == 0) {
        red_release_add_u32(&p.done1[(size_t)v.act[task / (p.I / 8)] * kCtrStride], 1u);
        __threadfence_block();
        *fin = u / p.nb + 1;
        atomicAdd(const_cast<int *>(rw.gu_done), 1);   // after the slots' last reads (fence above)
    }
    return true;
}

// ---- down + fused combine ----------------------------------------------------
// Output block c (rows 16c .. 16c + 15) of every token, from the block's slot
// buffer ys [T*k slots][16 rows] f32 in shared memory: out[t][n] = sum over
// j < k, in slot order, of w[t][j] * y[slot of (t, j)][n]; a slot whose id was
// invalid adds nothing (and a token with no valid slot gets 0). Lane l takes
// row l % 16 of tokens l / 16, l / 16 + 2, ... The stack variant keeps
// r = x + out and adds the block's share of sum(r^2) to the token's row sum.
__device__ __noinline__ void f_block_combine(const FusedParams &p, const Pro &v, const float *ys, int c, int lane) {
    const int r = lane & 15;
    const int n = kP2Rows * c + r;
    for (int t0 = 0; t0 < p.T; t0 += 2) {
        const int t = t0 + (lane >> 4);
        const bool on = t < p.T;
        float s = 0.f;
        if (on) {
            for (int j = 0; j < p.k; ++j) {
                const int slot = v.inv[t * p.k + j];
                if (slot >= 0) s += v.wv[t * p.k + j] * ys[slot * kP2Rows + r];
            }
        }
        if (p.out) {
            const __nv_bfloat16 b = __float2bfloat16_rn(s);
            if (on) p.out[(size_t)t * p.H + n] = *reinterpret_cast<const uint16_t *>(&b);
        } else {
            // stack step: keep r = x + moe(x) and add this block's share of sum(r^2)
            const float rr = on ? s + bf16_bits_to_f32(p.x[(size_t)t * p.H + n]) : 0.f;
            if (on) p.rbuf[(size_t)t * p.H + n] = rr;
            float ss = rr * rr;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (on && r == 0) atomicAdd(&p.rowss[t], ss);
        }
    }
}

// Stack step, after every CTA has combined its blocks (a grid barrier on two
// self-resetting counters; every CTA of the grid becomes resident, see the
// launch, and the wait is bounded): one CTA per token scales its row by
// 1/sqrt(mean(r^2) + eps) with 16-byte loads.
__device__ __noinline__ void f_stack_rows(const FusedParams &p) {
    __shared__ float s_scale;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add_u32(&p.ctrl->bar_arrive, 1u);
        uint32_t i = 0;
        while (ld_acquire_u32(&p.ctrl->bar_arrive) < gridDim.x)
            if (++i > kSpinLimit) {
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
    }
    __syncthreads();
    for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
        if (threadIdx.x == 0) {
            const float ss = __ldcg(&p.rowss[t]);
            p.rowss[t] = 0.f;
            s_scale = rsqrtf(ss / (float)p.H + p.eps);
        }
        __syncthreads();
        const float sc = s_scale;
        const float *row = p.rbuf + (size_t)t * p.H;
        uint16_t *nrow = p.next + (size_t)t * p.H;
        for (int n = 4 * threadIdx.x; n < p.H; n += 4 * blockDim.x) {
            const float4 r = __ldcg(reinterpret_cast<const float4 *>(row + n));
            __nv_bfloat162 lo = __floats2bfloat162_rn(r.x * sc, r.y * sc), hi = __floats2bfloat162_rn(r.z * sc, r.w * sc);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(nrow + n) = u;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0 && atomicAdd(&p.ctrl->bar_depart, 1u) + 1 == gridDim.x) {
        // every CTA has passed the barrier and finished its rows
        p.ctrl->bar_arrive = 0;
        p.ctrl->bar_depart = 0;
    }
}

// Down chunk t2 = (output block c, active expert a): y of the expert's slots for
// the block's 16 rows, into the block's slot buffer; the chunk that completes
// the block's count combines it. cb0: the CTA's first block (its blocks use
// the nyb buffers in turn).
__device__ inline bool f_down(const FusedParams &p, const Pro &v, uint8_t *smem, int t2, int cb0, int m1,
                              const uint8_t *stage, int lane, const uint32_t (&sk)[2 * kScW]) {
    const int tp1 = p.I / 8;
    const int nact = *v.nact;
    const int c = t2 / nact, a = t2 - c * nact;
    const int e = v.act[a];
    const int s0 = v.aoff[a], ne = v.acnt[a];
    const int g = lane >> 2, tig = lane & 3;
    const int G2 = p.I / 128;
    const uint32_t rb = p.I / 2;

    // wait until every gate_up task of expert e has published its h (polls
    // back off from 64 to 512 ns, so that the pollers of an expert leave its
    // counter's L2 line to the increments)
    uint32_t ok = 1;
    if (lane == 0) {
        uint32_t i = 0, ns = 64;
        while (ld_acquire_u32(&p.done1[(size_t)e * kCtrStride]) < (uint32_t)tp1) {
            if (++i > kSpinLimit) {
                ok = 0;
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
            __nanosleep(ns);
            if (ns < 512) ns *= 2;
        }
    }
    // the block's slot buffer is free once the block that used it before (nyb
    // blocks earlier) is combined, and, when it lies in the gate_up partial-sum
    // area, once every gate_up task of this CTA is finalised
    const RingWords rw = ring_words(smem, p);
    const int lb = c - cb0, buf = lb % p.nyb;
    if (lane == 0 && ok) {
        uint32_t i = 0;
        while ((!p.ys_off && *rw.gu_done < m1) || rw.dfin[buf] < lb / p.nyb)
            if (++i > kSpinLimit) {
                ok = 0;
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) return false;
    __threadfence_block();
    float *ys = reinterpret_cast<float *>(smem + (p.ys_off ? p.ys_off : p.red_off)) + (size_t)buf * p.T * p.k * kP2Rows;

    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int np = 0; np < ne; np += 8) {
        const int j = np + g;
        const bool valid = j < ne;
        const uint4 *hb = reinterpret_cast<const uint4 *>(p.hbuf + (size_t)(s0 + (valid ? j : 0)) * p.I) + 4 * tig;
        constexpr int kSub = kP2Rows / 16;
        float acc[kSub][4];
#pragma unroll
        for (int s = 0; s < kSub; ++s) acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
        // one group of K: dequantise the rows' words, 8 MMAs against h, scale
        auto group = [&](int q, const uint4 (&Y)[4]) {
#pragma unroll
            for (int s = 0; s < kSub; ++s) {
                const int R = 16 * s + g;
                const uint4 w0 = lds_v4(stage + R * rb + 64 * q + 16 * tig);
                const uint4 w1 = lds_v4(stage + (R + 8) * rb + 64 * q + 16 * tig);
                const float s0v = scale_of(sk, 0, q);
                const float s1v = scale_of(sk, 1, q);
                float cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t x0 = fw_word(w0, m), x1 = fw_word(w1, m);
                    const uint32_t f0[4] = {int4_pair(x0, 0), int4_pair(x1, 0), int4_pair(x0, 1), int4_pair(x1, 1)};
                    const uint32_t f1[4] = {int4_pair(x0, 2), int4_pair(x1, 2), int4_pair(x0, 3), int4_pair(x1, 3)};
                    mma_bf16_16816(cc, f0, Y[m].x, Y[m].y);
                    mma_bf16_16816(cc, f1, Y[m].z, Y[m].w);
                }
                acc[s][0] += s0v * cc[0];
                acc[s][1] += s0v * cc[1];
                acc[s][2] += s1v * cc[2];
                acc[s][3] += s1v * cc[3];
            }
        };
        // h comes from L2: a ring of 4 groups in registers, the first 4 loaded
        // before the first MMA and each slot refilled with the group 4 ahead
        // once it has been used, so the latencies overlap
        constexpr int kRing = 4, kUnrolled = 8;   // groups handled by the unrolled loop (I <= 1024)
        uint4 Yr[kRing][4];
#pragma unroll
        for (int q = 0; q < kRing; ++q)
#pragma unroll
            for (int m = 0; m < 4; ++m) Yr[q][m] = q < G2 ? ld_cg_v4(hb + 16 * q + m) : zero;
#pragma unroll
        for (int q = 0; q < kUnrolled; ++q)
            if (q < G2) {
                group(q, Yr[q % kRing]);
                if (q + kRing < kUnrolled && q + kRing < G2) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) Yr[q % kRing][m] = ld_cg_v4(hb + 16 * (q + kRing) + m);
                }
            }
#pragma unroll 1
        for (int q = kUnrolled; q < G2; ++q) {
            uint4 Y[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) Y[m] = ld_cg_v4(hb + 16 * q + m);
            group(q, Y);
        }
#pragma unroll
        for (int s = 0; s < kSub; ++s)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int jj = np + 2 * tig + b;
                if (jj < ne) {
                    float *yr = ys + (s0 + jj) * kP2Rows + 16 * s + g;
                    yr[0] = acc[s][b];
                    yr[8] = acc[s][2 + b];
                }
            }
    }

    // count the chunk in its block; the chunk that completes the block combines
    // it (the warp barrier and fence order every lane's stores before the count,
    // and the count's reader sees them after its own fence)
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(rw.dcnt + buf, 1) + 1 == nact;
        if (last) rw.dcnt[buf] = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
        __threadfence_block();
        f_block_combine(p, v, ys, c, lane);
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            rw.dfin[buf] = lb / p.nyb + 1;
        }
    }
    return true;
}

// The CTA that exits last (every other CTA has counted itself after all its
// work) sets the active experts' gate_up counters back to zero for the next
// call, and the exit count itself.
__device__ __noinline__ void f_exit(const FusedParams &p, const Pro &v) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) s_last = atom_acq_rel_add_u32(&p.ctrl->exit_count, 1u) + 1 == gridDim.x;
    __syncthreads();
    if (!s_last) return;
    const int nact = *v.nact;
    for (int a = threadIdx.x; a < nact; a += blockDim.x) p.done1[(size_t)v.act[a] * kCtrStride] = 0;
    if (threadIdx.x == 0) {
        p.ctrl->route_arrive = 0;
        p.ctrl->exit_count = 0;
    }
}

// The producer warp: lane l issues chunks l, l + 32, ... of the CTA's
// sequence, chunk i into ring stage i % kNS once the stage has been handed
// back for it (next[q] == i). The lanes poll without blocking, so they issue
// side by side and the requests go out nearly in sequence order. No cycle can
// form: consumers take chunks in sequence order (a ticket), gate_up chunks
// first; a consumer hands a gate_up stage back as soon as its words are in
// registers, and its one wait after that (for the previous user of its
// partial-sum buffer, an earlier task) never holds up the oldest unfinished
// task, whose chunks were all taken before; a down item holds its stage until
// the expert's gate_up tasks are done, in any CTA, and those need gate_up
// chunks only. The loop is bounded. Before the warp leaves, lane q waits
// (bounded) for the last copy issued into stage q, so that none lands after
// the CTA has exited.
__device__ __noinline__ void f_produce(const FusedParams &p, const Pro &v, uint8_t *smem, int b1, int m1, int cb0,
                                       int nblk, int n1, const uint16_t *tab, bool emaj) {
    const int l = threadIdx.x & 31;
    const RingWords rw = ring_words(smem, p);
    const int nact = *v.nact;
    const int nc = m1 * p.nkc + nblk * nact;
    int i = l;   // next chunk of this lane
    uint32_t polls = 0;
    bool ok = true;
    while (__any_sync(0xffffffffu, i < nc)) {
        // the consumers' first chunks go out one pass ahead of the rest, so
        // that they are not interleaved with later requests
        if (i < nc && (polls > 0 || i < kCons)) {
            const int q = i % kNS;
            if (rw.next[q] == i) {
                // (the previous consumer's reads of the stage completed before it
                // handed the stage back)
                rw.issued[q] = i;
                const ChunkRef r = chunk_at(i, b1, m1, cb0, nblk, nact, n1, p.nkc, tab, emaj);
                f_issue(p, v, r.task, r.chunk, n1, smem + (size_t)q * p.stage_bytes, full_bar(v, q), 0);
                i += 32;
            }
        }
        if (++polls > 16u * kSpinLimit) {
            ok = false;
            break;
        }
    }
    if (!ok && l == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
    __syncwarp();
    if (l < kNS) {
        const int j = rw.issued[l];
        if (j >= 0) mbar_wait(full_bar(v, l), (j / kNS) & 1);
    }
}

// ---- the router, run by the kernel itself ------------------------------------
// Router rows 4 (C r + b) .. 4 (C r + b) + 3 go to CTA b of C in pass r, four
// warps a row, with the small-batch router's own code (route_dev.cuh), so the
// logits, the selected experts and their weights are those of moe_route bit
// for bit. The logits go to the workspace; the CTAs meet at a grid-wide
// barrier (a count on the control block: each CTA adds itself with release
// semantics after its stores, thread 0 polls with acquire, bounded); then
// every CTA loads all T x E logits into its ring (free until the first weight
// copy) and selects for itself, so that no second hand-over follows. CTA 0
// writes the selection out. Thread a < T k leaves with assignment a's id and
// weight. The activations were copied into shared memory (row-major) at entry
// and are rewritten in fragment order only later (fused_stage). Inlined, so
// that its shared-memory accesses are known to be shared (a call passes a
// generic pointer).
__device__ __forceinline__ void f_route(const FusedParams &p, uint8_t *smem, const Pro &v, int &id_reg,
                                        float &w_reg) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Eg = p.E, Er = p.E - p.rgate, kr = p.k - p.rgate;
    uint64_t(*s_cand)[32] = reinterpret_cast<uint64_t(*)[32]>(smem + kRtCand);
    float(*s_part)[kRouteInlineMaxT] = reinterpret_cast<float(*)[kRouteInlineMaxT]>(smem + kRtPart);
    int32_t *s_ids = reinterpret_cast<int32_t *>(smem + kRtIds);
    float *s_w = reinterpret_cast<float *>(smem + kRtW);
    float *s_logit = reinterpret_cast<float *>(smem + kRtLogit);
    const uint4 *xs = reinterpret_cast<const uint4 *>(smem + p.xs_off);
    const int C = gridDim.x, b4 = 4 * (int)blockIdx.x;
    // the first pass's row loads go out before the wait for the activations
    RouteQuarter rq = route_quarter(p.wr, b4 + (warp >> 2), Eg, p.H, warp & 3);
    uint4 wv[kRouteLoads];
    route_quarter_load(rq, rq.c_lo, lane, wv);
    if (!mbar_wait(x_bar(v), 0) && tid == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
    for (int e0 = b4; e0 < Eg; e0 += 4 * C) {
        if (e0 != b4) {
            rq = route_quarter(p.wr, e0 + (warp >> 2), Eg, p.H, warp & 3);
            route_quarter_load(rq, rq.c_lo, lane, wv);
        }
        float acc[kRouteInlineMaxT];
        route_quarter_dot(rq, xs, p.T, p.H, lane, wv, acc);
#pragma unroll
        for (int t = 0; t < kRouteInlineMaxT; ++t) {
            if (t >= p.T) break;
            if (lane == 0) s_part[warp][t] = acc[t];
        }
        __syncthreads();
        if (tid < 4 * kRouteInlineMaxT) {
            const int jj = tid / kRouteInlineMaxT, t = tid % kRouteInlineMaxT;
            const int ee = e0 + jj;
            if (t < p.T && ee < Eg) p.logits[(size_t)t * Eg + ee] = route_logit(s_part, jj, t, p.rbias, ee, Er);
        }
        __syncthreads();   // (orders the logit stores before the release below, and s_part's reuse)
    }
    if (tid == 0) {
        red_release_add_u32(&p.ctrl->route_arrive, 1u);
        uint32_t i = 0;
        while (ld_acquire_u32(&p.ctrl->route_arrive) < (uint32_t)C)
            if (++i > kSpinLimit) {
                set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
    }
    __syncthreads();
    route_load_logits(s_logit, p.logits, p.T * Eg);
    __syncthreads();
    route_select(s_logit, p.T, Er, kr, p.rgate, s_cand, s_ids, s_w);
    __syncthreads();
    if (tid < p.T * p.k) {
        id_reg = s_ids[tid];
        w_reg = s_w[tid];
        if (blockIdx.x == 0) {
            p.ids_out[tid] = id_reg;
            p.w_out[tid] = w_reg;
        }
    }
}

// ---- work split ---------------------------------------------------------------
// CTA cb of C owns output blocks [cb0, cb1) = [B cb / C, B (cb + 1) / C), B = H/16.
// The gate_up tasks are shared out in proportion to each CTA's capacity: an
// equal share of all the bytes (gate_up tasks and down chunks) minus w times the
// bytes of its own blocks' down chunks (at least 0). Every term is a multiple of
// the number of active experts, so the capacities' prefix sums are those of
// launch constants (x0, x1: the capacity of a CTA with bmin or bmin + 1 blocks,
// per active expert, in units of 8 bytes): cum(c) = c x0 + nbig(c) (x1 - x0),
// nbig(c) the CTAs among [0, c) with bmin + 1 blocks. CTA c's tasks start at
// f(c) = floor(n1 * (fp32(cum(c)) * r)), r = fp32(1 / cum(C)) from the host,
// with f(0) = 0 and f(C) = n1: non-decreasing in c and the same value in every
// CTA that evaluates it, so the CTAs' ranges tile [0, n1) exactly. (A few
// multiplies on the critical path of every CTA; the exact quotient in 64-bit
// integers cost about 1 us at T = 1, measured.)
__device__ inline int split_at(const FusedParams &p, int c, int C, int n1, int wi) {
    if (c <= 0) return 0;
    if (c >= C) return n1;
    const float r = p.sr[wi];
    if (r == 0.f) return n1 * c / C;
    const int B = p.H / kP2Rows, bmin = B / C;
    const int nbig = B * c / C - bmin * c;
    const long long cum = (long long)c * p.sx0[wi] + (long long)nbig * (p.sx1[wi] - p.sx0[wi]);
    return __float2int_rd(__fmul_rn((float)n1, __fmul_rn((float)cum, r)));
}

// wi = 1: with the spread task order (see task_stride) and the down chunks
// expert by expert, the down work of a CTA with more blocks runs while the
// experts complete, so such CTAs take less gate_up work (w = 2; measured at
// T = 4: the CTAs with two blocks, then without gate_up work, end with the
// others; route + forward 56.9 -> 55.2 us at T = 4, 83.9 -> 81.7 us at T = 7).
constexpr int kSpreadDownWeight = 2;
__device__ inline void fused_split(const FusedParams &p, int nact, int C, int cb, int wi, int &b1, int &m1, int &cb0,
                                   int &cb1) {
    const int B = p.H / kP2Rows;
    const int n1 = nact * (p.I / 8);
    cb0 = B * cb / C;
    cb1 = B * (cb + 1) / C;
    b1 = split_at(p, cb, C, n1, wi);
    m1 = split_at(p, cb + 1, C, n1, wi) - b1;
}

// The host's half of the split: x0, x1 and r for w = 1 and w = kSpreadDownWeight.
void fused_split_constants(const moe_dims &d, int C, FusedParams &p) {
    const long long B = d.H / kP2Rows, bmin = B / C;
    const long long unit = (long long)(d.I / 8) * d.H + B * d.I;   // all bytes / 8, per active expert
    for (int wi = 0; wi < 2; ++wi) {
        const long long w = wi ? kSpreadDownWeight : 1;
        const long long c0 = unit - C * w * d.I * bmin, c1 = unit - C * w * d.I * (bmin + 1);
        const long long x0 = c0 > 0 ? c0 : 0, x1 = c1 > 0 ? c1 : 0;
        const long long all = C * x0 + (B - bmin * C) * (x1 - x0);
        p.sx0[wi] = x0;
        p.sx1[wi] = x1;
        p.sr[wi] = all > 0 ? (float)(1.0 / (double)all) : 0.f;
    }
}

// The CTA's gate_up tasks are the positions b1 .. b1 + m1 - 1 of a global
// order of all n1 tasks. When the gate_up work spans more than two rounds of
// the consumer warps, position x holds task x * M mod n1 (M coprime to n1, about
// 0.618 n1: consecutive positions land far apart), and each CTA takes its tasks
// in increasing order, i.e. expert by expert: every expert's tasks are then
// spread over many CTAs and sit at the same relative place in each CTA's
// sequence, so the experts complete one after another through the gate_up
// phase instead of all at its end, and a CTA whose gate_up work ends early
// (one with two output blocks) finds early experts' h ready for its down
// chunks. (Measured at T = 4 with the task order itself: the CTAs with two
// output blocks ended 25% after the others.) Otherwise (M = 0) position x is
// task x. The same in every CTA.
static_assert(kFastN * 4 >= kFW * 32 * 2, "the sorted task list (one uint16 per thread) fits the prologue's scratch");
static_assert(kDecodeMaxT * kMaxK * (1280 / 8) < 65536, "gate_up task ids fit 16 bits");
// gcd(a, b) == 1 for 0 < a, b < 2^16, by the binary method (shifts and
// subtractions: a chain of integer divisions cost about 3 us here, measured).
__device__ inline bool coprime(uint32_t a, uint32_t b) {
    if (((a | b) & 1u) == 0) return false;
    a >>= __ffs(a) - 1;
    while (b) {
        b >>= __ffs(b) - 1;
        if (a > b) {
            const uint32_t t = a;
            a = b;
            b = t;
        }
        b -= a;
    }
    return a == 1;
}

// Called by whole warps: the lanes test 32 candidates at a time.
__device__ inline int task_stride(int n1, int nkc, int C) {
    if ((long long)n1 * nkc <= 2LL * kCons * C) return 0;
    if (n1 <= 2) return 1;
    const int M0 = (int)(((long long)n1 * 633) >> 10);   // about 0.618 n1, at least 1
    const int lane = threadIdx.x & 31;
    for (int base = M0;; base += 32) {   // ends by M = n1 - 1, coprime to n1
        const int M = base + lane;
        const unsigned ok = __ballot_sync(0xffffffffu, M < n1 && coprime((uint32_t)M, (uint32_t)n1));
        if (ok) return base + __ffs(ok) - 1;
    }
}

// ---- kernel -----------------------------------------------------------------
// kSpread: the launch may hold enough gate_up work for the spread task order
// (see task_stride); without it the task order is the plain one, in code that
// carries nothing of the other (measured: 0.3 us at T = 1 otherwise).
// kRoute: the kernel runs the router itself (f_route; needs kStaged).
template <bool kStaged, bool kSpread, bool kRoute>
__global__ void __launch_bounds__(kFW * 32, 1) decode_fused_kernel(const __grid_constant__ FusedParams p) {
    static_assert(!kRoute || kStaged, "the router reads the staged activations");
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_w1) : "memory");
    const Pro v = pro_views(smem, p);
    if (p.xs_off && threadIdx.x == 0) {
        mbar_init(x_bar(v), 1);
        fence_mbar_init();
    }
    // The kernel behind this one may launch now: its CTAs take the SMs that
    // this grid's CTAs free and set up, and wait for this grid's end before
    // they read anything (every input of this kernel, too, is read only after
    // its own wait below, since the kernel ahead may be one of these).
    pdl_launch_dependents();
    if (!kRoute && p.xs_off && threadIdx.x == 4)   // x heads for L2 (read after the wait)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.x), "r"((uint32_t)p.T * p.H * 2) : "memory");
    if (kRoute && threadIdx.x < 5) {
        // the CTA's first router rows and the activations head for L2 while the
        // kernel ahead finishes (a prefetch into L2, the point of coherence,
        // reads nothing stale; the loads themselves come after the wait)
        const int e = 4 * (int)blockIdx.x + (int)threadIdx.x;
        if (threadIdx.x < 4 && e < p.E)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.wr + (size_t)e * p.H),
                         "r"((uint32_t)p.H * 2) : "memory");
        if (threadIdx.x == 4)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.x), "r"((uint32_t)p.T * p.H * 2)
                         : "memory");
    }
    // The launch is programmatic: the CTAs may start while the kernel ahead
    // (the router, or the layer before) still runs, and read its outputs (and
    // the workspace) only once it has finished.
    pdl_wait();
    // the ids are the first thing every path needs
    int id_reg = -1;
    float w_reg = 0.f;
    if (p.xs_off && threadIdx.x == 0) {
        // x may come from the kernel ahead, so it is copied only now
        const uint32_t xb = (uint32_t)p.T * p.H * 2;
        mbar_arrive_expect_tx(x_bar(v), xb);
        bulk_g2s(smem + p.xs_off, p.x, xb, x_bar(v));
    }
    if constexpr (kRoute) {
        __syncthreads();   // (the barrier's initialisation is visible to every thread)
        f_route(p, smem, v, id_reg, w_reg);
        if (p.T * p.k <= 32)
            f_route_prologue(p, smem, v);
        else
            fused_prologue(p, smem, v, id_reg, w_reg);
    } else {
        if ((int)threadIdx.x < p.T * p.k) {
            id_reg = p.ids[threadIdx.x];
            w_reg = p.topk_w[threadIdx.x];
        }
        fused_prologue(p, smem, v, id_reg, w_reg);
    }

    const int nact = *v.nact;
    const int n1 = nact * (p.I / 8);
    int b1, m1, cb0, cb1;
    // the task order (see task_stride; the same in every CTA), then the split,
    // whose weight w and the down order follow it: with the plain order,
    // w = 1 and block by block (measured faster at T = 1)
    const int M = kSpread ? task_stride(n1, p.nkc, gridDim.x) : 0;
    fused_split(p, nact, gridDim.x, blockIdx.x, M != 0 ? 1 : 0, b1, m1, cb0, cb1);
    const int nblk = cb1 - cb0, m2 = nblk * nact;   // down chunks of whole blocks
    const bool emaj = M != 0 && nblk <= p.nyb;
    // the CTA's gate_up tasks in increasing order, in the prologue's scratch
    // array, free now; with M = 0, or more tasks than threads, the tasks are
    // b1 + u (the partition is M's either way)
    const uint16_t *tab = nullptr;
    if (kSpread && M != 0 && m1 <= kFW * 32) {
        uint16_t *t16 = reinterpret_cast<uint16_t *>(v.cnt);
        const int j = threadIdx.x;
        if (j < m1) {
            const int tj = (int)(((unsigned)(b1 + j) * (unsigned)M) % (unsigned)n1);
            int rank = 0;
            int t2 = (int)(((unsigned)b1 * (unsigned)M) % (unsigned)n1);
            for (int i2 = 0; i2 < m1; ++i2) {
                rank += t2 < tj;
                t2 += M;
                if (t2 >= n1) t2 -= n1;
            }
            t16[rank] = (uint16_t)tj;
        }
        __syncthreads();
        tab = t16;
    }
    if (warp == kProd) {
        f_produce(p, v, smem, b1, m1, cb0, nblk, n1, tab, emaj);
    } else {
        // the activations, converted while the producer requests the first chunks
        fused_stage(p, smem, v);
        const int ngu = m1 * p.nkc, nc = ngu + m2;
        const RingWords rw = ring_words(smem, p);
        // no valid assignment at all: the blocks still get their output (0, or x
        // in the stack variant) from a combine over no slots
        if (nact == 0)
            for (int c = cb0 + warp; c < cb1; c += kCons) f_block_combine(p, v, nullptr, c, lane);
        float acc[kMaxNT][4];
        for (;;) {
            // chunks are taken in sequence order
            int i = 0;
            if (lane == 0) i = atomicAdd(rw.ticket, 1);
            i = __shfl_sync(0xffffffffu, i, 0);
            if (i >= nc) break;
            const int q = i % kNS;
            uint8_t *stage = smem + (size_t)q * p.stage_bytes;
            const ChunkRef r = chunk_at(i, b1, m1, cb0, nblk, nact, n1, p.nkc, tab, emaj);
            // the chunk's scales travel while it waits for its weights
            uint32_t sk[2 * kScW];
            if (r.task < n1) gate_up_scales(p, v, r.task, r.chunk, lane, sk);
            else down_scales(p, v, r.task - n1, lane, sk);
            // chunk i's copy has been issued into stage q (then the barrier's
            // pending phase is chunk i's), and has landed
            uint32_t ok = 1;
            if (lane == 0) {
                uint32_t n = 0;
                while (rw.issued[q] != i)
                    if (++n > kSpinLimit) {
                        ok = 0;
                        break;
                    }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || !mbar_wait(full_bar(v, q), (i / kNS) & 1)) {
                if (lane == 0) set_error(p.ctrl, MOE_ERR_TIMEOUT);
                break;
            }
            if (r.task < n1) {
                f_gate_up_chunk<kStaged>(p, v, r.task, r.chunk, true, stage, smem, lane, sk, acc);
                // the stage is free as soon as its words are in registers
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    rw.next[q] = i + kNS;
                }
                if (!f_gu_reduce(p, v, smem, r.task, r.u, r.chunk, lane, acc)) break;
            } else {
                f_down(p, v, smem, r.task - n1, cb0, m1, stage, lane, sk);
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    rw.next[q] = i + kNS;
                }
            }
        }
        if (p.xs_off && threadIdx.x == 0) mbar_wait(x_bar(v), 0);   // complete already, unless its wait gave up
    }
    if (!p.out) f_stack_rows(p);
    f_exit(p, v);
}

cudaError_t launch_decode_fused(const ExpertArgs &a, const moe_dims &d, void *ws, uint16_t *out, uint16_t *next,
                                float eps, cudaStream_t s, const RouteArgs *r) {
    const WsLayout W = ws_layout(d);
    const FusedLayout L = fused_layout(d);
    if (!L.ok || (r && !fused_route_supported(d))) return cudaErrorInvalidValue;
    FusedParams p;
    cudaError_t err = encode_tmap_2d(&p.tm_w1, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, a.w1p, (uint64_t)d.H / 8,
                                     (uint64_t)d.E * 2 * d.I, (uint64_t)d.H / 2, (uint32_t)L.gcw, 8u,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    p.x = a.x;
    p.ids = a.ids;
    p.topk_w = a.topk_w;
    p.w1s = a.w1s;
    p.w2p = a.w2p;
    p.w2s = a.w2s;
    p.out = next ? nullptr : out;
    p.next = next;
    p.eps = eps;
    p.ctrl = ws_at<Ctrl>(ws, W.ctrl);
    p.done1 = ws_at<uint32_t>(ws, W.done1);
    p.rowss = ws_at<float>(ws, W.rowss);
    p.hbuf = ws_at<uint16_t>(ws, W.hbuf);
    p.rbuf = ws_at<float>(ws, W.rbuf);
    p.T = d.T;
    p.H = d.H;
    p.E = d.E;
    p.k = d.k;
    p.I = d.I;
    p.gcw = L.gcw;
    p.nkc = L.nkc;
    p.stage_bytes = L.stage_bytes;
    p.red_off = L.red_off;
    p.nb = L.nb;
    p.nyb = L.nyb;
    p.red_area = L.red_area;
    p.pro_off = L.pro_off;
    p.xs_off = L.xs_off;
    p.ys_off = L.ys_off;
    p.wr = r ? r->wr : nullptr;
    p.rbias = r ? r->bias : nullptr;
    p.logits = ws_at<float>(ws, W.partial);
    p.ids_out = r ? r->ids : nullptr;
    p.w_out = r ? r->w : nullptr;
    p.rgate = r ? r->gate : 0;

    const bool staged = L.xs_off != 0;
    const long long max_active = (long long)d.T * d.k < d.E ? (long long)d.T * d.k : d.E;
    // enough CTAs that every consumer has a chunk
    const long long chunks = max_active * ((long long)(d.I / 8) * L.nkc + d.H / kP2Rows);
    long long grid = (chunks + kCons - 1) / kCons;
    if (grid > sm_count()) grid = sm_count();
    if (grid < 1) grid = 1;
    fused_split_constants(d, (int)grid, p);
    // the instantiation with the spread task order, where the gate_up work of the most
    // active experts there can be spans more than two rounds (the kernel decides on the
    // experts actually active)
    const bool spread = max_active * (d.I / 8) * L.nkc > 2LL * kCons * grid;
    const void *fn = r ? (spread ? reinterpret_cast<const void *>(decode_fused_kernel<true, true, true>)
                                 : reinterpret_cast<const void *>(decode_fused_kernel<true, false, true>))
                       : staged ? (spread ? reinterpret_cast<const void *>(decode_fused_kernel<true, true, false>)
                                          : reinterpret_cast<const void *>(decode_fused_kernel<true, false, false>))
                                : reinterpret_cast<const void *>(decode_fused_kernel<false, true, false>);
    err = set_smem_once(fn, kFusedSmem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFW * 32);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    // The CTAs wait on one another, so the launch is cooperative: the runtime
    // either makes every CTA co-resident or fails the launch (the grid is at
    // most one CTA per SM), whatever other work shares the device. It is also
    // programmatic: the CTAs take their SMs and set up while the router ahead
    // finishes. The waits are bounded all the same.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (r && spread) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<true, true, true>, p);
    if (r) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<true, false, true>, p);
    if (staged && spread) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<true, true, false>, p);
    if (staged) return cudaLaunchKernelEx(&cfg, decode_fused_kernel<true, false, false>, p);
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel<false, true, false>, p);
}

}  // namespace moe
