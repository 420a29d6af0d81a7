/*
 * w4a16moe.h - C ABI of the GB300 (sm_103a) W4A16 routed-expert MoE layer.
 *
 * The layer is the routed-expert block of the 125B-A6B MoE described in
 * "Running 125B MoE on Three 3090s - vLLM Optimization Edition", section 3.3
 * "MoE block (decode-05)": a BF16 router GEMV, softmax and top-k with
 * renormalised weights (norm_topk_prob), the token-to-expert alignment, and
 * the fused W4A16 expert GEMMs (gate_up, SiluAndMul, down) followed by the
 * weighted sum over the selected experts. Shapes are those of "Running 125B
 * MoE on Three 3090s - vLLM Edition", section 1 "Shape of This Model"
 * (hidden 2560, 512 experts, 10 per token, moe_intermediate 640); the weight
 * format is group A of the model card's "What is quantized" table (INT4,
 * group size 128, symmetric, compressed-tensors pack-quantized).
 *
 * Conventions for every call:
 *  - All pointers except `dims`/`bytes` outputs are DEVICE pointers of the
 *    current CUDA device, owned by the caller; the library never allocates,
 *    frees or synchronises inside moe_route / moe_w4a16_forward /
 *    moe_w4a16_forward_rms / moe_permute / moe_pack_int4.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *    enqueued asynchronously; results are valid once the stream reaches them.
 *  - bf16 tensors are passed as `uint16_t*` holding IEEE bfloat16 bits.
 *  - Every tensor is row-major and contiguous; every pointer is 16-byte
 *    aligned.
 *  - Supported shapes: T >= 0, H and I multiples of 128, 1 <= k <= 32,
 *    k <= E <= 1024, H <= 8064, I <= 4096, T <= 2^20 and T * H < 2^32.
 *    Others return MOE_ERR_UNSUPPORTED before anything is enqueued.
 *  - Argument errors are returned synchronously and enqueue nothing. A
 *    launch failure returns MOE_ERR_CUDA. Errors seen by a kernel (an expert
 *    id outside [0, E), an internal wait that gave up) are recorded in the
 *    workspace's error word and reported by moe_check_device_error.
 *  - Workspace: `ws` must hold at least moe_workspace_size() bytes and must
 *    be all zero before its first use (the library leaves the counters it
 *    uses at zero when a call completes, at offsets that depend on no
 *    dimension, so calls of different dims may share a workspace large
 *    enough for each). One workspace must not be used by two calls that may
 *    run concurrently. A call whose bounded wait gave up
 *    (MOE_ERR_TIMEOUT) can leave counters non-zero: moe_check_device_error
 *    then clears the whole workspace before it returns, and a caller that
 *    does not call it must clear the workspace itself before reusing it.
 */
#ifndef W4A16MOE_H
#define W4A16MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size */
    MOE_ERR_UNSUPPORTED = 2,  /* shape outside the supported set */
    MOE_ERR_WORKSPACE = 3,    /* workspace too small */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE = 5,       /* a kernel saw an expert id outside [0, E) */
    MOE_ERR_TIMEOUT = 6       /* a kernel's bounded wait gave up */
} moe_status;

/* Layer dimensions: T tokens, hidden H, E experts, k experts per token,
 * expert intermediate I. The quantisation group is fixed at 128. */
typedef struct {
    int32_t T, H, E, k, I;
} moe_dims;

/* Static description of a status code. Never NULL. */
MOE_API const char *moe_status_str(int status);

/* Library version as major*10000 + minor*100 + patch. */
MOE_API int moe_version(void);

/* Workspace bytes needed by moe_route, moe_permute and the forward calls
 * for dims `d`. Writes *bytes; returns MOE_OK or MOE_ERR_UNSUPPORTED /
 * MOE_ERR_INVALID_ARG. */
MOE_API int moe_workspace_size(moe_dims d, size_t *bytes);

/*
 * Router + softmax + top-k + renormalisation ("vLLM Optimization Edition",
 * section 3.3 "MoE block": router GEMV, topk_softmax, norm_topk_prob, and
 * the key that sends ties to the lower expert id).
 *
 *   logits[t][e] = sum_h hidden[t][h] * router_w[e][h] (+ bias[e])
 *   topk_ids[t][0..k) = the k largest logits, in order of descending logit,
 *                       ties to the lower id; ranked in fp32
 *   topk_w[t][j]      = softmax over the k selected logits, which equals the
 *                       renormalised full softmax
 *
 * hidden   bf16 [T][H]     router_w bf16 [E][H]
 * bias     f32 [E] or NULL (added to the logits for selection and weights)
 * topk_ids int32 [T][k]    topk_w   f32 [T][k]   (outputs)
 */
MOE_API int moe_route(const uint16_t *hidden, const uint16_t *router_w, const float *bias,
              moe_dims d, int32_t *topk_ids, float *topk_w,
              void *ws, size_t ws_bytes, void *stream);

/*
 * moe_route for a layer with a shared expert ("vLLM Optimization Edition",
 * section 3.3 "MoE block (decode-05)": the router and the shared expert's gate
 * are one GEMV of 512 + 1 rows, and the layer's output is routed +
 * sigmoid(gate) x shared).
 *
 * router_w bf16 [E+1][H]: rows [0, E) route, row E is the shared expert's gate.
 * d: the routed dims (E routed experts, k of them per token); k + 1 <= 32 and
 * E + 1 <= 1024. bias f32 [E] or NULL applies to the routed logits only.
 * topk_ids int32 [T][k+1], topk_w f32 [T][k+1] (outputs): slots [0, k) as
 * moe_route; slot k = expert E with weight sigmoid(x . router_w[E]) (fp32).
 * The workspace is sized by moe_workspace_size(d).
 *
 * The shared expert is then expert E of the weight tensors (stored as a
 * routed expert, INT4 g128, intermediate I): moe_w4a16_forward with dims
 * (T, H, E+1, k+1, I) and these ids and weights computes
 *   out = sum_j topk_w[j] * expert_j(x) + sigmoid(gate) * shared(x)
 * in one pass, with one rounding to bf16. Its workspace is sized by
 * moe_workspace_size(T, H, E+1, k+1, I).
 */
MOE_API int moe_route_shared(const uint16_t *hidden, const uint16_t *router_w, const float *bias,
                     moe_dims d, int32_t *topk_ids, float *topk_w,
                     void *ws, size_t ws_bytes, void *stream);

/*
 * Routed-expert forward ("vLLM Optimization Edition", section 3.3: the fused
 * Marlin MoE gate_up, SiluAndMul, down, and moe_sum; weights as in the model
 * card's group A):
 *
 *   W1[e][n][c] = (nibble c%8 of w1_packed[e][n][c/8] - 8) * w1_scales[e][n][c/128]
 *   W2[e][n][c] likewise from w2_packed / w2_scales
 *   for each token t and slot j, e = topk_ids[t][j]:
 *     g = W1[e][0:I] . x_t,  u = W1[e][I:2I] . x_t,  h = SiLU(g) * u
 *     out[t] += topk_w[t][j] * (W2[e] . h)
 *   out is rounded to bf16 once.
 *
 * hidden    bf16 [T][H]         topk_ids int32 [T][k] in [0, E)
 * topk_w    f32 [T][k]          (taken as given; need not sum to 1)
 * w1_packed int32 [E][2I][H/8]  (rows [0,I) gate, [I,2I) up; low nibble first)
 * w1_scales bf16 [E][2I][H/128]
 * w2_packed int32 [E][H][I/8]   w2_scales bf16 [E][H][I/128]
 * out       bf16 [T][H]         (output; must not overlap any input)
 *
 * Accumulation is fp32; the SiLU(g)*u activation is rounded to bf16 where it
 * feeds the down projection. An id outside [0, E) sets MOE_ERR_DEVICE in the
 * workspace and that slot contributes nothing.
 */
MOE_API int moe_w4a16_forward(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                      const int32_t *w1_packed, const uint16_t *w1_scales,
                      const int32_t *w2_packed, const uint16_t *w2_scales,
                      uint16_t *out, moe_dims d, void *ws, size_t ws_bytes, void *stream);

/*
 * Forward followed by the residual and RMS rescale used between the layers
 * of a stack (no learned weight):
 *   r = hidden + moe(hidden) (fp32),  next[t] = bf16(r / sqrt(mean(r^2) + eps))
 * Same arguments as moe_w4a16_forward; `next` bf16 [T][H] may not overlap
 * `hidden`.
 */
MOE_API int moe_w4a16_forward_rms(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                          const int32_t *w1_packed, const uint16_t *w1_scales,
                          const int32_t *w2_packed, const uint16_t *w2_scales,
                          uint16_t *next, float eps, moe_dims d, void *ws, size_t ws_bytes,
                          void *stream);

/*
 * The whole MoE block in one call ("vLLM Optimization Edition", section 3.3
 * "MoE block (decode-05)": the router GEMV, topk_softmax, the fused experts and
 * moe_sum; with `shared`, the shared expert's gate as one more router row):
 *
 *   moe_route (shared = 0) or moe_route_shared (shared = 1) with dims d,
 *   then moe_w4a16_forward (out not NULL) or moe_w4a16_forward_rms (next not
 *   NULL) with dims (T, H, E + shared, k + shared, I).
 *
 * Arguments are those of the calls above: router_w bf16 [E + shared][H], bias
 * f32 [E] or NULL, the weights of E + shared experts, topk_ids int32 and
 * topk_w f32 [T][k + shared] (outputs: the selection, as the router calls
 * write it), and exactly one of out / next (the other NULL; eps is read only
 * with next). The workspace must hold max(moe_workspace_size(d),
 * moe_workspace_size(T, H, E + shared, k + shared, I)) bytes; the rules on
 * zeroing are those of every call.
 *
 * Where moe_forward_plan reports bit 512 for the forward's dims (decode
 * batches, T <= 8, whose activations the expert kernel stages in shared
 * memory), one cooperative kernel runs the block: each CTA computes a few
 * router rows with the small-batch router's own arithmetic, the CTAs meet at a
 * grid-wide barrier, every CTA selects the top-k from all logits, and the
 * experts follow in the same launch. Selection, weights and outputs are then
 * bit-identical to the separate calls. Otherwise the router's kernels run,
 * then the forward's.
 */
MOE_API int moe_layer_forward(const uint16_t *hidden, const uint16_t *router_w, const float *bias, int32_t shared,
                      const int32_t *w1_packed, const uint16_t *w1_scales,
                      const int32_t *w2_packed, const uint16_t *w2_scales,
                      uint16_t *out, uint16_t *next, float eps, int32_t *topk_ids, float *topk_w,
                      moe_dims d, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_w4a16_forward for decode batches without a caller workspace. The pages
 * have no counterpart: this entry point exists for callers that cannot
 * provide or allocate a device scratch buffer where they run the layer (a
 * fully carved memory pool, a plugin signature without a workspace argument,
 * a loop where cudaMalloc's device-wide synchronisation is not acceptable).
 *
 * Same computation and arguments as moe_w4a16_forward minus ws/ws_bytes. The
 * scratch is a 1 MiB array that the library holds in device memory, one per
 * device per process; the call allocates and frees nothing.
 *  - Served shapes: those of the fused decode path (T <= 8) whose
 *    moe_workspace_size() is at most 1 MiB (T = 7 at H 2560, E 512, k 10,
 *    I 640 needs about 0.51 MiB). A larger workspace size returns
 *    MOE_ERR_WORKSPACE and T > 8 returns MOE_ERR_UNSUPPORTED, in both cases
 *    before anything is enqueued. T = 0 returns MOE_OK.
 *  - The first call on a device looks up the array's device address (which
 *    may load the module that holds it); make that call before any stream
 *    capture begins.
 *  - Each call first clears the kernel's completion counters in the array
 *    (one cudaMemsetAsync on `stream`), so nothing needs to be zero
 *    beforehand and an earlier call of another shape does not matter.
 *  - Calls on the same device that may overlap in time (other streams, other
 *    host threads) race on the array and give wrong results.
 *  - Ids outside [0, E) contribute nothing; the error word the kernel sets
 *    stays inside the array, where moe_noalloc_check_device_error reads it.
 */
MOE_API int moe_w4a16_forward_noalloc(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                              const int32_t *w1_packed, const uint16_t *w1_scales,
                              const int32_t *w2_packed, const uint16_t *w2_scales,
                              uint16_t *out, moe_dims d, void *stream);

/*
 * Token-to-expert permutation ("vLLM Optimization Edition", section 3.3:
 * moe_align_block_size, here without block padding): per-expert counts,
 * their exclusive prefix sum, and the assignments a = t*k + j listed expert
 * by expert, in increasing a within an expert. Exposed for testing; the
 * forward calls run the same kernels.
 *
 * topk_ids int32 [T][k]; offsets int32 [E+1] (output); perm int32 [T*k]
 * (output). An id outside [0, E) sets MOE_ERR_DEVICE; such assignments are
 * left out, so offsets[E] counts only valid ones.
 */
MOE_API int moe_permute(const int32_t *topk_ids, moe_dims d, int32_t *offsets, int32_t *perm,
                void *ws, size_t ws_bytes, void *stream);

/*
 * Pack signed int4 values into the storage format of the weights (model
 * card "What is quantized", pack-quantized): packed[n][w] holds
 * q[n][8w..8w+7] + 8, value 8w+i in bits [4i, 4i+4).
 * q int8 [N][K] with values in [-8, 7] (others are clamped and flagged in
 * *bad_count, a device int32 that is incremented, may be NULL);
 * packed int32 [N][K/8]. K must be a multiple of 8.
 */
MOE_API int moe_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed,
                  int32_t *bad_count, void *stream);

/*
 * W8A16 linear layer ("vLLM Optimization Edition", section 3.3
 * "Hyper-connection (decode-04)": INT8 GEMVs on the pack-quantized words as
 * stored, and a W8A16 GEMM for batches; model card "What is quantized",
 * groups C (INT8 gs64: hyper-connection mixers) and D (INT8 gs128: lm_head)):
 *   W[n][c] = (byte c%4 of w_packed[n][c/4] - 128) * scales[n][c/gs]
 *   y[t][n] = sum_c x[t][c] * W[n][c]   (fp32 accumulation, rounded to bf16 once)
 * x bf16 [T][K]; w_packed int32 [N][K/4] (four values per word, least
 * significant byte first, stored q + 128); scales bf16 [N][K/gs]; y bf16
 * [T][N] (output). gs is 64 or 128 and divides K (K a multiple of 64, at most
 * 65536); T <= 2^20.
 *  - 1 <= T <= 8: the decode GEMV (weights streamed from HBM, mma.sync), when
 *    T * (K + 8) * 2 <= 196608 (else MOE_ERR_UNSUPPORTED). ws may be NULL.
 *  - T > 8: the tcgen05 GEMM (tiles of 128 rows x 128 tokens; a layer with
 *    fewer tiles than SMs is split over K, and the splits are summed in a
 *    fixed order). ws: at least moe_w8a16_workspace_size() bytes, 16-byte
 *    aligned, its first 256 bytes zero before its first use: they hold the
 *    error word that moe_check_device_error reads (a bounded wait that gave
 *    up); the rest holds the splits' f32 results.
 * T = 0 or N = 0 return MOE_OK with nothing enqueued.
 */
MOE_API int moe_w8a16_linear(const uint16_t *x, const int32_t *w_packed, const uint16_t *scales, int32_t gs,
                     uint16_t *y, int32_t T, int32_t N, int32_t K, void *ws, size_t ws_bytes, void *stream);

/* Workspace bytes moe_w8a16_linear needs for these dims (256 for the GEMV and
 * for GEMMs that are not split). Returns MOE_ERR_INVALID_ARG for bad dims. */
MOE_API int moe_w8a16_workspace_size(int32_t T, int32_t N, int32_t K, int32_t gs, size_t *bytes);

/*
 * INT4 quantiser of BF16 weights into the experts' storage ("vLLM
 * Optimization Edition", section 7 "Putting MTP on the GPU", make_mtp_int4.py:
 * round to nearest, group size 128, symmetric, per-group search for the clip
 * that minimises the squared error). For each 128 consecutive values w of a
 * row, with amax = max |w| and clip c_j = (100 - j) / 100, j in [0, nclip):
 *   s_j = bf16(c_j * amax / 7)  (fp32 multiply and divide, bf16 round to nearest even)
 *   q_i = clamp(rint(w_i / s_j), -8, 7)  (fp32 divide; q = 0 when s_j = 0)
 * and the group keeps the j with the smallest sum_i (w_i - q_i s_j)^2 (the
 * lowest j on a tie; the sums are formed in fp32, in units of max|w|^2 so that
 * they neither underflow nor overflow). nclip = 1 is plain round to nearest.
 *
 * w bf16 [N][K], finite; K a multiple of 128; 1 <= nclip <= 100.
 * packed int32 [N][K/8] (outputs; q + 8, lowest nibble first), scales bf16
 * [N][K/128], choice int32 [N][K/128] (the chosen j; may be NULL).
 */
MOE_API int moe_quantize_int4(const uint16_t *w, int64_t N, int64_t K, int32_t nclip, int32_t *packed,
                      uint16_t *scales, int32_t *choice, void *stream);

/*
 * Which kernels a forward call of dims `d` runs (a host-only query, no
 * counterpart on the pages; for tests and tuning). Writes *plan = 0 for the
 * tensor-core pipeline (permute, grouped gate_up and down GEMMs, conversion);
 * otherwise the fused decode kernel runs and *plan = s + 16 * g + 256 * y + 512 * r,
 * where s = 1 if the activations are staged in shared memory and 2 if they
 * are read from global memory, g (at most 15) is the number of 128-wide
 * groups per gate_up chunk, and y = 1 if the down outputs' block buffers have
 * a shared-memory region of their own (0: they reuse the gate_up partial-sum
 * area once the CTA's gate_up work is done), and r = 1 if moe_layer_forward
 * runs the router inside the same kernel for these (forward) dims.
 * Returns the shape checks' status.
 */
MOE_API int moe_forward_plan(moe_dims d, int32_t *plan);

/*
 * Profiling aid (no counterpart on the pages): from now on, every forward
 * call records `before_experts` on its stream just before it launches the
 * expert kernel and `after_experts` just after it, so that the caller can
 * time that kernel alone with cudaEventElapsedTime. Both are cudaEvent_t
 * handles owned by the caller (created with timing enabled); while the stream
 * is being captured into a CUDA graph they become event-record nodes. Pass
 * NULL, NULL to stop. The setting is process-wide and not thread-safe.
 */
MOE_API int moe_profile_events(void *before_experts, void *after_experts);

/*
 * Synchronises `stream`, then reads and clears the workspace's error word.
 * Returns MOE_OK, MOE_ERR_DEVICE or MOE_ERR_TIMEOUT (or MOE_ERR_CUDA if the
 * synchronisation itself failed). On MOE_ERR_TIMEOUT it also sets all
 * ws_bytes of the workspace to zero (and waits for that), so that the
 * workspace is fit for the next call.
 */
MOE_API int moe_check_device_error(void *ws, size_t ws_bytes, void *stream);

/*
 * The same check for moe_w4a16_forward_noalloc (no counterpart on the pages):
 * synchronises `stream`, then reads and clears the error word of the
 * library's static scratch on the current device. Every no-alloc call clears
 * the word before it starts, so this reports on the last call only.
 */
MOE_API int moe_noalloc_check_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16MOE_H */
