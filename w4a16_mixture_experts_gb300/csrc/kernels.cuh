// Host-side launchers of the libw4a16moe kernels (all enqueue on `s`).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "w4a16moe.h"

namespace moe {

// Raises a kernel's dynamic shared memory limit once per device.
cudaError_t set_smem_once(const void *func, int bytes);

// 2-D tiled TMA descriptor over a row-major [rows][inner] tensor.
cudaError_t encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base,
                           uint64_t inner, uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                           uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Number of SMs of the current device (cached per device).
int sm_count();

// Records a caller's profiling event on `s` (nothing for a null event).
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t s);

// gate: the router has E + 1 rows, the last being a shared expert's gate; ids
// and w are then [T][k + 1] with slot k = (E, sigmoid(gate logit)).
cudaError_t launch_route(const uint16_t *x, const uint16_t *wr, const float *bias, const moe_dims &d,
                         int32_t *ids, float *w, void *ws, cudaStream_t s, bool gate = false);

// Router logits on the tensor core for T > 64 and E a multiple of 128:
// partial [ksplit][T][E] f32 (summed by the top-k kernel).
cudaError_t launch_route_logits_tc(const uint16_t *x, const uint16_t *wr, const moe_dims &d, float *partial,
                                   int ksplit, struct Ctrl *ctrl, cudaStream_t s);

cudaError_t launch_permute(const int32_t *ids, const moe_dims &d, void *ws, cudaStream_t s);

struct ExpertArgs {
    const uint16_t *x;
    const int32_t *ids;
    const float *topk_w;
    const int32_t *w1p;
    const uint16_t *w1s;
    const int32_t *w2p;
    const uint16_t *w2s;
};

// Prefill expert path (tcgen05 grouped GEMMs; needs launch_permute first):
// x reordering, gate_up, down, and the conversion of the fp32 accumulator.
// The two events (may be null) bracket the gate_up and down kernels.
bool prefill_supported(const moe_dims &d);
cudaError_t launch_prefill(const ExpertArgs &a, const moe_dims &d, void *ws, uint16_t *out, uint16_t *next, float eps,
                           cudaEvent_t ev_before, cudaEvent_t ev_after, cudaStream_t s);

// Fused decode forward (T <= 8): permute, experts and combine in one launch.
bool fused_supported(const moe_dims &d);
// 0 if the forward takes the tensor-core pipeline; else 1 (activations staged
// in shared memory) or 2 (read from global memory), plus 16 * quantisation
// groups per gate_up chunk, plus 256 if the down outputs' block buffers have a
// region of their own, plus 512 if the kernel can also run the router.
int fused_plan(const moe_dims &d);
// The router run by the fused decode kernel itself (moe_layer_forward): the
// router weights [E + gate][H] and bias, and the selection's outputs.
struct RouteArgs {
    const uint16_t *wr;
    const float *bias;
    int32_t *ids;
    float *w;
    int gate;
};
// True when the fused decode kernel can also run the router for the forward
// dims d (experts E + gate, slots k + gate): the activations are staged and its
// ring holds the router's scratch.
bool fused_route_supported(const moe_dims &d);
// With r, the kernel routes itself (d: the forward's dims) and a.ids / a.topk_w
// are not read.
cudaError_t launch_decode_fused(const ExpertArgs &a, const moe_dims &d, void *ws, uint16_t *out, uint16_t *next,
                                float eps, cudaStream_t s, const RouteArgs *r = nullptr);

// RTN INT4 g128 quantiser with the per-group clip search (quant.cu).
cudaError_t launch_quantize_int4(const uint16_t *w, int64_t N, int64_t K, int nclip, int32_t *packed,
                                 uint16_t *scales, int32_t *choice, cudaStream_t s);

// W8A16 linear layer (w8a16.cu): the GEMV for T <= 8.
bool w8a16_gemv_supported(int T, int K);
cudaError_t launch_w8a16(const uint16_t *x, const int32_t *w, const uint16_t *s, int gs, uint16_t *y, int T, int N,
                         int K, cudaStream_t st);
// ... and the tensor-core GEMM for larger T (prefill.cu, the INT8 instantiation).
// K is split over CTAs when the layer has fewer tiles than SMs; the splits' f32
// results go to part [splits][T][N] (the workspace after the control block).
int w8a16_gemm_splits(int T, int N, int K);
cudaError_t launch_w8a16_gemm(const uint16_t *x, const int32_t *w, const uint16_t *s, int gs, uint16_t *y, int T, int N,
                              int K, struct Ctrl *ctrl, float *part, cudaStream_t st);

cudaError_t launch_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed, int32_t *bad,
                             cudaStream_t s);

}  // namespace moe
