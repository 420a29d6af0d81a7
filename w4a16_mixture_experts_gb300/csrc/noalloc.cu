// moe_w4a16_forward_noalloc: the decode-batch forward with its scratch in a
// fixed device array of this library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand over, or allocate, a device buffer
// at the point where they run the layer. Examples are a host runtime whose
// device memory pool is fully carved up at start-up (weights and caches take
// all of it, and a fresh cudaMalloc would fail or force a pool resize), a
// plugin interface whose operator signature carries no workspace argument, and
// a latency-critical decode loop where cudaMalloc/cudaFree cannot be used
// because they may synchronise the whole device. For them the scratch lives
// in a file-scope __device__ array whose device address is looked up once per
// device; no call here allocates or frees memory, directly or through a
// library.
//
// Limits and rules (also stated in w4a16moe.h):
//  - Only the fused decode path (T <= 8) is served, and only when the
//    workspace layout of the shape fits in kStaticScratchBytes (1 MiB);
//    larger shapes are rejected with MOE_ERR_WORKSPACE before anything is
//    enqueued.
//  - There is one scratch array per device per process: two calls on the same
//    device that may overlap in time (two streams, two host threads) race on
//    it and give wrong results.
//  - The first call on a device does the set-up (the symbol lookup, which
//    may load this module); make that first call outside any stream capture.
//  - The fused kernel needs its completion counters and the control block
//    (error word, exit and barrier counts) at zero when it starts. Each call
//    clears both itself with one small cudaMemsetAsync on its stream, so
//    neither the module-load zero fill nor what an earlier call (of any shape,
//    finished or given up) left behind matters. Nothing else in the array must
//    start at zero.
//  - Errors seen by the kernel (an id outside [0, E), a bounded wait that
//    gave up) are recorded in the array's error word; a bad id still
//    contributes nothing to the output. moe_noalloc_check_device_error reads
//    the word (it synchronises, so it is meant for tests and error paths).
//    Since every call clears the word first, it reports the last call only.
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "w4a16moe.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;
constexpr int kMaxScratchDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void *g_scratch_ptr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device, looked up once.
cudaError_t static_scratch(void **ptr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (err != cudaSuccess) return err;
        if (!p || (reinterpret_cast<uintptr_t>(p) & 255u)) return cudaErrorInvalidDevicePointer;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ptr_ok(const void *p, bool empty) { return empty ? (p == nullptr || aligned16(p)) : (p && aligned16(p)); }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_w4a16_forward_noalloc(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                                         const int32_t *w1_packed, const uint16_t *w1_scales,
                                         const int32_t *w2_packed, const uint16_t *w2_scales, uint16_t *out,
                                         moe_dims d, void *stream) {
    size_t need = 0;
    int rc = moe_workspace_size(d, &need);   // shape checks of every forward call
    if (rc) return rc;
    const bool empty = d.T == 0;
    if (!ptr_ok(hidden, empty) || !ptr_ok(topk_ids, empty) || !ptr_ok(topk_w, empty) || !ptr_ok(out, empty))
        return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(w1_packed, false) || !ptr_ok(w1_scales, false) || !ptr_ok(w2_packed, false) ||
        !ptr_ok(w2_scales, false))
        return MOE_ERR_INVALID_ARG;
    if (!fused_supported(d)) return MOE_ERR_UNSUPPORTED;
    if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
    if (empty) return MOE_OK;

    void *ws = nullptr;
    cudaError_t err = static_scratch(&ws);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the control block, rowss and the counters of experts [0, E), the first
    // regions of the layout
    const WsLayout W = ws_layout(d);
    err = cudaMemsetAsync(ws_at<char>(ws, W.ctrl), 0, W.done1 + (size_t)d.E * kCtrStride * 4 - W.ctrl, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    const ExpertArgs a{hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales};
    err = launch_decode_fused(a, d, ws, out, nullptr, 0.f, s);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_noalloc_check_device_error(void *stream) {
    void *ws = nullptr;
    if (static_scratch(&ws) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t err_word = 0;
    if (cudaMemcpyAsync(&err_word, ws, sizeof(err_word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (!err_word) return MOE_OK;
    if (cudaMemsetAsync(ws, 0, sizeof(err_word), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    return err_word == MOE_ERR_TIMEOUT ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
}
