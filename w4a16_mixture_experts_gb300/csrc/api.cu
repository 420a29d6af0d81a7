// C-ABI entry points of libw4a16moe: argument checks, workspace layout and
// kernel sequencing. No allocation, no synchronisation (except in
// moe_check_device_error, which exists to synchronise).
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "w4a16moe.h"

namespace moe {

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];

struct SmemAttr {
    const void *func;
    int bytes;
    bool done[kMaxDevices];
};
constexpr int kMaxSmemKernels = 16;   // kernels that raise their shared-memory limit (9 today)
SmemAttr g_attrs[kMaxSmemKernels];
int g_nattrs = 0;
std::mutex g_attrs_mu;   // callers may launch from several host threads

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return dev;
}
}  // namespace

int sm_count() {
    const int dev = current_device();
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

cudaError_t set_smem_once(const void *func, int bytes) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_attrs_mu);
    int i = 0;
    for (; i < g_nattrs; ++i)
        if (g_attrs[i].func == func) break;
    if (i == g_nattrs) {
        if (g_nattrs == kMaxSmemKernels)
            return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        g_attrs[i].func = func;
        g_attrs[i].bytes = bytes;
        ++g_nattrs;
    }
    if (g_attrs[i].done[dev]) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) g_attrs[i].done[dev] = true;
    return err;
}

// A plain record outside stream capture; inside a capture, an external event
// node, so that the event can still be timed after each graph replay.
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t s) {
    if (!ev) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess) return err;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                               : cudaEventRecord(ev, s);
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Null is allowed only for empty tensors.
bool ptr_ok(const void *p, bool empty) { return empty ? (p == nullptr || aligned16(p)) : (p && aligned16(p)); }

int check_dims(const moe_dims &d) {
    if (d.T < 0 || d.H <= 0 || d.E <= 0 || d.k <= 0 || d.I <= 0) return MOE_ERR_INVALID_ARG;
    if (d.H % kGroup || d.I % kGroup || d.H > 8192 || d.I > 4096) return MOE_ERR_UNSUPPORTED;
    if (d.k > kMaxK || d.k > d.E || d.E > kMaxE) return MOE_ERR_UNSUPPORTED;
    if (d.T > (1 << 20)) return MOE_ERR_UNSUPPORTED;
    // token rows of the fp32 accumulator are addressed by 32-bit offsets t * H
    if ((int64_t)d.T * d.H >= ((int64_t)1 << 32)) return MOE_ERR_UNSUPPORTED;
    if (!prefill_supported(d)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_ws(const moe_dims &d, const void *ws, size_t ws_bytes) {
    if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < ws_layout(d).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

int forward_impl(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w, const int32_t *w1_packed,
                 const uint16_t *w1_scales, const int32_t *w2_packed, const uint16_t *w2_scales, uint16_t *out,
                 uint16_t *next, float eps, moe_dims d, void *ws, size_t ws_bytes, void *stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    const bool empty = d.T == 0;
    if (!ptr_ok(hidden, empty) || !ptr_ok(topk_ids, empty) || !ptr_ok(topk_w, empty)) return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(w1_packed, false) || !ptr_ok(w1_scales, false) || !ptr_ok(w2_packed, false) ||
        !ptr_ok(w2_scales, false))
        return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(next ? (const void *)next : (const void *)out, empty)) return MOE_ERR_INVALID_ARG;
    if (next && !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(d, ws, ws_bytes))) return rc;
    if (empty) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ExpertArgs a{hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales};
    cudaError_t err;
    if (fused_supported(d)) {
        err = record_profile_event(g_ev_before, s);
        if (err == cudaSuccess) err = launch_decode_fused(a, d, ws, out, next, eps, s);
        if (err == cudaSuccess) err = record_profile_event(g_ev_after, s);
        return cuda_status(err);
    }
    err = launch_permute(topk_ids, d, ws, s);
    if (err == cudaSuccess) err = launch_prefill(a, d, ws, out, next, eps, g_ev_before, g_ev_after, s);
    return cuda_status(err);
}

}  // namespace

extern "C" {

const char *moe_status_str(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size)";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime or launch error";
        case MOE_ERR_DEVICE: return "a kernel saw an expert id outside [0, E)";
        case MOE_ERR_TIMEOUT: return "a kernel's bounded wait gave up";
        default: return "unknown status";
    }
}

int moe_version(void) { return 100; }

int moe_workspace_size(moe_dims d, size_t *bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    const int rc = check_dims(d);
    if (rc) return rc;
    *bytes = ws_layout(d).total;
    return MOE_OK;
}

int moe_route(const uint16_t *hidden, const uint16_t *router_w, const float *bias, moe_dims d, int32_t *topk_ids,
              float *topk_w, void *ws, size_t ws_bytes, void *stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    const bool empty = d.T == 0;
    if (!ptr_ok(hidden, empty) || !ptr_ok(router_w, false) || !ptr_ok(topk_ids, empty) || !ptr_ok(topk_w, empty))
        return MOE_ERR_INVALID_ARG;
    if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(d, ws, ws_bytes))) return rc;
    if (empty) return MOE_OK;
    return cuda_status(launch_route(hidden, router_w, bias, d, topk_ids, topk_w, ws,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_shared(const uint16_t *hidden, const uint16_t *router_w, const float *bias, moe_dims d,
                     int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    // the forward then runs with one more expert and one more slot per token
    if (d.k + 1 > kMaxK || d.E + 1 > kMaxE) return MOE_ERR_UNSUPPORTED;
    const bool empty = d.T == 0;
    if (!ptr_ok(hidden, empty) || !ptr_ok(router_w, false) || !ptr_ok(topk_ids, empty) || !ptr_ok(topk_w, empty))
        return MOE_ERR_INVALID_ARG;
    if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(d, ws, ws_bytes))) return rc;
    if (empty) return MOE_OK;
    return cuda_status(launch_route(hidden, router_w, bias, d, topk_ids, topk_w, ws,
                                    reinterpret_cast<cudaStream_t>(stream), true));
}

int moe_w4a16_forward(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                      const int32_t *w1_packed, const uint16_t *w1_scales, const int32_t *w2_packed,
                      const uint16_t *w2_scales, uint16_t *out, moe_dims d, void *ws, size_t ws_bytes,
                      void *stream) {
    return forward_impl(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales, out, nullptr, 0.f, d,
                        ws, ws_bytes, stream);
}

int moe_w4a16_forward_rms(const uint16_t *hidden, const int32_t *topk_ids, const float *topk_w,
                          const int32_t *w1_packed, const uint16_t *w1_scales, const int32_t *w2_packed,
                          const uint16_t *w2_scales, uint16_t *next, float eps, moe_dims d, void *ws,
                          size_t ws_bytes, void *stream) {
    if (!next && d.T > 0) return MOE_ERR_INVALID_ARG;
    return forward_impl(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales, nullptr, next, eps, d,
                        ws, ws_bytes, stream);
}

int moe_layer_forward(const uint16_t *hidden, const uint16_t *router_w, const float *bias, int32_t shared,
                      const int32_t *w1_packed, const uint16_t *w1_scales, const int32_t *w2_packed,
                      const uint16_t *w2_scales, uint16_t *out, uint16_t *next, float eps, int32_t *topk_ids,
                      float *topk_w, moe_dims d, void *ws, size_t ws_bytes, void *stream) {
    if (shared != 0 && shared != 1) return MOE_ERR_INVALID_ARG;
    int rc = check_dims(d);
    if (rc) return rc;
    if (shared && (d.k + 1 > kMaxK || d.E + 1 > kMaxE)) return MOE_ERR_UNSUPPORTED;
    // the forward's dims: the shared expert is one more expert and one more slot
    const moe_dims df{d.T, d.H, d.E + shared, d.k + shared, d.I};
    if ((rc = check_dims(df))) return rc;
    const bool empty = d.T == 0;
    if (!empty && (out != nullptr) == (next != nullptr)) return MOE_ERR_INVALID_ARG;   // exactly one output
    if (!ptr_ok(hidden, empty) || !ptr_ok(router_w, false) || !ptr_ok(topk_ids, empty) || !ptr_ok(topk_w, empty))
        return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(w1_packed, false) || !ptr_ok(w1_scales, false) || !ptr_ok(w2_packed, false) ||
        !ptr_ok(w2_scales, false))
        return MOE_ERR_INVALID_ARG;
    if (!ptr_ok(next ? (const void *)next : (const void *)out, empty)) return MOE_ERR_INVALID_ARG;
    if (next && !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
    if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
    // one workspace serves the router (dims d) and the forward (dims df)
    if ((rc = check_ws(d, ws, ws_bytes)) || (rc = check_ws(df, ws, ws_bytes))) return rc;
    if (empty) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fused_route_supported(df)) {
        const ExpertArgs a{hidden, nullptr, nullptr, w1_packed, w1_scales, w2_packed, w2_scales};
        const RouteArgs r{router_w, bias, topk_ids, topk_w, shared};
        cudaError_t err = record_profile_event(g_ev_before, s);
        if (err == cudaSuccess) err = launch_decode_fused(a, df, ws, out, next, eps, s, &r);
        if (err == cudaSuccess) err = record_profile_event(g_ev_after, s);
        return cuda_status(err);
    }
    // otherwise the router's kernels, then the forward's
    const cudaError_t err = launch_route(hidden, router_w, bias, d, topk_ids, topk_w, ws, s, shared != 0);
    if (err != cudaSuccess) return cuda_status(err);
    return forward_impl(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales, out, next, eps, df, ws,
                        ws_bytes, stream);
}

int moe_permute(const int32_t *topk_ids, moe_dims d, int32_t *offsets, int32_t *perm, void *ws, size_t ws_bytes,
                void *stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    const bool empty = d.T == 0;
    if (!ptr_ok(topk_ids, empty) || !ptr_ok(offsets, false) || !ptr_ok(perm, empty)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(d, ws, ws_bytes))) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(d);
    cudaError_t err = launch_permute(topk_ids, d, ws, s);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(offsets, ws_at<int32_t>(ws, L.offsets), sizeof(int32_t) * (d.E + 1),
                              cudaMemcpyDeviceToDevice, s);
    if (err == cudaSuccess && d.T > 0)
        err = cudaMemcpyAsync(perm, ws_at<int32_t>(ws, L.perm), sizeof(int32_t) * (size_t)d.T * d.k,
                              cudaMemcpyDeviceToDevice, s);
    return cuda_status(err);
}

int moe_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed, int32_t *bad_count, void *stream) {
    if (N < 0 || K < 0 || K % 8) return MOE_ERR_INVALID_ARG;
    const bool empty = N == 0 || K == 0;
    if (!ptr_ok(q, empty) || !ptr_ok(packed, empty)) return MOE_ERR_INVALID_ARG;
    if (bad_count && (reinterpret_cast<uintptr_t>(bad_count) & 3u)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pack_int4(q, N, K, packed, bad_count, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_forward_plan(moe_dims d, int32_t *plan) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    const int rc = check_dims(d);
    if (rc) return rc;
    *plan = fused_plan(d);
    return MOE_OK;
}

int moe_quantize_int4(const uint16_t *w, int64_t N, int64_t K, int32_t nclip, int32_t *packed, uint16_t *scales,
                      int32_t *choice, void *stream) {
    if (N < 0 || K < 0 || K % kGroup || nclip < 1 || nclip > 100) return MOE_ERR_INVALID_ARG;
    const bool empty = N == 0 || K == 0;
    if (!ptr_ok(w, empty) || !ptr_ok(packed, empty) || !ptr_ok(scales, empty)) return MOE_ERR_INVALID_ARG;
    if (choice && !ptr_ok(choice, empty)) return MOE_ERR_INVALID_ARG;
    return cuda_status(
        launch_quantize_int4(w, N, K, nclip, packed, scales, choice, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_w8a16_linear(const uint16_t *x, const int32_t *w_packed, const uint16_t *scales, int32_t gs, uint16_t *y,
                     int32_t T, int32_t N, int32_t K, void *ws, size_t ws_bytes, void *stream) {
    if (T < 0 || N < 0 || K <= 0 || (gs != 64 && gs != 128) || K % gs) return MOE_ERR_INVALID_ARG;
    if (T > (1 << 20) || K > 65536) return MOE_ERR_UNSUPPORTED;
    const bool empty = T == 0 || N == 0;
    if (!ptr_ok(x, T == 0) || !ptr_ok(w_packed, N == 0) || !ptr_ok(scales, N == 0) || !ptr_ok(y, empty))
        return MOE_ERR_INVALID_ARG;
    if (empty) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T <= 8) {
        if (!w8a16_gemv_supported(T, K)) return MOE_ERR_UNSUPPORTED;
        return cuda_status(launch_w8a16(x, w_packed, scales, gs, y, T, N, K, s));
    }
    // the tensor-core GEMM records a wait that gave up in the workspace's error word, and
    // keeps the partial results of a split over K after it
    if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
    size_t need = 0;
    moe_w8a16_workspace_size(T, N, K, gs, &need);
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_w8a16_gemm(x, w_packed, scales, gs, y, T, N, K, reinterpret_cast<Ctrl *>(ws),
                                         ws_at<float>(ws, sizeof(Ctrl)), s));
}

int moe_w8a16_workspace_size(int32_t T, int32_t N, int32_t K, int32_t gs, size_t *bytes) {
    if (!bytes || T < 0 || N < 0 || K <= 0 || (gs != 64 && gs != 128) || K % gs) return MOE_ERR_INVALID_ARG;
    size_t n = sizeof(Ctrl);
    if (T > 8 && N > 0) {
        const int S = w8a16_gemm_splits(T, N, K);
        if (S > 1) n += (size_t)S * T * N * 4;
    }
    *bytes = n;
    return MOE_OK;
}

int moe_profile_events(void *before_experts, void *after_experts) {
    if ((before_experts == nullptr) != (after_experts == nullptr)) return MOE_ERR_INVALID_ARG;
    g_ev_before = reinterpret_cast<cudaEvent_t>(before_experts);
    g_ev_after = reinterpret_cast<cudaEvent_t>(after_experts);
    return MOE_OK;
}

int moe_check_device_error(void *ws, size_t ws_bytes, void *stream) {
    if (!ws || !aligned16(ws) || ws_bytes < sizeof(Ctrl)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t err_word = 0;
    if (cudaMemcpyAsync(&err_word, ws, sizeof(err_word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (err_word) {
        // A wait that gave up may leave completion counters anywhere in the
        // workspace non-zero; the whole workspace is cleared so that the next
        // call starts from the all-zero state. A bad id leaves the counters
        // consistent: only the error word is cleared.
        const size_t clear = err_word == MOE_ERR_TIMEOUT ? ws_bytes : sizeof(err_word);
        if (cudaMemsetAsync(ws, 0, clear, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
        return err_word == MOE_ERR_TIMEOUT ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
    }
    return MOE_OK;
}

}  // extern "C"
