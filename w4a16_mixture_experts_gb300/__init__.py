"""Python binding of libw4a16moe, the GB300 (sm_103a) W4A16 routed-expert MoE layer.

Argument marshalling only: each function here takes torch CUDA tensors (device
memory and streams come from PyTorch), derives the layer dims from their
shapes, and calls the C entry point of the same name in ``libw4a16moe.so``.
Every step of the layer runs in the library's CUDA kernels; there is no
fallback, and importing this module fails loudly if the library is missing.

Weights follow the storage of the model card "Minachist/Qwen3.8-Flash-Next-
INT4-Mixed-AutoRound" ("What is quantized", group A): int32 words holding
eight int4 values q + 8, lowest nibble first, with one bf16 scale per row and
128-wide K group. Shapes (E experts, hidden H, intermediate I):
w1_packed [E, 2I, H/8] int32 (gate rows then up rows), w1_scales [E, 2I, H/128]
bf16, w2_packed [E, H, I/8] int32, w2_scales [E, H, I/128] bf16.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MoeError", "moe_dims", "lib", "build", "moe_status_str", "moe_version", "moe_workspace_size",
    "workspace", "moe_route", "moe_route_shared", "shared_workspace", "moe_w4a16_forward", "moe_w4a16_forward_rms", "moe_permute",
    "moe_pack_int4", "moe_quantize_int4", "moe_w8a16_linear", "moe_w8a16_workspace_size", "moe_check_device_error", "moe_profile_events", "moe_w4a16_forward_noalloc",
    "moe_noalloc_check_device_error", "moe_forward_plan", "STATUS",
]

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_DIR, "libw4a16moe.so")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE", 6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status), moe_status_str(status)))


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32)]

    def __repr__(self):
        return "moe_dims(T=%d, H=%d, E=%d, k=%d, I=%d)" % (self.T, self.H, self.E, self.k, self.I)


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libw4a16moe.so in-tree for sm_103a (nvcc)."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libw4a16moe.so is not built (%s); run w4a16_mixture_experts_gb300.build()"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        D = moe_dims
        L.moe_status_str.argtypes, L.moe_status_str.restype = [I], ctypes.c_char_p
        L.moe_version.argtypes, L.moe_version.restype = [], I
        L.moe_workspace_size.argtypes, L.moe_workspace_size.restype = [D, ctypes.POINTER(Z)], I
        L.moe_route.argtypes, L.moe_route.restype = [P, P, P, D, P, P, P, Z, P], I
        L.moe_route_shared.argtypes, L.moe_route_shared.restype = [P, P, P, D, P, P, P, Z, P], I
        L.moe_w4a16_forward.argtypes = [P, P, P, P, P, P, P, P, D, P, Z, P]
        L.moe_w4a16_forward.restype = I
        L.moe_w4a16_forward_rms.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, D, P, Z, P]
        L.moe_w4a16_forward_rms.restype = I
        L.moe_layer_forward.argtypes = [P, P, P, ctypes.c_int32, P, P, P, P, P, P, ctypes.c_float, P, P, D, P, Z, P]
        L.moe_layer_forward.restype = I
        L.moe_w4a16_forward_noalloc.argtypes = [P, P, P, P, P, P, P, P, D, P]
        L.moe_w4a16_forward_noalloc.restype = I
        L.moe_permute.argtypes, L.moe_permute.restype = [P, D, P, P, P, Z, P], I
        L.moe_pack_int4.argtypes, L.moe_pack_int4.restype = [P, I64, I64, P, P, P], I
        L.moe_quantize_int4.argtypes = [P, I64, I64, ctypes.c_int32, P, P, P, P]
        L.moe_quantize_int4.restype = I
        L.moe_w8a16_linear.argtypes = [P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, Z,
                                       P]
        L.moe_w8a16_linear.restype = I
        L.moe_w8a16_workspace_size.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(Z)]
        L.moe_w8a16_workspace_size.restype = I
        L.moe_check_device_error.argtypes, L.moe_check_device_error.restype = [P, Z, P], I
        L.moe_noalloc_check_device_error.argtypes, L.moe_noalloc_check_device_error.restype = [P], I
        L.moe_profile_events.argtypes, L.moe_profile_events.restype = [P, P], I
        L.moe_forward_plan.argtypes, L.moe_forward_plan.restype = [D, ctypes.POINTER(ctypes.c_int32)], I
        _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _check(rc: int, where: str):
    if rc != 0:
        raise MoeError(rc, where)


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype or t.dim() != ndim:
        raise ValueError("%s must be %s with %d dims, got %s %s" % (name, dtype, ndim, t.dtype, tuple(t.shape)))
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)


def moe_status_str(status: int) -> str:
    return lib().moe_status_str(int(status)).decode()


def moe_version() -> int:
    return lib().moe_version()


def moe_workspace_size(T: int, H: int, E: int, k: int, I: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(moe_dims(T, H, E, k, I), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def workspace(T: int, H: int, E: int, k: int, I: int, device=None) -> torch.Tensor:
    """A zeroed uint8 workspace of moe_workspace_size bytes (owned by torch)."""
    return torch.zeros(moe_workspace_size(T, H, E, k, I), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _ws(ws, dims: moe_dims, device):
    if ws is None:
        ws = workspace(dims.T, dims.H, dims.E, dims.k, dims.I, device)
    return ws


def moe_route(hidden, router_w, k: int, bias=None, ws=None, topk_ids=None, topk_w=None, stream=None):
    """Router GEMM, softmax, top-k (ties to the lower id) and renormalised weights.

    Returns (topk_ids int32 [T, k], topk_w f32 [T, k]).
    """
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(router_w, "router_w", torch.bfloat16, 2)
    T, H = hidden.shape
    E = router_w.shape[0]
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
    dims = moe_dims(T, H, E, k, 128)
    ws = _ws(ws, dims, hidden.device)
    if topk_ids is None:
        topk_ids = torch.empty(T, k, dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty(T, k, dtype=torch.float32, device=hidden.device)
    _check(lib().moe_route(_p(hidden), _p(router_w), _p(bias), dims, _p(topk_ids), _p(topk_w), _p(ws),
                           ws.numel(), _stream(stream)), "moe_route")
    return topk_ids, topk_w


def shared_workspace(T: int, H: int, E: int, k: int, I: int, device=None) -> torch.Tensor:
    """A zeroed workspace that serves moe_route_shared (routed dims E, k) and the
    forward of the layer with its shared expert (E + 1 experts, k + 1 slots)."""
    n = max(moe_workspace_size(T, H, E, k, I), moe_workspace_size(T, H, E + 1, k + 1, I))
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def moe_route_shared(hidden, router_w, k: int, bias=None, ws=None, topk_ids=None, topk_w=None, stream=None):
    """Routing of a layer with a shared expert: router_w [E+1, H], row E the shared gate.

    Returns (topk_ids int32 [T, k+1], topk_w f32 [T, k+1]); slot k is expert E with
    weight sigmoid(gate). Pass them to moe_w4a16_forward with the E+1 experts' weights.
    """
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(router_w, "router_w", torch.bfloat16, 2)
    T, H = hidden.shape
    E = router_w.shape[0] - 1
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
    dims = moe_dims(T, H, E, k, 128)
    if ws is None:
        ws = shared_workspace(T, H, E, k, 128, hidden.device)
    if topk_ids is None:
        topk_ids = torch.empty(T, k + 1, dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty(T, k + 1, dtype=torch.float32, device=hidden.device)
    _check(lib().moe_route_shared(_p(hidden), _p(router_w), _p(bias), dims, _p(topk_ids), _p(topk_w), _p(ws),
                                  ws.numel(), _stream(stream)), "moe_route_shared")
    return topk_ids, topk_w


def _expert_dims(hidden, topk_ids, w1_packed, w2_packed):
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(topk_ids, "topk_ids", torch.int32, 2)
    _need(w1_packed, "w1_packed", torch.int32, 3)
    _need(w2_packed, "w2_packed", torch.int32, 3)
    T, H = hidden.shape
    E, two_i, _ = w1_packed.shape
    return moe_dims(T, H, E, topk_ids.shape[1], two_i // 2)


def moe_w4a16_forward(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales,
                      out=None, ws=None, stream=None):
    """Routed-expert forward: bf16 out [T, H] = sum_j w_j * W2 (SiLU(W1g x) * W1u x)."""
    dims = _expert_dims(hidden, topk_ids, w1_packed, w2_packed)
    _need(topk_w, "topk_w", torch.float32, 2)
    _need(w1_scales, "w1_scales", torch.bfloat16, 3)
    _need(w2_scales, "w2_scales", torch.bfloat16, 3)
    ws = _ws(ws, dims, hidden.device)
    if out is None:
        out = torch.empty_like(hidden)
    _check(lib().moe_w4a16_forward(_p(hidden), _p(topk_ids), _p(topk_w), _p(w1_packed), _p(w1_scales),
                                   _p(w2_packed), _p(w2_scales), _p(out), dims, _p(ws), ws.numel(),
                                   _stream(stream)), "moe_w4a16_forward")
    return out


def moe_w4a16_forward_noalloc(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales,
                              out=None, stream=None):
    """moe_w4a16_forward for decode batches (T <= 8) with the library's own static scratch.

    No workspace is passed or allocated; calls on one device must not overlap.
    """
    dims = _expert_dims(hidden, topk_ids, w1_packed, w2_packed)
    _need(topk_w, "topk_w", torch.float32, 2)
    _need(w1_scales, "w1_scales", torch.bfloat16, 3)
    _need(w2_scales, "w2_scales", torch.bfloat16, 3)
    if out is None:
        out = torch.empty_like(hidden)
    _check(lib().moe_w4a16_forward_noalloc(_p(hidden), _p(topk_ids), _p(topk_w), _p(w1_packed), _p(w1_scales),
                                           _p(w2_packed), _p(w2_scales), _p(out), dims, _stream(stream)),
           "moe_w4a16_forward_noalloc")
    return out


def moe_w4a16_forward_rms(hidden, topk_ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales,
                          eps: float = 1e-6, next=None, ws=None, stream=None):
    """Forward, then next = bf16((hidden + moe) / rms(hidden + moe)) (stack epilogue)."""
    dims = _expert_dims(hidden, topk_ids, w1_packed, w2_packed)
    _need(topk_w, "topk_w", torch.float32, 2)
    _need(w1_scales, "w1_scales", torch.bfloat16, 3)
    _need(w2_scales, "w2_scales", torch.bfloat16, 3)
    ws = _ws(ws, dims, hidden.device)
    if next is None:
        next = torch.empty_like(hidden)
    _check(lib().moe_w4a16_forward_rms(_p(hidden), _p(topk_ids), _p(topk_w), _p(w1_packed), _p(w1_scales),
                                       _p(w2_packed), _p(w2_scales), _p(next), float(eps), dims, _p(ws),
                                       ws.numel(), _stream(stream)), "moe_w4a16_forward_rms")
    return next


def moe_layer_forward(hidden, router_w, k: int, w1_packed, w1_scales, w2_packed, w2_scales, bias=None,
                      shared: bool = False, rms: bool = False, eps: float = 1e-6, out=None, topk_ids=None,
                      topk_w=None, ws=None, stream=None):
    """Router and experts in one call: moe_route (moe_route_shared with shared)
    then moe_w4a16_forward (moe_w4a16_forward_rms with rms), one kernel for
    decode batches. router_w [E (+1), H]; the weights hold E (+1) experts.

    Returns (out or next bf16 [T, H], topk_ids int32 [T, k (+1)], topk_w f32 [T, k (+1)]).
    """
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(router_w, "router_w", torch.bfloat16, 2)
    _need(w1_packed, "w1_packed", torch.int32, 3)
    _need(w2_packed, "w2_packed", torch.int32, 3)
    _need(w1_scales, "w1_scales", torch.bfloat16, 3)
    _need(w2_scales, "w2_scales", torch.bfloat16, 3)
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
    T, H = hidden.shape
    g = 1 if shared else 0
    E = router_w.shape[0] - g
    I = w1_packed.shape[1] // 2
    if w1_packed.shape[0] != E + g or w2_packed.shape[0] != E + g:
        raise ValueError("the weights must hold %d experts (router rows %d%s), got %d and %d"
                         % (E + g, router_w.shape[0], ", the last the shared gate" if g else "",
                            w1_packed.shape[0], w2_packed.shape[0]))
    dims = moe_dims(T, H, E, k, I)
    if ws is None:
        ws = shared_workspace(T, H, E, k, I, hidden.device) if shared else workspace(T, H, E, k, I, hidden.device)
    if topk_ids is None:
        topk_ids = torch.empty(T, k + g, dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty(T, k + g, dtype=torch.float32, device=hidden.device)
    if out is None:
        out = torch.empty_like(hidden)
    _check(lib().moe_layer_forward(_p(hidden), _p(router_w), _p(bias), g, _p(w1_packed), _p(w1_scales),
                                   _p(w2_packed), _p(w2_scales), None if rms else _p(out), _p(out) if rms else None,
                                   float(eps), _p(topk_ids), _p(topk_w), dims, _p(ws), ws.numel(), _stream(stream)),
           "moe_layer_forward")
    return out, topk_ids, topk_w


def moe_permute(topk_ids, E: int, H: int = 128, I: int = 128, ws=None, stream=None):
    """(offsets int32 [E+1], perm int32 [T*k]) of the stable token-to-expert permutation."""
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, k = topk_ids.shape
    dims = moe_dims(T, H, E, k, I)
    ws = _ws(ws, dims, topk_ids.device)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=topk_ids.device)
    perm = torch.empty(T * k, dtype=torch.int32, device=topk_ids.device)
    _check(lib().moe_permute(_p(topk_ids), dims, _p(offsets), _p(perm), _p(ws), ws.numel(), _stream(stream)),
           "moe_permute")
    return offsets, perm


def moe_pack_int4(q, bad_count=None, stream=None):
    """int32 [N, K/8] storage words of int8 q [N, K] in [-8, 7]."""
    _need(q, "q", torch.int8, 2)
    N, K = q.shape
    packed = torch.empty(N, K // 8, dtype=torch.int32, device=q.device)
    if bad_count is not None:
        _need(bad_count, "bad_count", torch.int32, 1)
    _check(lib().moe_pack_int4(_p(q), N, K, _p(packed), _p(bad_count), _stream(stream)), "moe_pack_int4")
    return packed


def moe_forward_plan(T: int, H: int, E: int, k: int, I: int):
    """None if a forward of these dims takes the tensor-core pipeline, else
    (staged, groups_per_chunk, separate_block_buffers, routes_itself) of the
    fused decode kernel it runs; routes_itself: moe_layer_forward runs the
    router in the same kernel for these (forward) dims."""
    v = ctypes.c_int32(-1)
    _check(lib().moe_forward_plan(moe_dims(T, H, E, k, I), ctypes.byref(v)), "moe_forward_plan")
    if v.value == 0:
        return None
    return (v.value & 15) == 1, (v.value >> 4) & 15, bool(v.value & 256), bool(v.value & 512)


def moe_quantize_int4(w, nclip: int = 50, with_choice: bool = False, stream=None):
    """RTN INT4 g128 symmetric quantisation of bf16 w [N, K] with a per-group clip search.

    Returns (packed int32 [N, K/8], scales bf16 [N, K/128]) and, with with_choice,
    the chosen clip index int32 [N, K/128] (clip = (100 - j) / 100).
    """
    _need(w, "w", torch.bfloat16, 2)
    N, K = w.shape
    packed = torch.empty(N, K // 8, dtype=torch.int32, device=w.device)
    scales = torch.empty(N, K // 128, dtype=torch.bfloat16, device=w.device)
    choice = torch.empty(N, K // 128, dtype=torch.int32, device=w.device) if with_choice else None
    _check(lib().moe_quantize_int4(_p(w), N, K, nclip, _p(packed), _p(scales), _p(choice), _stream(stream)),
           "moe_quantize_int4")
    return (packed, scales, choice) if with_choice else (packed, scales)


def moe_w8a16_linear(x, w_packed, scales, gs: int, y=None, ws=None, stream=None):
    """bf16 y [T, N] = x . W^T for INT8 pack-quantized W (q + 128, four per int32 word, LSB first)
    with bf16 scales per gs (64 or 128) values of K. T <= 8: the decode GEMV; larger T: the
    tensor-core GEMM, whose error word (and split partial results) live in ws (a zeroed uint8
    tensor of moe_w8a16_workspace_size bytes; allocated here when not given)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(w_packed, "w_packed", torch.int32, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    T, K = x.shape
    N = w_packed.shape[0]
    if w_packed.shape[1] * 4 != K or scales.shape != (N, K // gs):
        raise ValueError("w_packed must be [N, K/4] and scales [N, K/gs]")
    if y is None:
        y = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    if ws is None and T > 8:
        ws = torch.zeros(moe_w8a16_workspace_size(T, N, K, gs), dtype=torch.uint8, device=x.device)
    nbytes = 0 if ws is None else ws.numel()
    _check(lib().moe_w8a16_linear(_p(x), _p(w_packed), _p(scales), gs, _p(y), T, N, K, _p(ws), nbytes,
                                  _stream(stream)), "moe_w8a16_linear")
    return y


def moe_w8a16_workspace_size(T: int, N: int, K: int, gs: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_w8a16_workspace_size(T, N, K, gs, ctypes.byref(n)), "moe_w8a16_workspace_size")
    return n.value


def moe_profile_events(before=None, after=None):
    """Record two torch.cuda.Events (enable_timing=True, external=True) around
    the expert kernel of every later forward call; (None, None) stops."""
    b = None if before is None else ctypes.c_void_p(before.cuda_event)
    a = None if after is None else ctypes.c_void_p(after.cuda_event)
    _check(lib().moe_profile_events(b, a), "moe_profile_events")


def moe_check_device_error(ws, stream=None) -> int:
    """Synchronise the stream; return (and clear) the workspace's device error status."""
    return lib().moe_check_device_error(_p(ws), ws.numel(), _stream(stream))


def moe_noalloc_check_device_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the error status of the no-alloc scratch."""
    return lib().moe_noalloc_check_device_error(_stream(stream))
