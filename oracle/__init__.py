"""ctypes front end of the fp64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the entry module's smoke
check and the benchmark's CPU-baseline leg, never by the CUDA library or its
binding. It shares no code with the CUDA path; inputs come from ``synth``.

Parity of the expert outputs is pinned by brute force, closed forms and
invariants (tests/test_oracle.py); the pages print no worked example of the
layer's output values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "moe_oracle.c")
_LIB = os.path.join(_DIR, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c11",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_unpack_int4.argtypes = [P, I64, I64, P]
        L.oracle_pack_int4.argtypes = [P, I64, I64, P]
        L.oracle_pack_int4.restype = I
        L.oracle_dequant.argtypes = [P, P, I64, I64, P]
        L.oracle_router_logits.argtypes = [P, P, P, I, I, I, P, I]
        L.oracle_topk_softmax.argtypes = [P, I, I, I, P, P]
        L.oracle_topk_softmax.restype = I
        L.oracle_permute.argtypes = [P, I, I, I, P, P]
        L.oracle_permute.restype = I
        L.oracle_expert_forward.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, I]
        L.oracle_expert_forward.restype = I
        L.oracle_residual_rms.argtypes = [P, P, I, I, ctypes.c_double, P, P]
        L.oracle_round_bf16.argtypes = [P, I64, P]
        L.oracle_max_threads.restype = I
        L.oracle_shared_expert.argtypes = [P, P, P, P, P, P, I, I, I, P, P, I]
        L.oracle_shared_combine.argtypes = [P, P, P, I, I, P]
        L.oracle_quantize_int4.argtypes = [P, I64, I64, I, P, P, P, P]
        L.oracle_quantize_int4.restype = I
        L.oracle_unpack_int8.argtypes = [P, I64, I64, P]
        L.oracle_pack_int8.argtypes = [P, I64, I64, P]
        L.oracle_pack_int8.restype = I
        L.oracle_w8a16_linear.argtypes = [P, P, P, I, I, I64, I64, P, I]
        L.oracle_w8a16_linear.restype = I
        _lib = L
    return _lib


def _np(a, dtype) -> np.ndarray:
    """Contiguous numpy view of a host tensor/array; bf16 comes through as its bits."""
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().contiguous()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    dt = np.dtype(dtype)
    if a.dtype == dt:
        return a
    if dt.kind in "iu" and a.dtype.kind in "iu" and a.dtype.itemsize == dt.itemsize:
        return a.view(dt)
    return a.astype(dt)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return lib().oracle_max_threads()


def unpack_int4(packed, N: int, K: int) -> np.ndarray:
    p = _np(packed, np.int32)
    q = np.empty((N, K), np.int8)
    lib().oracle_unpack_int4(_p(p), N, K, _p(q))
    return q


def pack_int4(q) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    out = np.empty((N, K // 8), np.int32)
    if lib().oracle_pack_int4(_p(q), N, K, _p(out)) != 0:
        raise ValueError("value outside [-8, 7]")
    return out


def dequant(packed, scales, N: int, K: int) -> np.ndarray:
    p, s = _np(packed, np.int32), _np(scales, np.uint16)
    W = np.empty((N, K), np.float64)
    lib().oracle_dequant(_p(p), _p(s), N, K, _p(W))
    return W


def router_logits(x, wr, bias=None, nthreads: int = 0) -> np.ndarray:
    xs, ws = _np(x, np.uint16), _np(wr, np.uint16)
    T, H = xs.shape
    E = ws.shape[0]
    b = None if bias is None else _np(bias, np.float32)
    out = np.empty((T, E), np.float64)
    lib().oracle_router_logits(_p(xs), _p(ws), None if b is None else _p(b), T, H, E, _p(out), nthreads)
    return out


def topk_softmax(logits: np.ndarray, k: int):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = l.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib().oracle_topk_softmax(_p(l), T, E, k, _p(ids), _p(w)) != 0:
        raise ValueError("bad k")
    return ids, w


def route(x, wr, k: int, bias=None, nthreads: int = 0):
    """(ids [T,k] int32, weights [T,k] f64, logits [T,E] f64)."""
    logits = router_logits(x, wr, bias, nthreads)
    ids, w = topk_softmax(logits, k)
    return ids, w, logits


def permute(ids, E: int):
    i = _np(ids, np.int32)
    T, k = i.shape
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    if lib().oracle_permute(_p(i), T, k, E, _p(offsets), _p(perm)) != 0:
        raise ValueError("expert id out of range")
    return offsets, perm


def expert_forward(x, ids, topk_w, w1_packed, w1_scales, w2_packed, w2_scales,
                   E: int, I: int, expert_row=None, nthreads: int = 0) -> np.ndarray:
    """fp64 out [T, H] of the expert path for given routing (ids, weights)."""
    xs = _np(x, np.uint16)
    T, H = xs.shape
    i = _np(ids, np.int32)
    k = i.shape[1]
    w = _np(topk_w, np.float32)
    p1, s1 = _np(w1_packed, np.int32), _np(w1_scales, np.uint16)
    p2, s2 = _np(w2_packed, np.int32), _np(w2_scales, np.uint16)
    n_held = p1.shape[0]
    er = None if expert_row is None else np.ascontiguousarray(expert_row, dtype=np.int32)
    out = np.empty((T, H), np.float64)
    rc = lib().oracle_expert_forward(_p(xs), _p(i), _p(w), _p(p1), _p(s1), _p(p2), _p(s2),
                                     None if er is None else _p(er), n_held,
                                     T, H, E, k, I, _p(out), nthreads)
    if rc != 0:
        raise ValueError("expert id out of range or not held (rc=%d)" % rc)
    return out


def residual_rms(x, out: np.ndarray, eps: float = 1e-6):
    """(x_next bf16 bits as torch.bfloat16 [T,H], x_next before rounding f64)."""
    xs = _np(x, np.uint16)
    T, H = xs.shape
    o = np.ascontiguousarray(out, dtype=np.float64)
    nb = np.empty((T, H), np.uint16)
    nf = np.empty((T, H), np.float64)
    lib().oracle_residual_rms(_p(xs), _p(o), T, H, eps, _p(nb), _p(nf))
    return torch.from_numpy(nb.view(np.int16)).view(torch.bfloat16), nf


def round_bf16(v: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float64)
    bits = np.empty(a.shape, np.uint16)
    lib().oracle_round_bf16(_p(a), a.size, _p(bits))
    return bits


def shared_expert(x, wg, w1_packed, w1_scales, w2_packed, w2_scales, I: int, nthreads: int = 0):
    """(gate logits f64 [T], unweighted shared-expert output f64 [T, H]).

    wg bf16 [H] is the router's extra row; the weights are one expert in the
    routed experts' storage: w1 [2I, H/8] / [2I, H/128], w2 [H, I/8] / [H, I/128].
    """
    xs = _np(x, np.uint16)
    T, H = xs.shape
    g = _np(wg, np.uint16).reshape(-1)
    p1, s1 = _np(w1_packed, np.int32), _np(w1_scales, np.uint16)
    p2, s2 = _np(w2_packed, np.int32), _np(w2_scales, np.uint16)
    gate = np.empty(T, np.float64)
    y = np.empty((T, H), np.float64)
    lib().oracle_shared_expert(_p(xs), _p(g), _p(p1), _p(s1), _p(p2), _p(s2), T, H, I, _p(gate), _p(y), nthreads)
    return gate, y


def shared_combine(routed: np.ndarray, gate: np.ndarray, y: np.ndarray) -> np.ndarray:
    """routed + sigmoid(gate) * y, f64 [T, H]."""
    r = np.ascontiguousarray(routed, dtype=np.float64)
    g = np.ascontiguousarray(gate, dtype=np.float64)
    yy = np.ascontiguousarray(y, dtype=np.float64)
    T, H = r.shape
    out = np.empty((T, H), np.float64)
    lib().oracle_shared_combine(_p(r), _p(g), _p(yy), T, H, _p(out))
    return out


def quantize_int4(w, nclip: int = 50):
    """RTN INT4 g128 symmetric with a per-group clip search over nclip candidates.

    w bf16 [N, K]. Returns (packed int32 [N, K/8], scales bf16 bits uint16 [N, K/128],
    choice int32 [N, K/128] (the clip index j, c_j = (100 - j)/100), err f64 [N, K/128, nclip]).
    """
    ws = _np(w, np.uint16)
    N, K = ws.shape
    G = K // 128
    packed = np.empty((N, K // 8), np.int32)
    scales = np.empty((N, G), np.uint16)
    choice = np.empty((N, G), np.int32)
    err = np.empty((N, G, nclip), np.float64)
    if lib().oracle_quantize_int4(_p(ws), N, K, nclip, _p(err), _p(packed), _p(scales), _p(choice)) != 0:
        raise ValueError("K must be a multiple of 128 and 1 <= nclip <= 100")
    return packed, scales, choice, err


def unpack_int8(packed, N: int, K: int) -> np.ndarray:
    """q int16 [N, K] in [-128, 127] from INT8 pack-quantized words int32 [N, K/4]."""
    p = _np(packed, np.int32)
    q = np.empty((N, K), np.int16)
    lib().oracle_unpack_int8(_p(p), N, K, _p(q))
    return q


def pack_int8(q) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int16)
    N, K = q.shape
    out = np.empty((N, K // 4), np.int32)
    if lib().oracle_pack_int8(_p(q), N, K, _p(out)) != 0:
        raise ValueError("value outside [-128, 127]")
    return out


def w8a16_linear(x, packed, scales, gs: int, nthreads: int = 0) -> np.ndarray:
    """fp64 y [T, N] = x . W^T for INT8 weights (q + 128, LSB first) with bf16 scales per gs of K."""
    xs = _np(x, np.uint16)
    T, K = xs.shape
    p = _np(packed, np.int32)
    N = p.shape[0]
    s = _np(scales, np.uint16)
    y = np.empty((T, N), np.float64)
    if lib().oracle_w8a16_linear(_p(xs), _p(p), _p(s), gs, T, N, K, _p(y), nthreads) != 0:
        raise ValueError("gs must be 64 or 128 and divide K")
    return y
