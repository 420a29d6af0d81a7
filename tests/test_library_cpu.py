"""Host-side checks of the C-ABI library that need no GPU.

The library must build for sm_103a, load, export every entry point that
include/w4a16moe.h declares, and reject bad arguments synchronously, before
touching the device.
"""
import ctypes
import os
import re

import pytest

import w4a16_mixture_experts_gb300 as moe
from w4a16_mixture_experts_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16moe.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return moe.lib()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("moe_route", "moe_w4a16_forward", "moe_workspace_size", "moe_permute", "moe_pack_int4",
              "moe_check_device_error", "moe_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared():
        assert hasattr(L, name), name
    out = os.popen("nm -D --defined-only %s" % moe.LIB_PATH).read()
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    assert set(declared()) <= exported
    assert all(n in declared() for n in exported), "undeclared export"


def test_status_strings(L):
    for s in range(7):
        assert moe.moe_status_str(s)
    assert moe.moe_status_str(99) == "unknown status"
    assert moe.moe_version() >= 100


def test_workspace_size_and_shape_rules(L):
    n = moe.moe_workspace_size(1, 2560, 512, 10, 640)
    assert n > 0 and n % 256 == 0
    assert moe.moe_workspace_size(64, 2560, 512, 10, 640) > n
    bad = [
        (1, 2560 + 64, 512, 10, 640),   # H not a multiple of 128
        (1, 2560, 512, 10, 600),        # I not a multiple of 128
        (1, 2560, 512, 33, 640),        # k > 32
        (1, 2560, 2048, 10, 640),       # E > 1024
        (1, 2560, 8, 10, 640),          # k > E
        (1, 16384, 512, 10, 640),       # H > 8192
    ]
    for dims in bad:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_workspace_size(*dims)
        assert ei.value.status == 2
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(-1, 2560, 512, 10, 640)
    assert ei.value.status == 1
    # the fp32 accumulator's token rows are addressed by 32-bit offsets: T * H < 2^32
    assert moe.moe_workspace_size(500_000, 8064, 512, 10, 640) > 0
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(600_000, 8064, 512, 10, 640)
    assert ei.value.status == 2
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size((1 << 20) + 1, 128, 16, 2, 128)
    assert ei.value.status == 2


def _call_forward(L, dims, ptrs, ws_bytes):
    return L.moe_w4a16_forward(*[ctypes.c_void_p(p) for p in ptrs[:7]], ctypes.c_void_p(ptrs[7]), dims,
                               ctypes.c_void_p(ptrs[8]), ws_bytes, None)


def test_argument_errors_are_synchronous(L):
    """Fake, never-dereferenced addresses: every call must fail before any CUDA work."""
    d = moe.moe_dims(4, 256, 16, 2, 128)
    need = moe.moe_workspace_size(4, 256, 16, 2, 128)
    good = [0x10000 * (i + 1) for i in range(9)]
    # a null weight pointer
    ptrs = list(good)
    ptrs[3] = 0
    assert _call_forward(L, d, ptrs, need) == 1
    # a misaligned pointer
    ptrs = list(good)
    ptrs[0] += 8
    assert _call_forward(L, d, ptrs, need) == 1
    # a workspace that is too small
    assert _call_forward(L, d, good, need - 256) == 3
    # unsupported shape
    assert _call_forward(L, moe.moe_dims(4, 200, 16, 2, 128), good, need) == 2
    # route with a misaligned bias
    assert L.moe_route(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2] + 4), d,
                       ctypes.c_void_p(good[3]), ctypes.c_void_p(good[4]), ctypes.c_void_p(good[5]), need,
                       None) == 1
    # pack with K not a multiple of 8
    assert L.moe_pack_int4(ctypes.c_void_p(good[0]), 4, 12, ctypes.c_void_p(good[1]), None, None) == 1
    # quantiser: K not a multiple of 128, nclip outside [1, 100]
    assert L.moe_quantize_int4(ctypes.c_void_p(good[0]), 4, 200, 50, ctypes.c_void_p(good[1]),
                               ctypes.c_void_p(good[2]), None, None) == 1
    for nclip in (0, 101):
        assert L.moe_quantize_int4(ctypes.c_void_p(good[0]), 4, 256, nclip, ctypes.c_void_p(good[1]),
                                   ctypes.c_void_p(good[2]), None, None) == 1
    # W8A16: gs other than 64/128, K not a multiple of gs, a batch without its workspace
    assert L.moe_w8a16_linear(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2]), 32,
                              ctypes.c_void_p(good[3]), 4, 16, 256, None, 0, None) == 1
    assert L.moe_w8a16_linear(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2]), 128,
                              ctypes.c_void_p(good[3]), 4, 16, 320, None, 0, None) == 1
    assert L.moe_w8a16_linear(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2]), 64,
                              ctypes.c_void_p(good[3]), 64, 16, 256, None, 0, None) == 1
    assert L.moe_w8a16_linear(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2]), 64,
                              ctypes.c_void_p(good[3]), 64, 16, 256, ctypes.c_void_p(good[4]), 128, None) == 3
    # the split GEMM needs its partial results' room: less than the reported size is refused
    need = moe.moe_w8a16_workspace_size(512, 320, 10240, 64)
    assert need >= 256 + 2 * 512 * 320 * 4
    assert L.moe_w8a16_linear(ctypes.c_void_p(good[0]), ctypes.c_void_p(good[1]), ctypes.c_void_p(good[2]), 64,
                              ctypes.c_void_p(good[3]), 512, 320, 10240, ctypes.c_void_p(good[4]), need - 16,
                              None) == 3
    assert moe.moe_w8a16_workspace_size(1, 320, 10240, 64) == 256
    # shared-expert routing: k + 1 must stay within 32 slots, E + 1 within 1024 experts
    assert L.moe_route_shared(*[ctypes.c_void_p(p) for p in good[:3]], moe.moe_dims(4, 256, 64, 32, 128),
                              ctypes.c_void_p(good[3]), ctypes.c_void_p(good[4]), ctypes.c_void_p(good[5]),
                              1 << 30, None) == 2
    assert L.moe_route_shared(*[ctypes.c_void_p(p) for p in good[:3]], moe.moe_dims(4, 256, 1024, 8, 128),
                              ctypes.c_void_p(good[3]), ctypes.c_void_p(good[4]), ctypes.c_void_p(good[5]),
                              1 << 30, None) == 2
    # device-error check with no workspace
    assert L.moe_check_device_error(None, 0, None) == 1
    # empty batch: nothing to do, no device access
    e = moe.moe_dims(0, 256, 16, 2, 128)
    assert L.moe_w4a16_forward(None, None, None, *[ctypes.c_void_p(p) for p in good[:4]], None, e,
                               ctypes.c_void_p(good[5]), need, None) == 0


def test_workspace_holds_the_regions_of_the_path_taken():
    """A small batch the fused decode kernel cannot take (I > 1280) runs the
    prefill pipeline, so its workspace must hold the per-slot activations and
    the fp32 accumulator; a decode-sized batch of the same kind does not."""
    T, H, E, k = 4, 256, 16, 2
    big = moe.moe_workspace_size(T, H, E, k, 1408)
    small = moe.moe_workspace_size(T, H, E, k, 128)
    assert big >= T * k * H * 2 + T * H * 4 + T * k * 1408 * 2
    # the same fixed head (control block, per-expert counters for every id) in
    # both; only the prefill one adds the per-slot activations and the accumulator
    assert small + T * k * H * 2 + T * H * 4 <= big


def _call_layer(L, dims, p, ws_bytes, shared=0, out=True, nxt=False, eps=1e-6, bias=None):
    """moe_layer_forward with fake, never-dereferenced addresses p[0..12]."""
    v = lambda i: ctypes.c_void_p(p[i])
    return L.moe_layer_forward(v(0), v(1), None if bias is None else ctypes.c_void_p(bias), shared, v(2), v(3), v(4),
                               v(5), v(6) if out else None, v(7) if nxt else None, eps, v(8), v(9), dims, v(10),
                               ws_bytes, None)


def test_layer_call_argument_errors_are_synchronous(L):
    """moe_layer_forward's checks: every refusal comes before any CUDA work."""
    d = moe.moe_dims(2, 256, 16, 2, 128)
    need = max(moe.moe_workspace_size(2, 256, 16, 2, 128), moe.moe_workspace_size(2, 256, 17, 3, 128))
    good = [0x10000 * (i + 1) for i in range(11)]
    # `shared` is 0 or 1
    assert _call_layer(L, d, good, need, shared=2) == 1
    # exactly one of out and next
    assert _call_layer(L, d, good, need, out=True, nxt=True) == 1
    assert _call_layer(L, d, good, need, out=False, nxt=False) == 1
    # the stack step needs eps >= 0
    assert _call_layer(L, d, good, need, out=False, nxt=True, eps=-1.0) == 1
    # a null weight, a misaligned router, a misaligned bias
    p = list(good)
    p[4] = 0
    assert _call_layer(L, d, p, need) == 1
    p = list(good)
    p[1] += 8
    assert _call_layer(L, d, p, need) == 1
    assert _call_layer(L, d, good, need, bias=good[0] + 4) == 1
    # the shared expert: k + 1 within 32 slots, E + 1 within 1024 experts
    assert _call_layer(L, moe.moe_dims(2, 256, 64, 32, 128), good, 1 << 30, shared=1) == 2
    assert _call_layer(L, moe.moe_dims(2, 256, 1024, 8, 128), good, 1 << 30, shared=1) == 2
    # the workspace must serve the router's dims and the forward's (one more expert and slot)
    small = moe.moe_workspace_size(2, 256, 16, 2, 128)
    big = moe.moe_workspace_size(2, 256, 17, 3, 128)
    assert big > small
    assert _call_layer(L, d, good, big - 16, shared=1) == 3
    assert _call_layer(L, d, good, small - 16) == 3
    # an empty batch: nothing to do (no output needed)
    e = moe.moe_dims(0, 256, 16, 2, 128)
    assert _call_layer(L, e, [0, good[1], good[2], good[3], good[4], good[5], 0, 0, 0, 0, good[10]], need,
                       out=False) == 0
