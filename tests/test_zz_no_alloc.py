"""moe_w4a16_forward_noalloc: the decode forward with the library's static scratch.

The GPU tests compare it, through the C ABI, with moe_w4a16_forward (caller
workspace) on the same inputs: two calls in a row, shapes changing between
calls, and a fresh process whose first library call is the no-alloc one (the
call that does the per-device set-up). The bar is the forward's output bar,
max|a - b| <= 1e-2 * max|b|. The argument checks run before any CUDA call and
are tested on the CPU.

This file is named to be collected last, so that the no-alloc path also runs
after every other test has used the library in the same process.
"""
import ctypes
import os
import subprocess
import sys

import pytest
import torch

import synth
import w4a16_mixture_experts_gb300 as moe

OUT_TOL = 1e-2
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _close(a, b):
    a, b = a.float().cpu(), b.float().cpu()
    assert torch.isfinite(a).all()
    bound = OUT_TOL * b.abs().max().item()
    err = (a - b).abs().max().item()
    assert err <= bound, (err, bound)
    return err


# ------------------------------------------------------------ CPU checks ----

def _fake(nbytes=16):
    buf = (ctypes.c_char * (nbytes + 256))()
    return ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, ctypes.c_void_p), buf


def _call(T, H, E, k, I, null_out=False):
    p, keep = _fake()
    out = None if null_out else p
    return moe.lib().moe_w4a16_forward_noalloc(p, p, p, p, p, p, p, out, moe.moe_dims(T, H, E, k, I), None)


@pytest.fixture(scope="module")
def _built():
    moe.build()
    moe.lib()


def test_noalloc_rejects_shapes_before_any_cuda_call(_built):
    # T beyond the decode path
    assert _call(9, 2560, 512, 10, 640) == 2                       # MOE_ERR_UNSUPPORTED
    # a decode shape whose workspace exceeds the 1 MiB static scratch
    assert moe.moe_forward_plan(7, 6144, 1024, 32, 640) is not None
    need = moe.moe_workspace_size(7, 6144, 1024, 32, 640)
    assert need > (1 << 20)
    assert _call(7, 6144, 1024, 32, 640) == 3                      # MOE_ERR_WORKSPACE
    # shapes every forward rejects
    assert _call(1, 200, 512, 10, 640) == 2
    assert _call(-1, 2560, 512, 10, 640) == 1
    # a missing output pointer for a non-empty batch
    assert _call(1, 2560, 512, 10, 640, null_out=True) == 1


def test_noalloc_capacity_covers_the_decode_path_at_full_shape():
    assert moe.moe_workspace_size(7, 2560, 512, 10, 640) <= (1 << 20)


# ------------------------------------------------------------ GPU parity ----

_weights = {}


def _inputs(T, H, E, k, I, seed):
    key = (H, E, I, seed)
    if key not in _weights:
        _weights.clear()
        w = synth.expert_weights(E, H, I, seed=seed)
        _weights[key] = [w[n].cuda() for n in ("w1_packed", "w1_scales", "w2_packed", "w2_scales")]
    x = synth.hidden(T, H, seed=seed + T).cuda()
    ids, tw = synth.random_topk(T, E, k, seed=seed + T)
    return x, ids.cuda(), tw.cuda(), _weights[key]


def _pair(T, H, E, k, I, seed=11):
    x, ids, tw, W = _inputs(T, H, E, k, I, seed)
    ws = moe.workspace(T, H, E, k, I)
    ref = moe.moe_w4a16_forward(x, ids, tw, *W, ws=ws)
    a = moe.moe_w4a16_forward_noalloc(x, ids, tw, *W)
    a_err = moe.moe_noalloc_check_device_error()
    b = moe.moe_w4a16_forward_noalloc(x, ids, tw, *W)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    # neither call saw a bad id or gave up a wait inside the static scratch
    assert a_err == 0 and moe.moe_noalloc_check_device_error() == 0
    return ref, a, b


@pytest.mark.gpu
@pytest.mark.parametrize("T", [1, 4, 7])
def test_noalloc_matches_workspace_forward_twice(_built, T):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ref, a, b = _pair(T, 2560, 512, 10, 640)
    _close(a, ref)
    _close(b, ref)


@pytest.mark.gpu
def test_noalloc_shape_changes_between_calls(_built):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # each call's counters sit where the previous shape kept other data
    for T, k in [(7, 10), (1, 10), (5, 3), (7, 10), (3, 8)]:
        ref, a, b = _pair(T, 2560, 512, k, 640, seed=5)
        _close(a, ref)
        _close(b, ref)


@pytest.mark.gpu
def test_noalloc_reports_a_bad_id(_built):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x, ids, tw, W = _inputs(3, 2560, 512, 10, 640, seed=13)
    bad = ids.clone()
    bad[1, 2] = 512 + 7
    moe.moe_w4a16_forward_noalloc(x, bad, tw, *W)
    assert moe.moe_noalloc_check_device_error() == 5     # MOE_ERR_DEVICE, then cleared
    assert moe.moe_noalloc_check_device_error() == 0
    # the next call starts clean and matches the workspace forward
    ref, a, b = _pair(3, 2560, 512, 10, 640, seed=13)
    _close(a, ref)


@pytest.mark.gpu
def test_noalloc_empty_batch(_built):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    tw = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    w = synth.expert_weights(16, 256, 128, seed=1)
    W = [w[n].cuda() for n in ("w1_packed", "w1_scales", "w2_packed", "w2_scales")]
    out = moe.moe_w4a16_forward_noalloc(x, ids, tw, *W)
    assert out.shape == (0, 256)


_FRESH = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import synth, w4a16_mixture_experts_gb300 as moe
T, H, E, k, I = 4, 256, 16, 2, 128
w = synth.expert_weights(E, H, I, seed=2)
W = [w[n].cuda() for n in ("w1_packed", "w1_scales", "w2_packed", "w2_scales")]
x = synth.hidden(T, H, seed=2).cuda()
ids, tw = synth.random_topk(T, E, k, seed=2)
ids, tw = ids.cuda(), tw.cuda()
a = moe.moe_w4a16_forward_noalloc(x, ids, tw, *W)      # first library call: set-up
b = moe.moe_w4a16_forward_noalloc(x, ids, tw, *W)
assert moe.moe_noalloc_check_device_error() == 0
ref = moe.moe_w4a16_forward(x, ids, tw, *W, ws=moe.workspace(T, H, E, k, I))
torch.cuda.synchronize()
bound = 1e-2 * ref.float().abs().max().item()
ea = (a.float() - ref.float()).abs().max().item()
eb = (b.float() - ref.float()).abs().max().item()
print("fresh", ea, eb, bound)
sys.exit(0 if ea <= bound and eb <= bound else 1)
"""


@pytest.mark.gpu
def test_noalloc_first_call_in_fresh_process(_built):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
