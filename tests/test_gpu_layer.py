"""moe_layer_forward: the router and the routed experts in one call.

Where the decode kernel runs the router itself (moe_forward_plan reports
routes_itself for the forward's dims), it computes the logits and selects with
the small-batch router's own code and runs the same expert code, so the
selection, the weights and the output must equal those of the separate calls
(moe_route or moe_route_shared, then moe_w4a16_forward or _rms) bit for bit.
Elsewhere the call runs those calls' kernels one after the other. The separate
calls are checked against the fp64 oracle in test_gpu_parity.py and
test_gpu_shared.py; the layer call is also checked against the oracle here, at
the benchmark's shapes ("vLLM Optimization Edition", section 3.3 "MoE block
(decode-05)": router GEMV, top-k, fused experts, moe_sum).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a16_mixture_experts_gb300 as moe
from test_gpu_parity import assert_close, check_route

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()


def _inputs(T, H, E, k, I, shared, bias, seed):
    g = E + (1 if shared else 0)
    h = {
        "hidden": synth.hidden(T, H, seed=seed),
        "router_w": synth.router(g, H, seed=seed),
        "bias": synth.zipf_bias(E, 1.1, seed=seed) if bias else None,
    }
    h.update(synth.expert_weights(g, H, I, seed=seed))
    return h, {key: (v.cuda() if v is not None else None) for key, v in h.items()}


def _ws(T, H, E, k, I, shared):
    return moe.shared_workspace(T, H, E, k, I) if shared else moe.workspace(T, H, E, k, I)


def _weights(d):
    return d["w1_packed"], d["w1_scales"], d["w2_packed"], d["w2_scales"]


def _separate(d, k, shared, rms, eps, ws):
    x = d["hidden"]
    route = moe.moe_route_shared if shared else moe.moe_route
    ids, w = route(x, d["router_w"], k, bias=d["bias"], ws=ws)
    if rms:
        out = moe.moe_w4a16_forward_rms(x, ids, w, *_weights(d), eps=eps, ws=ws)
    else:
        out = moe.moe_w4a16_forward(x, ids, w, *_weights(d), ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    return out, ids, w


def _layer(d, k, shared, rms, eps, ws):
    out, ids, w = moe.moe_layer_forward(d["hidden"], d["router_w"], k, *_weights(d), bias=d["bias"], shared=shared,
                                        rms=rms, eps=eps, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    return out, ids, w


def _same(a, b, what, exact_out=True):
    for x, y, name in zip(a, b, ("out", "ids", "w")):
        if name == "out" and not exact_out:
            # the tensor-core pipeline sums the experts, and the decode stack step
            # the per-token sums of squares, in arrival order: within a bf16
            # rounding of the other call's output
            d = (x.float() - y.float()).abs().max().item()
            assert d <= 2.0 ** -7 * y.float().abs().max().item(), "%s: out differs by %g" % (what, d)
            continue
        assert torch.equal(x, y), "%s: %s differs from the separate calls" % (what, name)


# (T, H, E, k, I, shared, rms, bias, the kernel routes itself)
CASES = [
    (1, 2560, 512, 10, 640, False, False, False, True),    # decode1
    (2, 2560, 512, 10, 640, False, False, True, True),     # two tokens, a Zipf router bias
    (1, 2560, 512, 10, 640, True, False, False, True),     # a shared expert
    (2, 2560, 512, 10, 640, False, True, False, True),     # the stack step
    (1, 2560, 512, 10, 640, True, True, True, True),       # all three
    (2, 512, 1024, 16, 128, False, False, False, True),    # 1024 router rows: the CTAs' rows in two passes
    (2, 256, 16, 2, 128, False, False, False, True),       # a small grid, 4 rows a CTA
    (1, 512, 777, 31, 128, True, False, True, True),       # ragged rows, k + 1 = 32 slots
    (2, 128, 1024, 8, 128, False, True, False, True),      # the smallest ring holds the logits
    (2, 512, 256, 24, 128, False, False, True, True),      # 48 assignments: the CTA-wide prologue after the selection
    (4, 2560, 512, 10, 640, False, False, True, False),    # from 3 tokens: the router's kernel, then the forward's
    (8, 2560, 512, 10, 640, True, True, False, False),
    (9, 2560, 512, 10, 640, False, False, False, False),   # T > 8: router kernels, tensor-core pipeline
]


@pytest.mark.parametrize("T,H,E,k,I,shared,rms,bias,fused", CASES)
def test_layer_equals_separate_calls(T, H, E, k, I, shared, rms, bias, fused):
    g = 1 if shared else 0
    plan = moe.moe_forward_plan(T, H, E + g, k + g, I)
    assert (plan is not None and plan[3]) == fused
    h, d = _inputs(T, H, E, k, I, shared, bias, seed=T * 7 + E)
    ref = _separate(d, k, shared, rms, 1e-6, _ws(T, H, E, k, I, shared))
    got = _layer(d, k, shared, rms, 1e-6, _ws(T, H, E, k, I, shared))
    _same(got, ref, "T=%d E=%d shared=%d rms=%d" % (T, E, shared, rms), exact_out=plan is not None and not rms)


@pytest.mark.parametrize("name", ["decode1", "decode4", "shared_decode1", "tiny"])
def test_layer_parity_with_oracle(name):
    wl = synth.WORKLOADS[name]
    T, H, E, k, I = wl.dims
    h = synth.shared_layer_inputs(wl) if wl.shared else synth.layer_inputs(wl)
    d = {key: (v.cuda() if v is not None else None) for key, v in h.items()}
    out, ids, w = _layer(d, k, wl.shared, False, 0.0, _ws(T, H, E, k, I, wl.shared))
    # the routed slots against the oracle's logits over the first E rows
    logits = oracle.router_logits(h["hidden"], h["router_w"][:E], h["bias"])
    check_route(ids[:, :k], w[:, :k], logits, k)
    ids_h, w_h = ids.cpu().numpy(), w.cpu().numpy()
    if wl.shared:
        assert (ids_h[:, k] == E).all()
        gate = oracle.router_logits(h["hidden"], h["router_w"][E:E + 1], None)[:, 0]
        assert np.abs(w_h[:, k] - 1.0 / (1.0 + np.exp(-gate))).max() <= 2e-5
    Ef = E + (1 if wl.shared else 0)
    ref = oracle.expert_forward(h["hidden"], ids_h, w_h, h["w1_packed"], h["w1_scales"], h["w2_packed"],
                                h["w2_scales"], Ef, I)
    assert_close(out.float().cpu().numpy(), ref, name)


def test_layer_repeated_calls_one_workspace():
    # the grid barrier's count resets itself: calls in a row on one workspace,
    # with new inputs each time and a change of batch between them
    H, E, k, I = 2560, 512, 10, 640
    ws = moe.workspace(8, H, E, k, I)
    wts = synth.expert_weights(E, H, I, seed=5)
    wd = {key: v.cuda() for key, v in wts.items()}
    wr = synth.router(E, H, seed=5).cuda()
    for rep, T in enumerate([1, 2, 8, 3, 1, 2]):
        d = dict(wd, hidden=synth.hidden(T, H, seed=30 + rep).cuda(), router_w=wr, bias=None)
        ref = _separate(d, k, False, False, 0.0, moe.workspace(T, H, E, k, I))
        got = _layer(d, k, False, False, 0.0, ws)
        _same(got, ref, "call %d (T=%d)" % (rep, T))


def test_layer_stack_chained():
    # a decode stack step: each layer's `next` is the following layer's input,
    # read by a kernel launched (programmatically) right behind the one that
    # writes it; four layers with their own weights (64 experts, to keep the
    # host's drawing short), against the separate calls
    T, H, E, k, I = 2, 2560, 64, 8, 640
    assert moe.moe_forward_plan(T, H, E, k, I)[3]
    ws_a, ws_b = moe.workspace(T, H, E, k, I), moe.workspace(T, H, E, k, I)
    x_a = x_b = synth.hidden(T, H, seed=1).cuda()
    outs_a, outs_b = [], []
    layers = []
    for li in range(4):
        wts = synth.expert_weights(E, H, I, seed=1, layer=li)
        layers.append(dict({key: v.cuda() for key, v in wts.items()}, router_w=synth.router(E, H, seed=1, layer=li).cuda(),
                           bias=None))
    for li in range(4):
        d = dict(layers[li], hidden=x_a)
        out, ids, w = moe.moe_layer_forward(x_a, d["router_w"], k, *_weights(d), rms=True, eps=1e-6, ws=ws_a)
        outs_a.append((out, ids, w))
        x_a = out
    for li in range(4):
        d = dict(layers[li], hidden=x_b)
        ids, w = moe.moe_route(x_b, d["router_w"], k, ws=ws_b)
        out = moe.moe_w4a16_forward_rms(x_b, ids, w, *_weights(d), eps=1e-6, ws=ws_b)
        outs_b.append((out, ids, w))
        x_b = out
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws_a) == 0 and moe.moe_check_device_error(ws_b) == 0
    for li in range(4):
        # (the RMS scale sums the blocks' shares in arrival order: outputs within a bf16 rounding)
        _same(outs_a[li], outs_b[li], "layer %d" % li, exact_out=False)


def test_workspace_shared_across_batch_sizes():
    # the regions that must be zero when a call starts sit at offsets that
    # depend on no dimension (and the prefill accumulator is cleared by each
    # call), so one workspace serves calls of any batch in any order
    H, E, k, I = 1024, 64, 8, 256
    sizes = [600, 512, 4, 1, 700, 8, 3]
    ws = torch.zeros(max(moe.moe_workspace_size(T, H, E, k, I) for T in sizes), dtype=torch.uint8, device="cuda")
    wd = {key: v.cuda() for key, v in synth.expert_weights(E, H, I, seed=9).items()}
    wr = synth.router(E, H, seed=9).cuda()
    for i, T in enumerate(sizes):
        x = synth.hidden(T, H, seed=60 + i).cuda()
        ids, w = moe.moe_route(x, wr, k, ws=ws)
        out = moe.moe_w4a16_forward(x, ids, w, *_weights(wd), ws=ws)
        fresh = moe.moe_w4a16_forward(x, ids, w, *_weights(wd), ws=moe.workspace(T, H, E, k, I))
        torch.cuda.synchronize()
        assert moe.moe_check_device_error(ws) == 0
        if T <= 8:
            assert torch.equal(out, fresh), "T=%d" % T
        else:
            # prefill sums in arrival order: within a bf16 rounding of the fresh call
            a, b = out.float(), fresh.float()
            assert (a - b).abs().max().item() <= 2.0 ** -7 * b.abs().max().item(), "T=%d" % T
        if T <= 8:
            got = _layer(dict(wd, hidden=x, router_w=wr, bias=None), k, False, False, 0.0, ws)
            _same(got, (fresh, ids, w), "layer T=%d" % T)
