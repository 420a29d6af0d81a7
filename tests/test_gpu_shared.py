"""Parity of the shared-expert layer with the fp64 oracle, on the GPU.

The layer ("vLLM Optimization Edition", section 3.3 "MoE block (decode-05)"):
the router's extra row is the shared expert's gate, and the output is
routed + sigmoid(gate) * shared. moe_route_shared writes the gate as slot k
(expert E, weight sigmoid(gate)); moe_w4a16_forward over E + 1 experts and
k + 1 slots then computes the whole layer. The bars are those of the routed
layer: routed ids exact where the 10th-11th gap is at least 1e-3, weights
within 2e-5, outputs within 1e-2 * max|oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a16_mixture_experts_gb300 as moe

pytestmark = pytest.mark.gpu

GAP = 1e-3
W_TOL = 2e-5
OUT_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()


def check_routed(ids, w, logits, k):
    """Slots [0, k): a valid top-k within the gap, exact ids where the gap allows."""
    T, E = logits.shape
    for t in range(T):
        l = logits[t]
        order = np.lexsort((np.arange(E), -l))
        ls = l[order]
        got = ids[t, :k]
        assert len(set(got.tolist())) == k and got.min() >= 0 and got.max() < E
        assert l[got].min() >= ls[k - 1] - GAP
        if ls[k - 1] - ls[k] >= GAP:
            assert set(got.tolist()) == set(order[:k].tolist()), "token %d" % t
        sel = l[got]
        ref_w = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.abs(w[t, :k] - ref_w).max() <= W_TOL, "token %d" % t


def _layer(name, seed=0):
    wl = synth.WORKLOADS[name]
    h = synth.shared_layer_inputs(wl, seed=seed)
    return wl, h, {key: (v.cuda() if v is not None else None) for key, v in h.items()}


def _gpu_layer(wl, g, ws=None):
    T, H, E, k, I = wl.dims
    if ws is None:
        ws = moe.shared_workspace(T, H, E, k, I)
    ids, w = moe.moe_route_shared(g["hidden"], g["router_w"], k, bias=g["bias"], ws=ws)
    out = moe.moe_w4a16_forward(g["hidden"], ids, w, g["w1_packed"], g["w1_scales"], g["w2_packed"],
                                g["w2_scales"], ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    return ids.cpu().numpy(), w.cpu().numpy().astype(np.float64), out.float().cpu().numpy()


def _oracle_layer(wl, h, ids, w, rows):
    """routed (on the GPU's routing, an input here) + sigmoid(gate) * shared, fp64."""
    T, H, E, k, I = wl.dims
    x = h["hidden"][rows]
    W = (h["w1_packed"], h["w1_scales"], h["w2_packed"], h["w2_scales"])
    routed = oracle.expert_forward(x, ids[rows, :k], w[rows, :k].astype(np.float32), *W, E + 1, I)
    gate, y = oracle.shared_expert(x, h["router_w"][E], *(t[E] for t in W), I)
    return oracle.shared_combine(routed, gate, y), gate


@pytest.mark.parametrize("name,nrows", [("tiny", None), ("decode1", None), ("decode4", None), ("decode64", None),
                                        ("prefill512", 64)])
def test_shared_layer_parity(name, nrows):
    wl, h, g = _layer(name)
    T, H, E, k, I = wl.dims
    ids, w, out = _gpu_layer(wl, g)
    rows = np.arange(T) if nrows is None else np.sort(np.random.default_rng(3).choice(T, nrows, replace=False))
    logits = oracle.router_logits(h["hidden"][rows], h["router_w"][:E], h["bias"])
    check_routed(ids[rows], w[rows], logits, k)
    ref, gate = _oracle_layer(wl, h, ids, w, rows)
    # the gate slot: expert E with weight sigmoid(x . wg)
    assert (ids[:, k] == E).all()
    assert np.abs(w[rows, k] - 1.0 / (1.0 + np.exp(-gate))).max() <= W_TOL
    err = np.abs(out[rows] - ref).max()
    assert err <= OUT_TOL * np.abs(ref).max(), "%s: max err %g vs max|ref| %g" % (name, err, np.abs(ref).max())


def test_shared_gate_at_full_batch_sampled():
    # T = 4096: the tensor-core router, with the gate formed by the top-k kernel
    wl = synth.WORKLOADS["stack_prefill4096"]
    T, H, E, k, I = wl.dims
    x = synth.hidden(T, H, seed=5)
    wr = synth.router(E + 1, H, seed=5)
    ids, w = moe.moe_route_shared(x.cuda(), wr.cuda(), k)
    ids, w = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    rows = np.sort(np.random.default_rng(5).choice(T, 64, replace=False))
    check_routed(ids[rows], w[rows], oracle.router_logits(x[rows], wr[:E]), k)
    gate = oracle.router_logits(x[rows], wr[E:])[:, 0]
    assert (ids[:, k] == E).all()
    assert np.abs(w[rows, k] - 1.0 / (1.0 + np.exp(-gate))).max() <= W_TOL


@pytest.mark.parametrize("T", [1, 8, 9, 64])
def test_shared_routing_equals_plain_routing_plus_gate(T):
    # the routed slots of moe_route_shared are exactly those of moe_route over the first E rows
    H, E, k = 2560, 512, 10
    x = synth.hidden(T, H, seed=9).cuda()
    wr = synth.router(E + 1, H, seed=9).cuda()
    ids_s, w_s = moe.moe_route_shared(x, wr, k)
    ids_p, w_p = moe.moe_route(x, wr[:E].contiguous(), k)
    assert torch.equal(ids_s[:, :k], ids_p)
    assert torch.equal(w_s[:, :k], w_p)


def test_shared_gate_weight_zero_row_is_one_half():
    # a zero gate row: sigmoid(0) = 1/2 exactly, so the shared expert enters with weight 0.5
    wl, h, g = _layer("decode4", seed=2)
    T, H, E, k, I = wl.dims
    g["router_w"][E].zero_()
    ids, w = moe.moe_route_shared(g["hidden"], g["router_w"], k)
    assert (w[:, k] == 0.5).all()
