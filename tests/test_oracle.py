"""Pins of the fp64 oracle against facts it does not compute itself.

Each test checks the oracle against something other than its own formula:
hand-worked storage words, byte totals printed on the pages, closed forms,
library routines (numpy matmul, argsort, scipy's logistic), brute force over
all experts, and invariants that a dropped term, a wrong sign or index, or a
transposed operand would break.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- storage ----

def _golden_pack():
    rows = []
    for line in open(os.path.join(GOLDEN, "int4_pack.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        rows.append(([int(v) for v in lhs.split()], int(rhs, 16)))
    return rows


def test_pack_matches_hand_worked_words():
    for q, word in _golden_pack():
        packed = oracle.pack_int4(np.array([q], np.int8))
        assert int(packed.view(np.uint32)[0, 0]) == word
        assert oracle.unpack_int4(packed, 1, 8).tolist() == [q]


def test_pack_unpack_round_trip_random():
    g = np.random.default_rng(1)
    words = g.integers(0, 2**32, (37, 48), dtype=np.uint32).view(np.int32)
    q = oracle.unpack_int4(words, 37, 384)
    assert q.min() == -8 and q.max() == 7
    assert np.array_equal(oracle.pack_int4(q), words)
    with pytest.raises(ValueError):
        oracle.pack_int4(np.full((1, 8), 8, np.int8))


def test_dequant_closed_form():
    # word 0xfedcba98 holds q = 0..7; scale 0.5 -> 0, 0.5, ..., 3.5 (exact)
    K = 128
    words = np.full((1, K // 8), 0xFEDCBA98, np.uint32).view(np.int32)
    scale = torch.tensor([[0.5]], dtype=torch.bfloat16)
    W = oracle.dequant(words, scale, 1, K)
    assert np.array_equal(W[0, :8], np.arange(8) * 0.5)
    # two groups with different scales: group index is c // 128
    K = 256
    words = np.full((1, K // 8), 0x76543210, np.uint32).view(np.int32)  # q = -8..-1
    scale = torch.tensor([[0.25, -2.0]], dtype=torch.bfloat16)
    W = oracle.dequant(words, scale, 1, K)
    q = np.tile(np.arange(-8, 0), K // 8)
    assert np.array_equal(W[0, :128], q[:128] * 0.25)
    assert np.array_equal(W[0, 128:], q[128:] * -2.0)


def test_byte_totals_match_the_pages():
    """Per-expert and per-model sizes of INT4 gs128 with bf16 scales.

    "vLLM Optimization Edition" 4.2: top-10 x 2.46 MB per token-row;
    model card "What is quantized": group A = 58.0 GiB;
    "vLLM Edition" 2: routed experts 120.8B parameters;
    "vLLM Edition" 5.6: 1.22 GB of expert reads per decoded token.
    """
    H, E, I, L, k = 2560, 512, 640, 48, 10
    w = synth.expert_weights(E, H, I, seed=0, layer=0, experts=[3])
    payload = w["w1_packed"][0].numel() * 4 + w["w2_packed"][0].numel() * 4
    scales = w["w1_scales"][0].numel() * 2 + w["w2_scales"][0].numel() * 2
    assert payload == 2_457_600 and round(payload / 1e6, 2) == 2.46
    assert payload + scales == 2_534_400
    assert round((payload + scales) * E * L / 2**30, 1) == 58.0
    assert round(3 * H * I * E * L / 1e9, 1) == 120.8
    assert round(k * L * (payload + scales) / 1e9, 2) == 1.22


# ---------------------------------------------------------------- routing ----

def test_logits_equal_library_matmul():
    x, wr = synth.hidden(5, 256, seed=2), synth.router(16, 256, seed=2)
    bias = synth.zipf_bias(16, 1.1, seed=2)
    ref = _f64(x) @ _f64(wr).T + bias.numpy().astype(np.float64)
    assert np.allclose(oracle.router_logits(x, wr, bias), ref, rtol=0, atol=1e-12)
    assert np.allclose(oracle.router_logits(x, wr), _f64(x) @ _f64(wr).T, rtol=0, atol=1e-12)


def test_topk_brute_force_sort_and_weights():
    g = np.random.default_rng(3)
    T, E, k = 64, 16, 4
    logits = g.standard_normal((T, E))
    ids, w = oracle.topk_softmax(logits, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))      # by logit desc, then id asc
        assert ids[t].tolist() == order[:k].tolist()
        # renormalised full softmax == softmax over the selected logits
        # ("vLLM Optimization Edition" 3.3: with norm_topk_prob the full
        # denominator cancels)
        sel = logits[t, order[:k]]
        soft_sel = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w[t], soft_sel, rtol=0, atol=1e-14)
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(w[t]) <= 0)


def test_topk_ties_go_to_lower_id():
    # "vLLM Optimization Edition" 3.3: ties go to the lower expert id
    logits = np.array([[0.0, 2.0, 1.0, 2.0, 1.0, 2.0, -1.0, 1.0]])
    ids, w = oracle.topk_softmax(logits, 4)
    assert ids[0].tolist() == [1, 3, 5, 2]
    assert np.allclose(w[0], [math.exp(2) / (3 * math.exp(2) + math.exp(1))] * 3
                       + [math.exp(1) / (3 * math.exp(2) + math.exp(1))], atol=1e-15)
    ids, _ = oracle.topk_softmax(np.zeros((1, 6)), 3)
    assert ids[0].tolist() == [0, 1, 2]


def test_topk_shift_invariance():
    g = np.random.default_rng(4)
    logits = g.standard_normal((8, 32))
    a = oracle.topk_softmax(logits, 5)
    b = oracle.topk_softmax(logits + 123.0, 5)
    assert np.array_equal(a[0], b[0]) and np.allclose(a[1], b[1], atol=1e-13)


# ---------------------------------------------------------------- permute ----

def test_permute_brute_force():
    g = np.random.default_rng(5)
    for T, k, E in [(1, 1, 1), (4, 2, 16), (33, 5, 64), (7, 3, 1024)]:
        ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        offsets, perm = oracle.permute(ids, E)
        counts = np.bincount(ids.ravel(), minlength=E)
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(perm, np.argsort(ids.ravel(), kind="stable"))
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 16]], np.int32), 16)


# ---------------------------------------------------------------- experts ----

def _dense_numpy(packed: torch.Tensor, scales: torch.Tensor) -> np.ndarray:
    """Dequantise with numpy bit operations, written apart from the oracle."""
    w = packed.numpy().view(np.uint32)
    shifts = np.arange(8, dtype=np.uint32) * 4
    q = ((w[..., None] >> shifts) & 0xF).astype(np.int64) - 8
    q = q.reshape(*w.shape[:-1], w.shape[-1] * 8)
    s = np.repeat(_f64(scales), 128, axis=-1)
    return q * s


def _tiny_inputs(seed=0):
    wl = synth.WORKLOADS["tiny"]
    T, H, E, k, I = wl.dims
    d = synth.layer_inputs(wl, seed=seed)
    ids, w, _ = oracle.route(d["hidden"], d["router_w"], k)
    return wl, d, ids, w.astype(np.float32)


def test_experts_equal_dense_masked_loop_over_all_experts():
    """Brute force: every expert applied to every token, masked by w or 0."""
    wl, d, ids, w = _tiny_inputs()
    T, H, E, k, I = wl.dims
    out = oracle.expert_forward(d["hidden"], ids, w, d["w1_packed"], d["w1_scales"],
                                d["w2_packed"], d["w2_scales"], E, I)
    W1 = _dense_numpy(d["w1_packed"], d["w1_scales"])   # [E, 2I, H]
    W2 = _dense_numpy(d["w2_packed"], d["w2_scales"])   # [E, H, I]
    x = _f64(d["hidden"])
    mask = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            mask[t, ids[t, j]] = w[t, j]
    ref = np.zeros((T, H))
    for e in range(E):
        gu = x @ W1[e].T
        h = gu[:, :I] * expit(gu[:, :I]) * gu[:, I:]
        ref += mask[:, e:e + 1] * (h @ W2[e].T)
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_single_forced_expert_is_dense_swiglu_mlp():
    wl = synth.WORKLOADS["tiny"]
    T, H, E, k, I = wl.dims
    d = synth.layer_inputs(wl, seed=7)
    x = _f64(d["hidden"])
    for e in (0, 5, E - 1):
        ids = np.full((T, 1), e, np.int32)
        w = np.ones((T, 1), np.float32)
        out = oracle.expert_forward(d["hidden"], ids, w, d["w1_packed"], d["w1_scales"],
                                    d["w2_packed"], d["w2_scales"], E, I)
        W1 = _dense_numpy(d["w1_packed"][e], d["w1_scales"][e])
        W2 = _dense_numpy(d["w2_packed"][e], d["w2_scales"][e])
        g, u = x @ W1[:I].T, x @ W1[I:].T
        ref = (g * expit(g) * u) @ W2.T
        assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_doubling_down_scales_doubles_output_exactly():
    wl, d, ids, w = _tiny_inputs(seed=8)
    T, H, E, k, I = wl.dims
    args = (d["hidden"], ids, w, d["w1_packed"], d["w1_scales"], d["w2_packed"])
    a = oracle.expert_forward(*args, d["w2_scales"], E, I)
    b = oracle.expert_forward(*args, (d["w2_scales"].float() * 2).to(torch.bfloat16), E, I)
    assert np.array_equal(b, 2 * a)


def test_expert_relabelling_and_token_order():
    wl, d, ids, w = _tiny_inputs(seed=9)
    T, H, E, k, I = wl.dims
    base = oracle.expert_forward(d["hidden"], ids, w, d["w1_packed"], d["w1_scales"],
                                 d["w2_packed"], d["w2_scales"], E, I)
    pi = np.random.default_rng(9).permutation(E)              # new label of expert e
    inv = np.argsort(pi)
    rel = {key: d[key][torch.from_numpy(inv)] for key in ("w1_packed", "w1_scales", "w2_packed", "w2_scales")}
    out = oracle.expert_forward(d["hidden"], pi[ids].astype(np.int32), w, rel["w1_packed"],
                                rel["w1_scales"], rel["w2_packed"], rel["w2_scales"], E, I)
    assert np.allclose(out, base, rtol=0, atol=1e-13)
    # slot order within a token does not matter; token order permutes rows
    rev = oracle.expert_forward(d["hidden"].flip(0), ids[::-1, ::-1], w[::-1, ::-1],
                                d["w1_packed"], d["w1_scales"], d["w2_packed"], d["w2_scales"], E, I)
    assert np.allclose(rev[::-1], base, rtol=0, atol=1e-13)
    # a subset of held experts gives the same result
    held = np.unique(ids)
    row = np.full(E, -1, np.int32)
    row[held] = np.arange(len(held))
    sub = synth.expert_weights(E, H, I, seed=9, experts=held)
    part = oracle.expert_forward(d["hidden"], ids, w, sub["w1_packed"], sub["w1_scales"],
                                 sub["w2_packed"], sub["w2_scales"], E, I, expert_row=row)
    assert np.array_equal(part, base)


def test_zero_weight_and_zero_input():
    wl, d, ids, w = _tiny_inputs(seed=10)
    T, H, E, k, I = wl.dims
    W = (d["w1_packed"], d["w1_scales"], d["w2_packed"], d["w2_scales"])
    zero_w = np.zeros_like(w)
    assert not oracle.expert_forward(d["hidden"], ids, zero_w, *W, E, I).any()
    zero_x = torch.zeros_like(d["hidden"])
    assert not oracle.expert_forward(zero_x, ids, w, *W, E, I).any()
    # linear in the routing weights
    w2 = w.copy()
    w2[:, 1] = 0
    a = oracle.expert_forward(d["hidden"], ids, w2, *W, E, I)
    w3 = w - w2
    b = oracle.expert_forward(d["hidden"], ids, w3, *W, E, I)
    c = oracle.expert_forward(d["hidden"], ids, w, *W, E, I)
    assert np.allclose(a + b, c, rtol=0, atol=1e-12 * np.abs(c).max())


# ------------------------------------------------------------------ stack ----

def test_round_bf16_matches_torch():
    g = np.random.default_rng(11)
    v = np.concatenate([g.standard_normal(10000) * 10.0 ** g.integers(-6, 6, 10000),
                        [0.0, -0.0, 1.0, 1 + 2**-8, 1 + 3 * 2**-8, 65504.0, 1e-40]])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(oracle.round_bf16(v), _bits(ref))


def test_residual_rms_closed_form():
    T, H = 3, 256
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    out = np.zeros((T, H))
    out[0] = 3.0
    out[1, ::2], out[1, 1::2] = 2.0, -2.0
    out[2, 0] = 16.0
    nb, nf = oracle.residual_rms(x, out, eps=0.0)
    assert np.allclose(nf[0], 1.0, atol=1e-15)
    assert np.allclose(nf[1], np.where(np.arange(H) % 2 == 0, 1.0, -1.0), atol=1e-15)
    assert abs(nf[2, 0] - math.sqrt(H)) < 1e-12 and not nf[2, 1:].any()
    g = np.random.default_rng(12)
    xr = synth.hidden(4, 256, seed=12)
    o = g.standard_normal((4, 256)) * 5
    _, nf = oracle.residual_rms(xr, o, eps=1e-6)
    r = _f64(xr) + o
    assert np.allclose(np.sqrt((nf ** 2).mean(1)), np.sqrt((r ** 2).mean(1) / ((r ** 2).mean(1) + 1e-6)),
                       atol=1e-14)
