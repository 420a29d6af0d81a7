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


# ---------------------------------------------------------- shared expert ----
# "vLLM Optimization Edition" 3.3 "MoE block": the shared expert's gate is one
# more row of the router GEMV, and the layer's output is routed + sigmoid(gate)
# x shared.

def _shared_tiny(seed=0):
    wl = synth.WORKLOADS["tiny"]
    T, H, E, k, I = wl.dims
    d = synth.shared_layer_inputs(wl, seed=seed)
    return wl, d


def test_shared_gate_and_expert_equal_library_forms():
    wl, d = _shared_tiny(seed=20)
    T, H, E, k, I = wl.dims
    wg = d["router_w"][E]
    gate, y = oracle.shared_expert(d["hidden"], wg, d["w1_packed"][E], d["w1_scales"][E],
                                   d["w2_packed"][E], d["w2_scales"][E], I)
    x = _f64(d["hidden"])
    assert np.allclose(gate, x @ _f64(wg), rtol=0, atol=1e-12)
    W1 = _dense_numpy(d["w1_packed"][E], d["w1_scales"][E])
    W2 = _dense_numpy(d["w2_packed"][E], d["w2_scales"][E])
    g, u = x @ W1[:I].T, x @ W1[I:].T
    ref = (g * expit(g) * u) @ W2.T
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max()


def test_shared_combine_closed_forms():
    g = np.random.default_rng(21)
    routed, y = g.standard_normal((3, 256)), g.standard_normal((3, 256))
    # sigmoid(0) = 1/2 exactly
    out = oracle.shared_combine(routed, np.zeros(3), y)
    assert np.array_equal(out, routed + 0.5 * y)
    # a gate far below zero leaves the routed output; far above, adds all of the shared one
    assert np.allclose(oracle.shared_combine(routed, np.full(3, -800.0), y), routed, rtol=0, atol=0)
    assert np.allclose(oracle.shared_combine(routed, np.full(3, 800.0), y), routed + y, rtol=0, atol=1e-15)
    gate = np.array([-1.0, 0.3, 2.0])
    ref = routed + y / (1.0 + np.exp(-gate))[:, None]
    assert np.allclose(oracle.shared_combine(routed, gate, y), ref, rtol=0, atol=1e-14)


def test_shared_expert_is_one_more_expert_with_weight_sigmoid_gate():
    """routed + sigmoid(g) * shared equals the routed-expert sum over k + 1 slots
    whose last slot is the shared expert (index E) with weight sigmoid(g)."""
    wl, d = _shared_tiny(seed=22)
    T, H, E, k, I = wl.dims
    logits = oracle.router_logits(d["hidden"], d["router_w"][:E])
    ids, w = oracle.topk_softmax(logits, k)
    W = (d["w1_packed"], d["w1_scales"], d["w2_packed"], d["w2_scales"])
    routed = oracle.expert_forward(d["hidden"], ids, w.astype(np.float32), *W, E + 1, I)
    gate, y = oracle.shared_expert(d["hidden"], d["router_w"][E], *(t[E] for t in W), I)
    layer = oracle.shared_combine(routed, gate, y)
    sg = (1.0 / (1.0 + np.exp(-gate))).astype(np.float32)
    ids1 = np.concatenate([ids, np.full((T, 1), E, np.int32)], axis=1)
    w1 = np.concatenate([w.astype(np.float32), sg[:, None]], axis=1)
    one = oracle.expert_forward(d["hidden"], ids1, w1, *W, E + 1, I)
    # the only difference: the gate weight passes through float32 in the slot form
    assert np.abs(one - layer).max() <= 1e-6 * np.abs(layer).max()
    # the router's first E rows are those of the layer without a shared expert
    assert torch.equal(d["router_w"][:E], synth.router(E, H, seed=22))


# -------------------------------------------------------------- quantiser ----
# "vLLM Optimization Edition" 7 "Putting MTP on the GPU": RTN, g128,
# symmetric, with a per-group search for the clip that minimises squared error.

def _bf16_tensor(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16)


def test_quantize_exactly_representable_group():
    # w = q0 * 2^-6 with q0 in [-7, 7] reaching 7: the unclipped scale is 2^-6
    # exactly, every value is hit, and no other candidate has zero error
    g = np.random.default_rng(30)
    q0 = g.integers(-7, 8, (3, 256))
    q0[:, 5] = 7
    q0[:, 133] = -7
    w = _bf16_tensor(q0 * 2.0 ** -6)
    packed, scales, choice, err = oracle.quantize_int4(w, 50)
    assert (choice == 0).all() and (err[:, :, 0] == 0).all()
    assert np.array_equal(_f64(torch.from_numpy(scales.view(np.int16)).view(torch.bfloat16)),
                          np.full((3, 2), 2.0 ** -6))
    assert np.array_equal(oracle.unpack_int4(packed, 3, 256), q0)


def test_quantize_single_candidate_is_plain_round_to_nearest():
    # nclip = 1 (no search): s = bf16(amax / 7), q = clip(round_half_even(w / s), -8, 7)
    w = synth.bf16_weights(16, 512, seed=31)
    packed, scales, choice, _ = oracle.quantize_int4(w, 1)
    wf = w.float().numpy().reshape(16, 4, 128)
    amax = np.abs(wf).max(axis=2)
    s = torch.from_numpy((amax / np.float32(7.0)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    q = np.clip(np.round(wf / s[:, :, None]), -8, 7).astype(np.int64).reshape(16, 512)
    assert np.array_equal(oracle.unpack_int4(packed, 16, 512), q)
    assert np.array_equal(scales, _bits(torch.from_numpy(s).to(torch.bfloat16)))
    assert (choice == 0).all()


def test_quantize_choice_minimises_the_error_of_its_own_output():
    w = synth.bf16_weights(32, 384, seed=32)
    packed, scales, choice, err = oracle.quantize_int4(w, 50)
    # the choice is the first minimum of the candidates' errors
    assert np.array_equal(choice, err.argmin(axis=2))
    # the packed output, dequantised by a separate routine, has exactly that error
    W = oracle.dequant(packed, torch.from_numpy(scales.view(np.int16)).view(torch.bfloat16), 32, 384)
    e = ((_f64(w) - W) ** 2).reshape(32, 3, 128).sum(axis=2)
    assert np.allclose(e, err.min(axis=2), rtol=1e-12, atol=0)
    # a search over more candidates never does worse than plain rounding
    _, _, _, err1 = oracle.quantize_int4(w, 1)
    assert (err.min(axis=2) <= err1[:, :, 0]).all()
    assert (err.min(axis=2) < err1[:, :, 0]).mean() > 0.5


def test_quantize_power_of_two_scaling_and_zero_groups():
    w = synth.bf16_weights(8, 256, seed=33)
    a = oracle.quantize_int4(w, 50)
    b = oracle.quantize_int4((w.float() * 8.0).to(torch.bfloat16), 50)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    sa = torch.from_numpy(a[1].view(np.int16)).view(torch.bfloat16).float()
    sb = torch.from_numpy(b[1].view(np.int16)).view(torch.bfloat16).float()
    assert torch.equal(sb, sa * 8.0)
    # an all-zero group stores scale 0 and the nibble of q = 0 (8) everywhere
    z = torch.zeros(2, 128, dtype=torch.bfloat16)
    p, s, c, e = oracle.quantize_int4(z, 50)
    assert (p.view(np.uint32) == 0x88888888).all() and (s == 0).all() and (e == 0).all()


def test_quantize_single_outlier_closed_form():
    # one value 7 * 2^-3 and 127 zeros: the unclipped scale 2^-3 gives q = 7 and zero error
    v = np.zeros((1, 128), np.float32)
    v[0, 77] = 7 * 2.0 ** -3
    p, s, c, e = oracle.quantize_int4(_bf16_tensor(v), 50)
    assert c[0, 0] == 0 and e[0, 0, 0] == 0
    q = oracle.unpack_int4(p, 1, 128)
    assert q[0, 77] == 7 and not np.delete(q[0], 77).any()
    # the last candidate, c = 0.51: 0.51 * 0.875 / 7 = 0.06375 = 2^-4 * 1.02, and
    # 1.02 * 128 = 130.56 rounds to 131, so the bf16 scale is 2^-4 * 131/128 =
    # 0.06396484375; 0.875 / 0.06396484375 = 13.7 saturates q at 7, leaving
    # (0.875 - 7 * 0.06396484375)^2 = 0.42724609375^2
    assert e[0, 0, 49] == 0.42724609375 ** 2


# ------------------------------------------------------------------- W8A16 ----
# "vLLM Optimization Edition" 3.3 "Hyper-connection (decode-04)": INT8
# pack-quantized puts four values in each int32 word, least significant byte
# first, stored as value + 128, so the words viewed as bytes already are
# q + 128 as [N, K]; model card "What is quantized", groups C (gs64) and D (gs128).

def _golden_int8():
    rows = []
    for line in open(os.path.join(GOLDEN, "int8_pack.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        rows.append(([int(v) for v in lhs.split()], int(rhs, 16)))
    return rows


def test_int8_pack_matches_hand_worked_words():
    for q, word in _golden_int8():
        packed = oracle.pack_int8(np.array([q], np.int16))
        assert int(packed.view(np.uint32)[0, 0]) == word
        assert oracle.unpack_int8(packed, 1, 4).tolist() == [q]


def test_int8_words_viewed_as_bytes_are_q_plus_128():
    # the pages' observation: weight_packed.view(uint8) already is q + 128 as [N, K]
    w = synth.int8_weights(7, 256, 64, seed=40)["w_packed"].numpy()
    q = oracle.unpack_int8(w, 7, 256)
    assert np.array_equal(w.view(np.uint8).reshape(7, 256).astype(np.int16) - 128, q)
    assert np.array_equal(oracle.pack_int8(q), w)
    with pytest.raises(ValueError):
        oracle.pack_int8(np.full((1, 4), 128, np.int16))


@pytest.mark.parametrize("gs", [64, 128])
def test_w8a16_linear_equals_library_matmul(gs):
    T, N, K = 5, 24, 512
    d = synth.int8_weights(N, K, gs, seed=41)
    x = synth.hidden(T, K, seed=41)
    y = oracle.w8a16_linear(x, d["w_packed"], d["scales"], gs)
    q = d["w_packed"].numpy().view(np.uint8).reshape(N, K).astype(np.float64) - 128
    W = q * np.repeat(_f64(d["scales"]), gs, axis=1)
    assert np.allclose(y, _f64(x) @ W.T, rtol=0, atol=1e-12 * np.abs(y).max())


def test_w8a16_group_index_and_closed_form():
    # all bytes 0x81 (q = 1): y = x . (scale per group), so the group index c // gs shows
    N, K = 2, 256
    words = np.full((N, K // 4), 0x81818181, np.uint32).view(np.int32)
    for gs in (64, 128):
        sc = torch.tensor([[1.0, 2.0, 4.0, 8.0][: K // gs], [0.5, -1.0, 0.25, 3.0][: K // gs]], dtype=torch.bfloat16)
        x = synth.hidden(3, K, seed=42)
        y = oracle.w8a16_linear(x, words, sc, gs)
        xg = _f64(x).reshape(3, K // gs, gs).sum(axis=2)
        assert np.allclose(y, xg @ _f64(sc).T, rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.w8a16_linear(x, words, sc, 32)
