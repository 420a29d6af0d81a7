"""Parity of the on-device INT4 quantiser with the fp64 oracle.

The quantiser ("vLLM Optimization Edition", section 7 "Putting MTP on the
GPU": RTN, g128, symmetric, per-group clip search minimising squared error)
makes its scale and code decisions in fp32 on both sides, so for a given clip
candidate the codes and the scale are bit-exact. The choice of candidate
compares error sums, fp32 on the GPU and fp64 in the oracle: where the oracle's
best candidate beats the GPU's choice by more than the rounding of a 128-term
fp32 sum (2e-5 relative), the choice must be the oracle's, and then codes and
scale are compared bit for bit. Where the two candidates are closer than that,
the GPU's output must reach exactly the oracle's error of the candidate it chose.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a16_mixture_experts_gb300 as moe

pytestmark = pytest.mark.gpu

REL_GAP = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def check_quant(w, nclip):
    N, K = w.shape
    G = K // 128
    p_g, s_g, c_g = moe.moe_quantize_int4(w.cuda(), nclip, with_choice=True)
    p_g, s_g, c_g = p_g.cpu().numpy(), _bits(s_g), c_g.cpu().numpy()
    p_o, s_o, c_o, err = oracle.quantize_int4(w, nclip)
    same = c_g == c_o
    # where the choices agree: codes and scales bit-exact
    words = p_g.reshape(N, G, 16)
    assert np.array_equal(words[same], p_o.reshape(N, G, 16)[same])
    assert np.array_equal(s_g[same], s_o[same])
    if not same.all():
        n, g = np.nonzero(~same)
        e_best = err[n, g, c_o[n, g]]
        e_gpu = err[n, g, c_g[n, g]]
        assert (e_gpu - e_best <= REL_GAP * e_best).all(), "a clearly worse candidate was chosen"
        # the GPU's output has exactly the oracle's error of the candidate it chose
        W = oracle.dequant(p_g, torch.from_numpy(s_g.view(np.int16)).view(torch.bfloat16), N, K)
        e_out = ((w.double().numpy() - W) ** 2).reshape(N, G, 128).sum(axis=2)
        assert np.allclose(e_out[n, g], e_gpu, rtol=1e-12, atol=0)
    return same.mean()


@pytest.mark.parametrize("N,K,nclip", [(256, 2560, 50), (640, 640, 50), (33, 384, 17), (128, 1280, 100)])
def test_quantize_matches_oracle(N, K, nclip):
    w = synth.bf16_weights(N, K, seed=N + K)
    agree = check_quant(w, nclip)
    assert agree > 0.99


def test_quantize_plain_rtn_bit_exact():
    # one candidate: no search, nothing to disagree on
    w = synth.bf16_weights(300, 1024, seed=4)
    p_g, s_g = moe.moe_quantize_int4(w.cuda(), 1)
    p_o, s_o, _, _ = oracle.quantize_int4(w, 1)
    assert np.array_equal(p_g.cpu().numpy(), p_o)
    assert np.array_equal(_bits(s_g), s_o)


def test_quantize_special_groups():
    g = np.random.default_rng(5)
    rows = []
    q0 = g.integers(-7, 8, 128)
    q0[3] = 7
    rows.append(q0 * 2.0 ** -6)                 # exactly representable: c = 1 and zero error
    rows.append(np.zeros(128))                  # scale 0, q = 0
    z = np.zeros(128)
    z[77] = 0.875
    rows.append(z)                              # one value: q = 7 at scale 1/8
    rows.append(np.full(128, -3.0))             # constant negative group
    rows.append(g.standard_normal(128) * 1e-30)  # tiny values: scales far below 1
    w = torch.from_numpy(np.array(rows, np.float32)).to(torch.bfloat16)
    p_g, s_g, c_g = moe.moe_quantize_int4(w.cuda(), 50, with_choice=True)
    p_o, s_o, c_o, _ = oracle.quantize_int4(w, 50)
    assert np.array_equal(c_g.cpu().numpy(), c_o)
    assert np.array_equal(p_g.cpu().numpy(), p_o)
    assert np.array_equal(_bits(s_g), s_o)


def test_quantized_experts_run_through_the_layer():
    """Experts quantised on the device feed moe_w4a16_forward, which matches the
    oracle's forward on the oracle's quantisation of the same bf16 weights."""
    T, H, E, k, I = 4, 256, 8, 2, 128
    w1 = synth.bf16_weights(E * 2 * I, H, seed=6)
    w2 = synth.bf16_weights(E * H, I, seed=7)
    p1, s1 = moe.moe_quantize_int4(w1.cuda(), 50)
    p2, s2 = moe.moe_quantize_int4(w2.cuda(), 50)
    W = [p1.view(E, 2 * I, H // 8), s1.view(E, 2 * I, H // 128), p2.view(E, H, I // 8), s2.view(E, H, I // 128)]
    x = synth.hidden(T, H, seed=8)
    ids, tw = synth.random_topk(T, E, k, seed=8)
    out = moe.moe_w4a16_forward(x.cuda(), ids.cuda(), tw.cuda(), *W).float().cpu().numpy()
    o1 = oracle.quantize_int4(w1, 50)
    o2 = oracle.quantize_int4(w2, 50)
    bf = lambda s, shape: torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).reshape(shape)
    ref = oracle.expert_forward(x, ids, tw, o1[0].reshape(E, 2 * I, H // 8), bf(o1[1], (E, 2 * I, H // 128)),
                                o2[0].reshape(E, H, I // 8), bf(o2[1], (E, H, I // 128)), E, I)
    assert np.abs(out - ref).max() <= 1e-2 * np.abs(ref).max()
