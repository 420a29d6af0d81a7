"""Parity of the W8A16 linear layer with the fp64 oracle, on the GPU.

"vLLM Optimization Edition", section 3.3 "Hyper-connection (decode-04)": INT8
pack-quantized weights (q + 128, four per int32 word, least significant byte
first) read as stored, with a bf16 scale per 64 (group C: the hyper-connection
mixers [320, 10240] and [10240, 320]) or 128 (group D: lm_head [248320, 2560])
values. The bar is the layer's: max|gpu - oracle| <= 1e-2 * max|oracle|, with
fp32 accumulation; the dequantisation itself is exact, checked bit for bit
through weights whose products are exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a16_mixture_experts_gb300 as moe

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.lib()


def _check(T, N, K, gs, seed):
    d = synth.int8_weights(N, K, gs, seed=seed)
    x = synth.hidden(T, K, seed=seed)
    y = moe.moe_w8a16_linear(x.cuda(), d["w_packed"].cuda(), d["scales"].cuda(), gs).float().cpu().numpy()
    ref = oracle.w8a16_linear(x, d["w_packed"], d["scales"], gs)
    err = np.abs(y - ref).max()
    assert err <= OUT_TOL * np.abs(ref).max(), "T=%d N=%d K=%d gs=%d: %g vs %g" % (T, N, K, gs, err, np.abs(ref).max())
    return y, ref


@pytest.mark.parametrize("T,N,K,gs", [
    (1, 4096, 2560, 128),     # lm_head rows, one token
    (4, 320, 10240, 64),      # hyper-connection down mixer
    (3, 10240, 320, 64),      # hyper-connection up mixer (K = 5 groups)
    (8, 257, 512, 128),       # ragged rows, the largest decode batch
    (7, 100, 1024, 64),       # ragged rows, odd batch
    (2, 16, 64, 64),          # smallest
])
def test_w8a16_gemv_parity(T, N, K, gs):
    _check(T, N, K, gs, seed=T * 1000 + N + K)


def test_w8a16_lm_head_full_shape():
    # the whole lm_head of the model: 248320 x 2560, INT8 gs128, one decode token
    _check(1, 248320, 2560, 128, seed=9)


def test_w8a16_exact_products():
    # bytes chosen so that every product and partial sum is exact in fp32:
    # q in {-2, .., 2}, x in {-1, 0, 1}, scale 1: the result is an integer
    N, K, T = 64, 256, 5
    g = np.random.default_rng(3)
    q = g.integers(-2, 3, (N, K)).astype(np.int16)
    w = oracle.pack_int8(q)
    sc = torch.ones(N, K // 64, dtype=torch.bfloat16)
    x = torch.from_numpy(g.integers(-1, 2, (T, K)).astype(np.float32)).to(torch.bfloat16)
    y = moe.moe_w8a16_linear(x.cuda(), torch.from_numpy(w).cuda(), sc.cuda(), 64).float().cpu().numpy()
    ref = x.double().numpy() @ q.astype(np.float64).T
    assert np.array_equal(y, ref)


def test_w8a16_every_byte_value():
    # one row per byte value b (q = b - 128) against x = 1: y = q * scale * K exactly
    K = 64
    q = np.repeat(np.arange(-128, 128, dtype=np.int16)[:, None], K, axis=1)
    w = oracle.pack_int8(q)
    sc = torch.full((256, 1), 0.5, dtype=torch.bfloat16)
    x = torch.ones(1, K, dtype=torch.bfloat16)
    y = moe.moe_w8a16_linear(x.cuda(), torch.from_numpy(w).cuda(), sc.cuda(), 64).float().cpu().numpy()
    assert np.array_equal(y[0], np.arange(-128, 128) * 0.5 * K)


@pytest.mark.parametrize("T,N,K,gs", [
    (512, 320, 10240, 64),    # the pages' batch: hyper-connection down mixer at 512 tokens (split over K)
    (512, 10240, 320, 64),    # up mixer: K = 320, the last 128-wide stage half full
    (9, 1000, 2560, 128),     # just above the GEMV, ragged rows
    (300, 2048, 2560, 128),   # lm_head rows, ragged token chunk
    (129, 130, 256, 64),      # one token past a chunk, two rows past a block
])
def test_w8a16_gemm_parity(T, N, K, gs):
    ws = torch.zeros(moe.moe_w8a16_workspace_size(T, N, K, gs), dtype=torch.uint8, device="cuda")
    d = synth.int8_weights(N, K, gs, seed=T + N + K)
    x = synth.hidden(T, K, seed=T + N + K)
    y = moe.moe_w8a16_linear(x.cuda(), d["w_packed"].cuda(), d["scales"].cuda(), gs, ws=ws).float().cpu().numpy()
    assert moe.moe_check_device_error(ws) == 0
    ref = oracle.w8a16_linear(x, d["w_packed"], d["scales"], gs)
    err = np.abs(y - ref).max()
    assert err <= OUT_TOL * np.abs(ref).max(), "T=%d N=%d K=%d gs=%d: %g vs %g" % (T, N, K, gs, err, np.abs(ref).max())


def test_w8a16_gemm_matches_gemv_rows():
    # the two paths agree on the same rows (a 9-token batch against its first 8 tokens)
    N, K, gs = 512, 1024, 128
    d = synth.int8_weights(N, K, gs, seed=77)
    x = synth.hidden(9, K, seed=77).cuda()
    W = (d["w_packed"].cuda(), d["scales"].cuda())
    a = moe.moe_w8a16_linear(x, *W, gs)
    b = moe.moe_w8a16_linear(x[:8].contiguous(), *W, gs)
    assert (a[:8].float() - b.float()).abs().max().item() <= OUT_TOL * b.float().abs().max().item()


def test_w8a16_empty_batch():
    w = torch.zeros(16, 16, dtype=torch.int32, device="cuda")
    s = torch.ones(16, 1, dtype=torch.bfloat16, device="cuda")
    y = moe.moe_w8a16_linear(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), w, s, 64)
    assert y.shape == (0, 16)


def test_w8a16_split_gemm_is_deterministic():
    # the splits over K are summed in a fixed order: two calls give the same bits
    T, N, K, gs = 256, 256, 8192, 64
    assert moe.moe_w8a16_workspace_size(T, N, K, gs) > 256, "this shape should split over K"
    d = synth.int8_weights(N, K, gs, seed=5)
    x = synth.hidden(T, K, seed=5).cuda()
    W = (d["w_packed"].cuda(), d["scales"].cuda())
    a = moe.moe_w8a16_linear(x, *W, gs)
    b = moe.moe_w8a16_linear(x, *W, gs)
    assert torch.equal(a, b)
    ref = oracle.w8a16_linear(x.cpu(), d["w_packed"], d["scales"], gs)
    assert np.abs(a.float().cpu().numpy() - ref).max() <= OUT_TOL * np.abs(ref).max()
