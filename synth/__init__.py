"""Seeded synthetic inputs for the W4A16 routed-expert MoE layer.

This module only draws numbers. It holds none of the layer's arithmetic
(no routing, no dequantisation, no matmul), so both the CUDA library's
tests and the fp64 oracle can take their inputs from it.

Every tensor is drawn on the host from numpy's SFC64 generator, seeded by a
``SeedSequence`` of (seed, layer, tensor id[, expert]). Expert tensors get one
stream per expert, so any subset of experts can be regenerated bit for bit
without drawing the others, and the draws run in parallel threads.

Distributions follow the workloads of the pages ("Running 125B MoE on Three
3090s - vLLM Edition", section 1, model shape; the model card's "What is
quantized" table, group A = INT4 gs128 symmetric pack-quantized experts):

- hidden states ~ N(0, 1), rounded to bf16;
- router weight ~ N(0, std = 1/sqrt(H)), rounded to bf16 (the router stays
  BF16, model card "What is quantized");
- expert weights: each int32 word is 32 uniform random bits, i.e. eight
  nibbles uniform on [0, 15], which are the stored values q + 8 of signed
  int4 q uniform on [-8, 7];
- per-group scales: bf16(0.002 + 0.018 * u), u = m / 2**24 with m uniform
  on [0, 2**24), evaluated in float32 as one multiply then one add;
- skewed routing: a router bias of -s * ln(rank), rank = 1 + a seeded
  random permutation of the experts (Zipf with exponent s = 1.1);
- INT8 linear layers (W8A16): uniform bytes q + 128, bf16 scales
  0.0002 + 0.0018 u per group of 64 or 128 values.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

GROUP = 128  # quantisation group size along K

# tensor ids inside a SeedSequence
_T_HIDDEN, _T_ROUTER, _T_W1, _T_W1S, _T_W2, _T_W2S, _T_ZIPF, _T_TOPK, _T_QW, _T_W8, _T_W8S = range(11)


@dataclass(frozen=True)
class Dims:
    T: int   # tokens
    H: int   # hidden size
    E: int   # experts
    k: int   # experts per token
    I: int   # expert intermediate size

    def __iter__(self):
        return iter((self.T, self.H, self.E, self.k, self.I))


@dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    zipf: float | None = None   # exponent of the router-bias ranking, or None
    layers: int = 1
    shared: bool = False        # a shared expert beside the routed ones (router row E, expert E)


# The five workloads: tiny layer; one full-shape layer at decode T=1, 4, 64;
# a T=512 prefill chunk with Zipf-skewed routing; a 48-layer stack run on a
# T=4096 prefill and a T=4 decode.
FULL = dict(H=2560, E=512, k=10, I=640)
WORKLOADS = {
    "tiny": Workload("tiny", Dims(T=4, H=256, E=16, k=2, I=128)),
    "decode1": Workload("decode1", Dims(T=1, **FULL)),
    "decode4": Workload("decode4", Dims(T=4, **FULL)),
    "decode64": Workload("decode64", Dims(T=64, **FULL)),
    "prefill512": Workload("prefill512", Dims(T=512, **FULL), zipf=1.1),
    "stack_prefill4096": Workload("stack_prefill4096", Dims(T=4096, **FULL), layers=48),
    "stack_decode4": Workload("stack_decode4", Dims(T=4, **FULL), layers=48),
    # the layer with its shared expert (intermediate 640 like a routed one) at decode T = 1
    "shared_decode1": Workload("shared_decode1", Dims(T=1, **FULL), shared=True),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence(list(key))))


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _threads() -> int:
    return max(1, min(32, len(os.sched_getaffinity(0))))


def hidden(T: int, H: int, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """bf16 [T, H], N(0, 1)."""
    return _bf16(_rng(seed, layer, _T_HIDDEN).standard_normal((T, H), dtype=np.float32))


def router(E: int, H: int, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """bf16 [E, H], N(0, std = 1/sqrt(H))."""
    z = _rng(seed, layer, _T_ROUTER).standard_normal((E, H), dtype=np.float32)
    return _bf16(z * np.float32(1.0 / np.sqrt(H)))


def zipf_bias(E: int, s: float, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """f32 [E]: -s * ln(rank_e), rank = 1 + seeded permutation of the experts."""
    rank = _rng(seed, layer, _T_ZIPF).permutation(E).astype(np.float64) + 1.0
    return torch.from_numpy((-s * np.log(rank)).astype(np.float32))


def _words(key, n: int) -> np.ndarray:
    return _rng(*key).integers(0, 2**32, n, dtype=np.uint32).view(np.int32)


def _scales(key, n: int) -> np.ndarray:
    m = _rng(*key).integers(0, 2**24, n, dtype=np.int64).astype(np.float32)
    u = m * np.float32(1.0 / 2**24)
    return np.float32(0.002) + np.float32(0.018) * u


def expert_weights(E: int, H: int, I: int, seed: int = 0, layer: int = 0,
                   experts=None) -> dict:
    """Packed INT4 experts and their bf16 scales, on the host.

    Returns w1_packed int32 [n, 2I, H/8], w1_scales bf16 [n, 2I, H/128],
    w2_packed int32 [n, H, I/8], w2_scales bf16 [n, H, I/128] for the experts
    listed in ``experts`` (default: all E, in order). Rows [0, I) of w1 are the
    gate projection, rows [I, 2I) the up projection.
    """
    ids = list(range(E)) if experts is None else [int(e) for e in experts]
    n = len(ids)
    w1p = np.empty((n, 2 * I, H // 8), np.int32)
    w2p = np.empty((n, H, I // 8), np.int32)
    w1s = np.empty((n, 2 * I, H // GROUP), np.float32)
    w2s = np.empty((n, H, I // GROUP), np.float32)

    def fill(i: int) -> None:
        e = ids[i]
        w1p[i] = _words((seed, layer, _T_W1, e), w1p[i].size).reshape(w1p[i].shape)
        w2p[i] = _words((seed, layer, _T_W2, e), w2p[i].size).reshape(w2p[i].shape)
        w1s[i] = _scales((seed, layer, _T_W1S, e), w1s[i].size).reshape(w1s[i].shape)
        w2s[i] = _scales((seed, layer, _T_W2S, e), w2s[i].size).reshape(w2s[i].shape)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(n)))
    return {
        "w1_packed": torch.from_numpy(w1p),
        "w1_scales": _bf16(w1s),
        "w2_packed": torch.from_numpy(w2p),
        "w2_scales": _bf16(w2s),
    }


def random_topk(T: int, E: int, k: int, seed: int = 0, layer: int = 0):
    """Distinct random expert ids int32 [T, k] and positive weights f32 [T, k].

    Stand-in routing for driving the expert path on its own; the weights are
    U(0.05, 1) and are not normalised (the expert path takes them as given).
    """
    g = _rng(seed, layer, _T_TOPK)
    ids = np.stack([g.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = (np.float32(0.05) + np.float32(0.95) * g.random((T, k), dtype=np.float32))
    return torch.from_numpy(ids.reshape(T, k)), torch.from_numpy(w.reshape(T, k))


def shared_layer_inputs(wl: Workload, seed: int = 0, layer: int = 0) -> dict:
    """Inputs of one layer with a shared expert beside the E routed ones.

    The router gets one more row (the shared expert's gate, drawn like the
    others: the first E rows are those of router(E, H)), and the expert
    tensors one more expert, the shared one, at index E (drawn from the
    per-expert streams like a routed expert E would be).
    """
    T, H, E, k, I = wl.dims
    d = {
        "hidden": hidden(T, H, seed, 0),
        "router_w": router(E + 1, H, seed, layer),
        "bias": zipf_bias(E, wl.zipf, seed, layer) if wl.zipf else None,
    }
    d.update(expert_weights(E + 1, H, I, seed, layer))
    return d


def bf16_weights(N: int, K: int, seed: int = 0, layer: int = 0, outliers: float = 1.0 / 512) -> torch.Tensor:
    """bf16 [N, K] weights to quantise: N(0, 0.02^2) with a few outliers.

    A fraction `outliers` of the values is multiplied by a factor uniform on
    [4, 12], so that some groups hold one large value: the groups where a
    clipped scale beats the plain maximum.
    """
    g = _rng(seed, layer, _T_QW)
    w = g.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    mask = g.random((N, K), dtype=np.float32) < np.float32(outliers)
    w[mask] *= np.float32(4.0) + np.float32(8.0) * g.random(int(mask.sum()), dtype=np.float32)
    return _bf16(w)


def int8_weights(N: int, K: int, gs: int, seed: int = 0, layer: int = 0) -> dict:
    """INT8 pack-quantized weights of an [N, K] linear layer, on the host.

    Each int32 word is 32 uniform random bits: four bytes uniform on
    [0, 255], the stored values q + 128 of int8 q uniform on [-128, 127]
    (least significant byte first). Scales bf16 [N, K/gs] = 0.0002 + 0.0018 u
    (u uniform on [0, 1), as for the INT4 scales, a tenth of their size since
    |q| reaches 128). Rows are drawn in blocks of 4096 from their own streams,
    so a large matrix is drawn in parallel.
    """
    words = np.empty((N, K // 4), np.int32)
    sc = np.empty((N, K // gs), np.float32)
    blocks = list(range(0, N, 4096))

    def fill(b0: int) -> None:
        b1 = min(N, b0 + 4096)
        words[b0:b1] = _words((seed, layer, _T_W8, b0), (b1 - b0) * (K // 4)).reshape(b1 - b0, K // 4)
        m = _rng(seed, layer, _T_W8S, b0).integers(0, 2**24, (b1 - b0) * (K // gs), dtype=np.int64).astype(np.float32)
        sc[b0:b1] = (np.float32(0.0002) + np.float32(0.0018) * (m * np.float32(1.0 / 2**24))).reshape(b1 - b0, K // gs)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, blocks))
    return {"w_packed": torch.from_numpy(words), "scales": _bf16(sc)}


def layer_inputs(wl: Workload, seed: int = 0, layer: int = 0, experts=None) -> dict:
    """All host inputs of one layer of a workload."""
    T, H, E, k, I = wl.dims
    d = {
        "hidden": hidden(T, H, seed, 0),
        "router_w": router(E, H, seed, layer),
        "bias": zipf_bias(E, wl.zipf, seed, layer) if wl.zipf else None,
    }
    d.update(expert_weights(E, H, I, seed, layer, experts))
    return d
