"""Seeded synthetic inputs for the MoE layer -- shared by the tests, the bench,
the CUDA path and the oracle.  Holds none of the layer's arithmetic: it only
draws numbers, scales them to N(0, 1/fan_in) and casts them.

Recipe (one torch generator per seed, numbers drawn in fp32, then cast with
round-to-nearest-even to the storage type):
  tokens   x [T, d] ~ N(0, 1) drawn first;
  weights  W_g [E, d] ~ N(0, 1/d), then for each expert e in order
           W1[e] [ffn, d] ~ N(0, 1/d), W3[e] [ffn, d] ~ N(0, 1/d),
           W2[e] [d, ffn] ~ N(0, 1/ffn).
A single-layer workload draws tokens and then weights from one generator; the
stacked-layer workload draws tokens from seed 0 and layer l's weights from seed
1000 + l.  torch's CPU and CUDA generators give different streams, so a run
draws everything on one device and copies it to the other side.

Duplicates (skewed workload): round(frac * T) destination rows and as many
source rows are taken from one seeded permutation of the token indices
(destinations first, sources next, so no source is also a destination) and
x[dst] = x[src], giving exact copies.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

MIXTRAL_SHAPE = dict(d=4096, ffn=14336, E=8, k=2)

SKEW_BIAS = (2.0, 1.0, 0.0, 0.0, 0.0, 0.0, -1.0, -2.0)

# The five workloads: the first is small enough for the oracle to do whole;
# the other four are the Mixtral shape (hidden 4096, expert width 14336,
# 8 experts, 2 per token).
WORKLOADS = {
    "tiny": dict(T=64, d=128, ffn=448, E=8, k=2, dtype="f32", seed=0),
    "decode": dict(T=16, **MIXTRAL_SHAPE, dtype="bf16", seed=0),
    "prefill": dict(T=4096, **MIXTRAL_SHAPE, dtype="bf16", seed=0),
    "skewed": dict(T=8192, **MIXTRAL_SHAPE, dtype="bf16", seed=0,
                   bias=SKEW_BIAS, dup_frac=0.05),
    "sweep": dict(Ts=(1, 4, 32, 256, 1024, 4096, 16384), layers=32,
                  **MIXTRAL_SHAPE, dtype="bf16", seed=0, layer_seed0=1000),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Layer:
    Wg: torch.Tensor            # [E, d]
    W1: torch.Tensor            # [E, ffn, d]  gate projection
    W3: torch.Tensor            # [E, ffn, d]  up projection
    W2: torch.Tensor            # [E, d, ffn]  down projection
    bias: torch.Tensor | None = None   # [E] fp32, added to the logits
    meta: dict = field(default_factory=dict)

    @property
    def E(self):
        return self.Wg.shape[0]

    @property
    def d(self):
        return self.Wg.shape[1]

    @property
    def ffn(self):
        return self.W1.shape[1]


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def draw_tokens(gen, T, d, dtype, device, dup_frac=0.0):
    x = torch.randn(T, d, generator=gen, device=device, dtype=torch.float32)
    dups = None
    n_dup = int(round(dup_frac * T))
    if n_dup > 0:
        assert 2 * n_dup <= T
        p = torch.randperm(T, generator=gen, device=device)
        dst, src = p[:n_dup], p[n_dup:2 * n_dup]
        x[dst] = x[src]
        dups = (dst.cpu().numpy(), src.cpu().numpy())
    return x.to(TORCH_DTYPE[dtype]), dups


def draw_weights(gen, d, ffn, E, dtype, device, bias=None) -> Layer:
    tdt = TORCH_DTYPE[dtype]
    Wg = (torch.randn(E, d, generator=gen, device=device) / math.sqrt(d)).to(tdt)
    W1 = torch.empty(E, ffn, d, dtype=tdt, device=device)
    W3 = torch.empty(E, ffn, d, dtype=tdt, device=device)
    W2 = torch.empty(E, d, ffn, dtype=tdt, device=device)
    for e in range(E):
        W1[e] = (torch.randn(ffn, d, generator=gen, device=device) / math.sqrt(d)).to(tdt)
        W3[e] = (torch.randn(ffn, d, generator=gen, device=device) / math.sqrt(d)).to(tdt)
        W2[e] = (torch.randn(d, ffn, generator=gen, device=device) / math.sqrt(ffn)).to(tdt)
    b = None
    if bias is not None:
        b = torch.tensor(bias, dtype=torch.float32, device=device)
        assert b.numel() == E
    return Layer(Wg=Wg, W1=W1, W3=W3, W2=W2, bias=b)


def make_workload(T, d, ffn, E, k=2, dtype="bf16", seed=0, device="cpu",
                  bias=None, dup_frac=0.0):
    """Tokens then weights from one generator.  Returns (x, layer)."""
    gen = generator(seed, device)
    x, dups = draw_tokens(gen, T, d, dtype, device, dup_frac)
    layer = draw_weights(gen, d, ffn, E, dtype, device, bias)
    layer.meta = dict(T=T, d=d, ffn=ffn, E=E, k=k, dtype=dtype, seed=seed,
                      dups=dups)
    return x, layer


def make_named(name, device="cpu", T=None):
    """One of the single-layer workloads by name (optionally with another T)."""
    cfg = dict(WORKLOADS[name])
    if T is not None:
        cfg["T"] = T
    return make_workload(cfg["T"], cfg["d"], cfg["ffn"], cfg["E"], cfg["k"],
                         cfg["dtype"], cfg["seed"], device, cfg.get("bias"),
                         cfg.get("dup_frac", 0.0))


def sweep_tokens(T, d, dtype="bf16", device="cpu", seed=0):
    x, _ = draw_tokens(generator(seed, device), T, d, dtype, device)
    return x


def sweep_layer(l, d, ffn, E, dtype="bf16", device="cpu", seed0=1000):
    return draw_weights(generator(seed0 + l, device), d, ffn, E, dtype, device)


# ---- host views for the oracle -------------------------------------------

def to_host(t: torch.Tensor) -> np.ndarray:
    """fp32 -> float32 array, bf16 -> uint16 array of the raw bit patterns."""
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    raise TypeError(t.dtype)


def from_host(a: np.ndarray, device="cpu") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def layer_to_host(layer: Layer):
    """(Wg, [W1[e]], [W3[e]], [W2[e]], bias) as host arrays for the oracle."""
    E = layer.E
    Wg = to_host(layer.Wg)
    W1 = [to_host(layer.W1[e]) for e in range(E)]
    W3 = [to_host(layer.W3[e]) for e in range(E)]
    W2 = [to_host(layer.W2[e]) for e in range(E)]
    bias = None if layer.bias is None else layer.bias.detach().cpu().numpy()
    return Wg, W1, W3, W2, bias
