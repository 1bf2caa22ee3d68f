"""Shared helpers for the GPU parity tests: running the oracle on host copies
of a workload and the parity measures."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import bf16_bits_to_f64
from sparse_mixture_experts_58_b300 import inputs

# Parity bounds.  fp32 layers: max|gpu - ref| / max|ref| <= TOL_F32.  bf16
# layers: max over elements of (|gpu - exact| - half a bf16 ulp of gpu),
# divided by RMS(exact), <= TOL_BF16, where `exact` is the oracle's result
# before its final rounding -- the error beyond the one rounding every bf16
# output carries.  The raw max|gpu - exact| / RMS(exact) is printed beside it
# (not gated).  Tokens whose kept/next logits are closer than NEAR_TIE on the
# oracle's fp32 logits are left out of index and output comparisons and
# counted.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
NEAR_TIE = 1e-3


def host_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def near_tie_mask(logits: np.ndarray, k: int) -> np.ndarray:
    """True for tokens whose sorted top-(k+1) logits have an adjacent gap
    below NEAR_TIE (a selection or slot order that rounding may flip)."""
    s = -np.sort(-logits.astype(np.float64), axis=1)
    m = min(k + 1, logits.shape[1])
    if m < 2:
        return np.zeros(logits.shape[0], bool)
    gaps = s[:, :m - 1] - s[:, 1:m]
    return (gaps < NEAR_TIE).any(1)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at each value (0 at 0): for |v| in [2^e, 2^(e+1))
    the spacing of bf16 values is 2^(e-7)."""
    _, ex = np.frexp(np.abs(v))          # |v| = m * 2^ex, m in [0.5, 1)
    return np.where(v == 0, 0.0, np.ldexp(1.0, ex - 9))


def rel_error(gpu: np.ndarray, ref: np.ndarray, dtype: str) -> float:
    """Parity measure.  fp32: max|gpu - ref| / max|ref|.  bf16:
    max(|gpu - ref| - half_ulp(gpu), 0) / RMS(ref) with ref the exact
    (unrounded) result: the error beyond the one rounding every bf16 output
    must carry (half a bf16 ulp, up to 2^-8 of the value), relative to RMS."""
    g = host_f64(gpu)
    r = host_f64(ref) if ref.dtype == np.uint16 else ref.astype(np.float64)
    if g.size == 0:
        return 0.0
    if dtype == "f32":
        diff = np.abs(g - r).max()
        den = np.abs(r).max()
    else:
        diff = np.maximum(np.abs(g - r) - bf16_half_ulp(g), 0.0).max()
        den = np.sqrt((r ** 2).mean())
    return float(diff / den) if den > 0 else float(diff)


def raw_rel_error(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max|gpu - ref| / RMS(ref), rounding included (reported, not gated)."""
    g = host_f64(gpu)
    r = ref.astype(np.float64) if ref.dtype != np.uint16 else host_f64(ref)
    den = np.sqrt((r ** 2).mean()) if r.size else 0.0
    return float(np.abs(g - r).max() / den) if den > 0 else 0.0


def tol(dtype: str) -> float:
    return TOL_F32 if dtype == "f32" else TOL_BF16


def oracle_on_rows(x: torch.Tensor, layer: inputs.Layer, k: int, rows=None, threads=0,
                   host_layer=None):
    """Run the oracle on the given token rows (all when rows is None).
    Returns (ref, logits, idx, gates) as host arrays for those rows, where
    ref is the oracle's result before its final rounding (float64).

    The bf16 comparison is made against that exact value: comparing two
    independently rounded bf16 outputs would add a possible one-ulp flip
    (2^-7 relative) on the largest elements, which alone can exceed a
    2e-2 * RMS bound."""
    o = oracle.load()
    xs = x if rows is None else x[torch.as_tensor(rows, device=x.device, dtype=torch.long)]
    xh = inputs.to_host(xs)
    Wg, W1, W3, W2, bias = host_layer if host_layer is not None else inputs.layer_to_host(layer)
    out, logits, idx, gates, exact = o.moe_forward(xh, Wg, W1, W3, W2, k, bias=bias,
                                                   threads=threads, exact=True)
    return exact, logits, idx, gates


def sample_rows(T: int, n: int, seed: int, must=()) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(int(v) for v in must)
    n = min(n, T)
    if len(pick) < n:
        extra = rng.choice(T, size=min(T, n), replace=False)
        for v in extra:
            if len(pick) >= n:
                break
            pick.add(int(v))
    return np.array(sorted(pick), dtype=np.int64)


def pair_token_tiles(cnt: int, max_tok: int = 256):
    """Token tiles of one expert's `cnt` grouped rows in the CTA-pair GEMMs:
    ceil(cnt / 256) tiles of equal height rounded up to 16 (the MMA's N
    granularity).  Returns [(first row, rows)] relative to the expert."""
    if cnt <= 0:
        return []
    t0 = -(-cnt // max_tok)
    nt = ((-(-cnt // t0)) + 15) // 16 * 16
    return [(s, min(nt, cnt - s)) for s in range(0, cnt, nt)]


def layout_rows(idx: np.ndarray, offsets: np.ndarray, perm: np.ndarray, k: int,
                per_expert: int = 16, seed: int = 0, must=(), halves: bool = True,
                row_tiles=(128,)) -> np.ndarray:
    """Tokens to compare for a batch too large for the oracle to do whole,
    chosen from the grouped layout (rows ordered by expert, then token) so
    that the rows where tiling bugs hide are covered: for every expert with
    rows, the tokens holding its first and last grouped rows; the first and
    last rows of each of its CTA-pair token tiles (and, with `halves`, the
    two rows either side of the split between the pair's two CTAs); the rows
    either side of every multiple of each height in `row_tiles` (the one-CTA
    kernel's token tiles); then random rows of the expert until at least
    `per_expert` of its rows are covered.  idx [T][k], offsets [E+1], perm
    [T*k] are one routing of the batch (the oracle's)."""
    rng = np.random.default_rng(seed)
    E = len(offsets) - 1
    pick = set(int(t) for t in must)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        cnt = hi - lo
        if cnt == 0:
            continue
        rel = {0, cnt - 1}
        for s0, n in pair_token_tiles(cnt):
            rel.update((s0, s0 + n - 1))
            if halves:
                half = (((n + 15) // 16 * 16) // 2)
                rel.update((s0 + half - 1, s0 + half))
        for h in row_tiles:
            for b in range(h, cnt, h):
                rel.update((b - 1, b))
        for r in rel:
            if 0 <= r < cnt:
                pick.add(int(perm[lo + r]) // k)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        have = sum(1 for t in pick if (idx[t] == e).any())
        need = min(per_expert, hi - lo) - have
        if need > 0:
            cand = [int(perm[r]) // k for r in rng.permutation(np.arange(lo, hi))]
            for t in cand:
                if need <= 0:
                    break
                if t not in pick:
                    pick.add(t)
                    need -= 1
    return np.array(sorted(pick), dtype=np.int64)


def oracle_layout(x_host: np.ndarray, host_layer, k: int):
    """The oracle's routing of a whole batch (router and grouping only):
    (logits, idx, offsets, perm)."""
    o = oracle.load()
    Wg, _, _, _, bias = host_layer
    logits, _, _ = o.router(x_host, Wg, k, bias=bias)
    idx, _, _, offsets, perm, _ = o.route(logits, k)
    return logits, idx, offsets, perm
