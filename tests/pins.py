"""Pins for the CPU oracle: facts the pages and plain mathematics fix, each
checked against the oracle without using the oracle's own formulas.

Each pin takes an ``oracle.Oracle`` (any build of ``oracle/moe_oracle.c``) and
raises AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them on the
real build; ``test_oracle_mutants.py`` runs them on builds with a planted
mistake and checks that some pin fails for each.

Where a pin needs a second computation it is a different one: a closed form
worked by hand, a library routine (numpy sort/matmul, torch casts), or a dense
brute force that evaluates every expert.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

from oracle import bf16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def silu(u):
    return u / (1.0 + math.exp(-u))


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_layer(rng, T, d, ffn, E, scale=1.0):
    x = rng.standard_normal((T, d)).astype(np.float32) * np.float32(scale)
    Wg = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    W1 = (rng.standard_normal((E, ffn, d)) / math.sqrt(d)).astype(np.float32)
    W3 = (rng.standard_normal((E, ffn, d)) / math.sqrt(d)).astype(np.float32)
    W2 = (rng.standard_normal((E, d, ffn)) / math.sqrt(ffn)).astype(np.float32)
    return x, Wg, W1, W3, W2


def _dense_swiglu(x, W1, W3, W2):
    """Textbook SwiGLU FFN on a batch of row vectors, float64 matmuls."""
    x = x.astype(np.float64)
    u = x @ W1.astype(np.float64).T
    v = x @ W3.astype(np.float64).T
    h = u / (1.0 + np.exp(-u)) * v
    return h @ W2.astype(np.float64).T


# ---------------------------------------------------------------------------
# 1. A worked example, done by hand.
#
# d=2, ffn=2, E=3, k=2, fp32.  a = fp32(ln 3), so exp(-a) = 1/3 up to fp32.
#   W_g = [[a,0],[0,a],[0,0]]
#   expert 0: W1=[[1,0],[0,1]]  W3=[[2,0],[1,3]]  W2=[[1,0],[1,2]]
#   expert 1: W1=[[0,1],[1,0]]  W3=[[1,1],[1,0]]  W2=[[0,1],[2,0]]
#   expert 2: W1=[[-1,0],[0,1]] W3=[[1,0],[0,1]]  W2=[[1,1],[0,1]]
# (row c of W1/W3 is feature c's input weights; row n of W2 is output n's.)
# With s1=silu(1), s2=silu(2), m1=silu(-1):
#   t0 x=[1,0]:  logits (a,0,0): keeps 0, then 1 (tie with 2 -> lower index);
#                gates 3/4, 1/4.
#                e0: u=(1,0) v=(2,1) h=(2s1,0) y=(2s1,2s1)
#                e1: u=(0,1) v=(1,1) h=(0,s1)  y=(s1,0)
#                out = (1.75 s1, 1.5 s1)
#   t1 x=[1,2]:  logits (a,2a,0): keeps 1 then 0; gates 3/4, 1/4.
#                e1: u=(2,1) v=(3,1) h=(3s2,s1) y=(s1,6s2)
#                e0: u=(1,2) v=(2,7) h=(2s1,7s2) y=(2s1,2s1+14s2)
#                out = (1.25 s1, 0.5 s1 + 8 s2)
#   t2 x=[-1,-1]: logits (-a,-a,0): keeps 2, then 0 (tie with 1); gates 3/4, 1/4.
#                e2: u=(1,-1) v=(-1,-1) h=(-s1,-m1) y=(-s1-m1,-m1)
#                e0: u=(-1,-1) v=(-2,-4) h=(-2m1,-4m1) y=(-2m1,-10m1)
#                out = (-0.75 s1 - 1.25 m1, -3.25 m1)
# Grouping: expert 0 gets (t0,slot0),(t1,slot1),(t2,slot1); expert 1 gets
# (t0,slot1),(t1,slot0); expert 2 gets (t2,slot0):
#   counts (3,2,1), offsets (0,3,5,6), perm (0,3,5,1,2,4), inv (0,3,4,1,5,2).
# ---------------------------------------------------------------------------

def hand_example():
    a = np.float32(math.log(3.0))
    x = np.array([[1, 0], [1, 2], [-1, -1]], np.float32)
    Wg = np.array([[a, 0], [0, a], [0, 0]], np.float32)
    W1 = np.array([[[1, 0], [0, 1]], [[0, 1], [1, 0]], [[-1, 0], [0, 1]]], np.float32)
    W3 = np.array([[[2, 0], [1, 3]], [[1, 1], [1, 0]], [[1, 0], [0, 1]]], np.float32)
    W2 = np.array([[[1, 0], [1, 2]], [[0, 1], [2, 0]], [[1, 1], [0, 1]]], np.float32)
    s1, s2, m1 = silu(1.0), silu(2.0), silu(-1.0)
    out = np.array([[1.75 * s1, 1.5 * s1],
                    [1.25 * s1, 0.5 * s1 + 8 * s2],
                    [-0.75 * s1 - 1.25 * m1, -3.25 * m1]])
    return dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, out=out,
                idx=np.array([[0, 1], [1, 0], [2, 0]]),
                gates=np.array([[0.75, 0.25]] * 3),
                counts=np.array([3, 2, 1]), offsets=np.array([0, 3, 5, 6]),
                perm=np.array([0, 3, 5, 1, 2, 4]), inv=np.array([0, 3, 4, 1, 5, 2]))


def pin_hand_example(o):
    h = hand_example()
    out, logits, idx, gates = o.moe_forward(h["x"], h["Wg"], h["W1"], h["W3"], h["W2"], 2)
    assert np.array_equal(idx, h["idx"]), idx
    assert np.allclose(gates, h["gates"], rtol=0, atol=1e-7), gates
    assert np.allclose(out, h["out"], rtol=1e-6, atol=1e-7), (out, h["out"])
    ridx, rg, counts, offsets, perm, inv = o.route(logits, 2)
    assert np.array_equal(ridx, h["idx"])
    assert np.array_equal(counts, h["counts"]), counts
    assert np.array_equal(offsets, h["offsets"]), offsets
    assert np.array_equal(perm, h["perm"]), perm
    assert np.array_equal(inv, h["inv"]), inv


def pin_hand_example_bf16(o):
    """Same example stored as bf16: every input is exact in bf16 except a,
    whose bf16 rounding moves the gates by < 1e-2; outputs round once."""
    h = hand_example()
    to = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _, idx, gates = o.moe_forward(to(h["x"]), to(h["Wg"]), to(h["W1"]),
                                       to(h["W3"]), to(h["W2"]), 2)
    assert np.array_equal(idx, h["idx"])
    a16 = float(torch.tensor(math.log(3.0)).to(torch.bfloat16).float())
    g0 = 1.0 / (1.0 + math.exp(-a16))
    g = np.array([[g0, 1 - g0]] * 3)
    # t1's gates compare 2a with a: same difference a
    assert np.allclose(gates, g, atol=1e-12)
    s1, s2, m1 = silu(1.0), silu(2.0), silu(-1.0)
    exp = np.array([[g0 * 2 * s1 + (1 - g0) * s1, g0 * 2 * s1],
                    [g0 * s1 + (1 - g0) * 2 * s1, g0 * 6 * s2 + (1 - g0) * (2 * s1 + 14 * s2)],
                    [g0 * (-s1 - m1) + (1 - g0) * (-2 * m1), g0 * (-m1) + (1 - g0) * (-10 * m1)]])
    got = bf16_bits_to_f64(out)
    assert np.all(np.abs(got - exp) <= np.abs(exp) * 2.0 ** -8 + 1e-12), (got, exp)


# ---------------------------------------------------------------------------
# 2. Router: gates and selection.
# ---------------------------------------------------------------------------

def pin_gates_sum_and_renormalised_softmax(o):
    rng = _rng(1)
    for E, k in ((8, 2), (5, 2), (3, 1), (16, 2), (2, 2)):
        logits = (rng.standard_normal((200, E)) * 3).astype(np.float32)
        idx, gates, *_ = o.route(logits, k)
        assert np.all(np.abs(gates.sum(1) - 1.0) <= 4e-16)
        if k == 1:
            assert np.all(gates == 1.0)
        l64 = logits.astype(np.float64)
        p = np.exp(l64 - l64.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        sel = np.take_along_axis(p, idx.astype(np.int64), 1)
        ref = sel / sel.sum(1, keepdims=True)
        assert np.allclose(gates, ref, rtol=1e-13, atol=1e-15)
        # slot 0 carries the larger gate
        assert np.all(gates[:, 0] >= gates[:, -1])


def pin_selection_bruteforce(o):
    rng = _rng(2)
    for E, k in ((8, 2), (4, 2), (6, 1), (32, 2)):
        # coarse values make ties common
        logits = rng.integers(-3, 4, size=(300, E)).astype(np.float32) * np.float32(0.5)
        idx, *_ = o.route(logits, k)
        for t in range(logits.shape[0]):
            key = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
            assert list(idx[t]) == key[:k], (t, logits[t], idx[t])
            if k == 2:
                best = max(logits[t, a] + logits[t, b]
                           for a, b in itertools.combinations(range(E), 2))
                assert logits[t, idx[t, 0]] + logits[t, idx[t, 1]] == best


def pin_zero_router(o):
    rng = _rng(3)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 7, 16, 24, 6)
    Wg[:] = 0
    out, logits, idx, gates = o.moe_forward(x, Wg, W1, W3, W2, 2)
    assert np.all(logits == 0)
    assert np.all(idx == np.array([0, 1]))
    assert np.all(gates == 0.5)
    ref = 0.5 * _dense_swiglu(x, W1[0], W3[0], W2[0]) + 0.5 * _dense_swiglu(x, W1[1], W3[1], W2[1])
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)


def pin_duplicate_router_rows(o):
    """Two experts with identical router weights always tie; the lower index
    is taken first."""
    rng = _rng(4)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 50, 16, 8, 6)
    Wg[4] = Wg[1] * 10
    Wg[1] = Wg[4]
    _, logits, idx, _ = o.moe_forward(x, Wg, W1, W3, W2, 2)
    assert np.array_equal(logits[:, 1], logits[:, 4])
    for t in range(50):
        if 1 in idx[t] or 4 in idx[t]:
            pos1 = list(idx[t]).index(1) if 1 in idx[t] else None
            pos4 = list(idx[t]).index(4) if 4 in idx[t] else None
            assert pos1 is not None          # 4 never beats 1
            if pos4 is not None:
                assert pos1 < pos4


def pin_router_bias(o):
    """A bias added to the logits: big enough to force experts 0 and 1."""
    rng = _rng(5)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 20, 16, 8, 8)
    bias = np.array([100.0, 50.0, 0, 0, 0, 0, -1, -2], np.float32)
    logits0, _, _ = o.router(x, Wg, 2)
    logits, idx, gates = o.router(x, Wg, 2, bias=bias)
    assert np.all(idx == np.array([0, 1]))
    assert np.allclose(logits, logits0 + bias, rtol=0, atol=1e-4)


def pin_router_logits_exact(o):
    """Logits are the dot products rounded once to fp32: checked with small
    integers, where every product and sum is exact."""
    rng = _rng(6)
    x = rng.integers(-8, 9, size=(30, 40)).astype(np.float32)
    Wg = rng.integers(-8, 9, size=(7, 40)).astype(np.float32)
    logits, _, _ = o.router(x, Wg, 2)
    ref = x.astype(np.int64) @ Wg.astype(np.int64).T
    assert np.array_equal(logits, ref.astype(np.float32))


# ---------------------------------------------------------------------------
# 3. Grouping tokens by expert.
# ---------------------------------------------------------------------------

def pin_route_invariants(o):
    rng = _rng(7)
    for T, E, k in ((257, 8, 2), (64, 3, 1), (1, 8, 2), (100, 2, 2), (40, 32, 2)):
        logits = rng.standard_normal((T, E)).astype(np.float32)
        idx, gates, counts, offsets, perm, inv = o.route(logits, k)
        assert counts.sum() == T * k
        assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        assert offsets[0] == 0 and offsets[-1] == T * k
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(np.sort(perm), np.arange(T * k))      # bijection
        assert np.array_equal(inv[perm], np.arange(T * k))          # inv o perm = id
        assert np.array_equal(perm[inv], np.arange(T * k))
        flat = idx.ravel()
        for e in range(E):
            rows = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[rows] == e)
            assert np.all(np.diff(rows // k) > 0)                    # ascending tokens


def pin_route_empty(o):
    logits = np.zeros((0, 8), np.float32)
    idx, gates, counts, offsets, perm, inv = o.route(logits, 2)
    assert counts.sum() == 0 and np.all(offsets == 0)


def pin_forward_matches_route(o):
    """The forward's own selection equals grouping from its logits."""
    rng = _rng(8)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 33, 16, 8, 8)
    _, logits, idx, gates = o.moe_forward(x, Wg, W1, W3, W2, 2)
    ridx, rg, *_ = o.route(logits, 2)
    assert np.array_equal(idx, ridx) and np.array_equal(gates, rg)


# ---------------------------------------------------------------------------
# 4. Expert FFN and the whole layer.
# ---------------------------------------------------------------------------

def pin_dense_bruteforce(o):
    """Sparse result == all E experts evaluated densely, weighted by the full
    softmax masked to the kept experts and renormalised."""
    rng = _rng(9)
    for T, d, ffn, E, k in ((16, 8, 12, 5, 2), (9, 6, 10, 4, 1), (12, 4, 4, 8, 2)):
        x, Wg, W1, W3, W2 = _rand_layer(rng, T, d, ffn, E)
        out, logits, idx, _ = o.moe_forward(x, Wg, W1, W3, W2, k)
        l64 = (x.astype(np.float64) @ Wg.astype(np.float64).T).astype(np.float32)
        assert np.allclose(logits, l64, rtol=0, atol=1e-6)
        l = logits.astype(np.float64)
        mask = np.zeros_like(l, dtype=bool)
        order = np.argsort(-l, axis=1, kind="stable")[:, :k]
        np.put_along_axis(mask, order, True, 1)
        p = np.exp(l - l.max(1, keepdims=True))
        w = np.where(mask, p, 0.0)
        w /= w.sum(1, keepdims=True)
        ys = np.stack([_dense_swiglu(x, W1[e], W3[e], W2[e]) for e in range(E)], 1)
        ref = (w[:, :, None] * ys).sum(1)
        assert np.allclose(out, ref, rtol=2e-6, atol=2e-7), np.abs(out - ref).max()


def pin_single_expert_dense(o):
    """E=1, k=1: the layer is one dense SwiGLU FFN."""
    rng = _rng(10)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 11, 12, 20, 1)
    out, _, idx, gates = o.moe_forward(x, Wg, W1, W3, W2, 1)
    assert np.all(idx == 0) and np.all(gates == 1.0)
    ref = _dense_swiglu(x, W1[0], W3[0], W2[0])
    assert np.allclose(out, ref, rtol=2e-6, atol=2e-7)


def pin_identical_experts(o):
    """All experts equal: the gates sum to 1, so any routing gives the dense FFN."""
    rng = _rng(11)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 21, 10, 14, 6)
    W1[:] = W1[0]
    W3[:] = W3[0]
    W2[:] = W2[0]
    out, *_ = o.moe_forward(x, Wg, W1, W3, W2, 2)
    ref = _dense_swiglu(x, W1[0], W3[0], W2[0])
    assert np.allclose(out, ref, rtol=2e-6, atol=2e-7)


def pin_token_independence(o):
    """Tokens are processed independently: permuting them permutes the
    outputs bit for bit, and duplicated tokens give identical rows."""
    rng = _rng(12)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 24, 8, 12, 8)
    x[5] = x[17]
    out, _, idx, _ = o.moe_forward(x, Wg, W1, W3, W2, 2)
    assert np.array_equal(out[5], out[17]) and np.array_equal(idx[5], idx[17])
    p = rng.permutation(24)
    outp, *_ = o.moe_forward(x[p], Wg, W1, W3, W2, 2)
    assert np.array_equal(outp, out[p])


def pin_exact_output_rounds_to_out(o):
    """The unrounded result the oracle exposes is the value its output rounds
    from: one nearest-even rounding per element, in both storage types."""
    rng = _rng(16)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 12, 16, 24, 4)
    out, _, _, _, ex = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True)
    assert np.array_equal(out, ex.astype(np.float32))
    to = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    outb, _, _, _, exb = o.moe_forward(to(x), to(Wg), to(W1), to(W3), to(W2), 2, exact=True)
    assert np.array_equal(outb, np.array([o.to_bf16(v) for v in exb.ravel()],
                                         np.uint16).reshape(outb.shape))
    assert np.all(np.abs(bf16_bits_to_f64(outb) - exb) <= np.abs(exb) * 2.0 ** -8)


def pin_down_projection_linear(o):
    """Doubling W2 doubles the output exactly (a power-of-two scale commutes
    with every rounding)."""
    rng = _rng(13)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 10, 8, 12, 4)
    out, *_ = o.moe_forward(x, Wg, W1, W3, W2, 2)
    out2, *_ = o.moe_forward(x, Wg, W1, W3, W2 * 2, 2)
    assert np.array_equal(out2, out * 2)


def pin_silu_limits(o):
    """One expert, one feature: a large positive gate input passes u*v
    through, a large negative one gives 0 (silu(u) -> u, -> 0)."""
    x = np.array([[1.0]], np.float32)
    Wg = np.array([[0.0]], np.float32)
    for u, expect in ((40.0, 40.0 * 3.0 * 0.5), (-40.0, 0.0), (0.0, 0.0)):
        W1 = np.array([[[u]]], np.float32)
        W3 = np.array([[[3.0]]], np.float32)
        W2 = np.array([[[0.5]]], np.float32)
        out, *_ = o.moe_forward(x, Wg, W1, W3, W2, 1)
        assert abs(float(out[0, 0]) - expect) <= 1e-5 * max(1.0, abs(expect)), (u, out)


# ---------------------------------------------------------------------------
# 5. Number formats and the stacked-layer helpers.
# ---------------------------------------------------------------------------

def pin_bf16_rounding(o):
    rng = _rng(14)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                           [0.0, -0.0, 1.0, -1.0, 65504.0, 1e-40]]).astype(np.float32)
    # exact bf16 midpoints: a bf16 value plus half its ulp
    base = torch.from_numpy(rng.standard_normal(2000).astype(np.float32)).to(torch.bfloat16).float()
    mids = (base.view(torch.int32) + 0x8000).view(torch.float32).numpy()
    vals = np.concatenate([vals, mids])
    lib = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([o.to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(mine, lib), np.flatnonzero(mine != lib)[:5]
    # one rounding from double: 1 + 2^-8 + 2^-30 is above the midpoint between
    # 1 and 1 + 2^-7, although its fp32 rounding lands exactly on it
    assert o.to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert o.to_bf16(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even
    assert o.to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (up)
    for h in (0x3F80, 0xBF81, 0x0001, 0x7F7F):
        b = np.array([h], np.uint16)
        assert o.from_bf16(h) == float(bf16_bits_to_f64(b)[0])


def pin_rmsnorm(o):
    eps = 1e-5
    c = np.float32(0.01)
    x = np.full((2, 64), c, np.float32)
    x[1] = -c
    y = o.rmsnorm(x, eps)
    ref = float(c) / math.sqrt(float(c) ** 2 + eps)
    assert np.allclose(y[0], ref, rtol=1e-6) and np.allclose(y[1], -ref, rtol=1e-6)
    rng = _rng(15)
    x = rng.standard_normal((8, 96)).astype(np.float32)
    y = o.rmsnorm(x, eps)
    lib = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (96,), eps=eps).float().numpy()
    assert np.allclose(y, lib, rtol=1e-6, atol=1e-7)


def pin_add(o):
    a = np.array([1.0, 2.0 ** 20, -3.5], np.float32)
    b = np.array([2.0 ** -30, 1.0, 3.5], np.float32)
    z = o.add(a, b)
    assert np.array_equal(z, np.array([1.0, 2.0 ** 20 + 1, 0.0], np.float32))
    to = lambda v: np.array([o.to_bf16(t) for t in v], np.uint16)
    zb = o.add(to([1.0, 256.0]), to([2.0 ** -9, 1.0]))
    # 1 + 2^-9 rounds to 1 (below the midpoint); 256 + 1 is a tie -> 256 (even)
    assert list(zb) == [0x3F80, 0x4380]


# ---------------------------------------------------------------------------
# 6. Router variant: softmax over all experts, then top-k, no renormalisation.
# ---------------------------------------------------------------------------

def pin_hand_example_softmax_then_topk(o):
    """The worked example with gating 1.  t0 logits (a,0,0), a = ln 3: the
    full softmax is (3/5, 1/5, 1/5), experts 0 and 1 kept with gates 3/5 and
    1/5: out = 3/5 (2s1, 2s1) + 1/5 (s1, 0) = (1.4 s1, 1.2 s1).
    t1 logits (a,2a,0): softmax (3, 9, 1)/13, experts 1 then 0, gates 9/13,
    3/13: out = 9/13 (s1, 6s2) + 3/13 (2s1, 2s1+14s2)."""
    h = hand_example()
    out, _, idx, gates = o.moe_forward(h["x"], h["Wg"], h["W1"], h["W3"], h["W2"], 2, gating=1)
    s1, s2 = silu(1.0), silu(2.0)
    assert np.array_equal(idx, h["idx"])
    assert np.allclose(gates[0], [0.6, 0.2], atol=1e-7)
    assert np.allclose(gates[1], [9 / 13, 3 / 13], atol=1e-7)
    assert np.allclose(out[0], [1.4 * s1, 1.2 * s1], rtol=1e-6)
    want1 = [9 / 13 * s1 + 3 / 13 * 2 * s1, 9 / 13 * 6 * s2 + 3 / 13 * (2 * s1 + 14 * s2)]
    assert np.allclose(out[1], want1, rtol=1e-6)


def pin_softmax_then_topk_gates(o):
    """Gating 1: each gate is the full softmax probability of its expert
    (library softmax), the gates sum to at most 1 (exactly 1 when k = E), and
    the layer output is the gating-0 output scaled per token by that sum."""
    from scipy.special import softmax
    rng = _rng(20)
    for E, k in ((8, 2), (5, 5), (16, 4), (64, 8)):
        logits = (rng.standard_normal((100, E)) * 2).astype(np.float32)
        idx, g, *_ = o.route(logits, k, gating=1)
        p = softmax(logits.astype(np.float64), axis=1)
        assert np.allclose(g, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-13)
        assert np.all(g.sum(1) <= 1 + 1e-15)
        if k == E:
            assert np.allclose(g.sum(1), 1.0, atol=1e-15)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 9, 8, 12, 6)
    _, l0, i0, g0, ex0 = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True)
    _, l1, i1, g1, ex1 = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True, gating=1)
    assert np.array_equal(i0, i1)
    assert np.allclose(ex1, ex0 * g1.sum(1, keepdims=True), rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# 7. Capacity-limited routing.
# ---------------------------------------------------------------------------

def pin_capacity_hand_example(o):
    """Capacity 1 on the worked example: expert 0's selections in token order
    are (t0,slot0), (t1,slot1), (t2,slot1); expert 1's (t0,slot1), (t1,slot0);
    expert 2's (t2,slot0).  Kept: t0 both slots, t1 none, t2 slot 0 only.
    Lost mass: out[t1] = 0, out[t2] = 3/4 y2 = 3/4 (-s1-m1, -m1);
    renormalised: out[t2] = y2."""
    h = hand_example()
    s1, m1 = silu(1.0), silu(-1.0)
    y2 = np.array([-s1 - m1, -m1])
    for renorm, scale in ((0, 0.75), (1, 1.0)):
        out, *_ = o.moe_forward(h["x"], h["Wg"], h["W1"], h["W3"], h["W2"], 2, capacity=1,
                                drop_renorm=renorm)
        assert np.allclose(out[0], h["out"][0], rtol=1e-6)
        assert np.all(out[1] == 0)
        assert np.allclose(out[2], scale * y2, rtol=1e-6)
    idx, g, counts, offsets, perm, inv = o.route(
        o.moe_forward(h["x"], h["Wg"], h["W1"], h["W3"], h["W2"], 2)[1], 2, capacity=1)
    assert list(counts) == [1, 1, 1] and list(offsets) == [0, 1, 2, 3]
    assert list(perm) == [0, 1, 4] and list(inv) == [0, 1, -1, -1, 2, -1]


def pin_capacity_route_bruteforce(o):
    """Kept selections = each expert's first C selections in token order
    (built here with a stable sort); rows as in the dropless grouping."""
    rng = _rng(21)
    for T, E, k, C in ((200, 8, 2, 30), (64, 4, 2, 1), (100, 16, 4, 20), (50, 8, 2, 1000),
                       (80, 64, 8, 9)):
        logits = rng.standard_normal((T, E)).astype(np.float32)
        logits[:, 0] += 2.0                       # make expert 0 overflow
        idx, g, counts, offsets, perm, inv = o.route(logits, k, capacity=C)
        flat = idx.ravel()
        order = np.argsort(flat, kind="stable")   # by expert, then (token, slot)
        kept = np.zeros(T * k, bool)
        for e in range(E):
            sel = order[flat[order] == e]
            kept[sel[:C]] = True
        assert np.array_equal(counts, np.minimum(np.bincount(flat, minlength=E), C))
        assert np.array_equal(inv < 0, ~kept)
        assert np.array_equal(np.sort(perm), np.flatnonzero(kept))
        assert np.array_equal(inv[perm], np.arange(offsets[-1]))
        for e in range(E):
            rows = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[rows] == e) and np.all(np.diff(rows // k) > 0)


def pin_capacity_gate_policies(o):
    """Lost mass: kept slots keep their gates.  Renormalised: each token's kept
    gates sum to its full gate mass (1 in gating 0, the kept softmax mass in
    gating 1).  A capacity that drops nothing changes nothing."""
    rng = _rng(22)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 40, 8, 12, 4)
    Wg[0] *= 0.0
    Wg[0, 0] = 5.0                                 # expert 0 popular
    base = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True)
    same = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True, capacity=40)
    assert np.array_equal(base[4], same[4])
    for gating in (0, 1):
        _, _, idx, g, ex_lost = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True, gating=gating,
                                              capacity=6)
        _, _, _, _, ex_ren = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True, gating=gating,
                                           capacity=6, drop_renorm=1)
        _, _, _, _, ex_full = o.moe_forward(x, Wg, W1, W3, W2, 2, exact=True, gating=gating)
        _, _, _, _, _, inv = o.route(base[1], 2, gating=gating, capacity=6)
        kept = (inv >= 0).reshape(-1, 2)
        # per-expert contributions from single-expert layers (k = 1 on a copy)
        for t in range(40):
            if kept[t].all():
                assert np.allclose(ex_lost[t], ex_full[t], rtol=1e-12, atol=1e-15)
                assert np.allclose(ex_ren[t], ex_full[t], rtol=1e-12, atol=1e-15)
            elif not kept[t].any():
                assert np.all(ex_lost[t] == 0) and np.all(ex_ren[t] == 0)
            else:
                j = int(np.flatnonzero(kept[t])[0])
                # renormalised = lost-mass output scaled by total / kept gate
                scale = g[t].sum() / g[t, j]
                assert np.allclose(ex_ren[t], ex_lost[t] * scale, rtol=1e-12, atol=1e-15)


def pin_large_E_and_k(o):
    """64 experts and k up to 8 (k = E too): the dense brute force."""
    rng = _rng(23)
    for T, d, ffn, E, k in ((6, 8, 8, 64, 8), (5, 6, 4, 4, 4), (7, 8, 6, 16, 3)):
        x, Wg, W1, W3, W2 = _rand_layer(rng, T, d, ffn, E)
        out, logits, idx, _ = o.moe_forward(x, Wg, W1, W3, W2, k)
        l = logits.astype(np.float64)
        order = np.argsort(-l, axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, order)
        mask = np.zeros_like(l, dtype=bool)
        np.put_along_axis(mask, order, True, 1)
        p = np.where(mask, np.exp(l - l.max(1, keepdims=True)), 0.0)
        w = p / p.sum(1, keepdims=True)
        ys = np.stack([_dense_swiglu(x, W1[e], W3[e], W2[e]) for e in range(E)], 1)
        ref = (w[:, :, None] * ys).sum(1)
        assert np.allclose(out, ref, rtol=2e-6, atol=2e-7)


# ---------------------------------------------------------------------------
# 8. The pages' printed numbers for the Mixtral shape.
# ---------------------------------------------------------------------------

def pin_page_shape_numbers(o=None):
    with open(os.path.join(GOLDEN, "mixtral_shape.json")) as f:
        g = json.load(f)
    from sparse_mixture_experts_58_b300.inputs import MIXTRAL_SHAPE
    v = g["values"]
    assert MIXTRAL_SHAPE["d"] == v["hidden_dimension"]
    assert MIXTRAL_SHAPE["ffn"] == v["expert_ffn_intermediate_dimension"]
    assert MIXTRAL_SHAPE["E"] == v["experts_per_layer"]
    assert MIXTRAL_SHAPE["k"] == v["active_experts_per_token"]
    per_proj = MIXTRAL_SHAPE["d"] * MIXTRAL_SHAPE["ffn"]
    assert round(per_proj / 1e6, 1) == v["params_per_projection_millions"]
    ffn_total = 3 * per_proj * MIXTRAL_SHAPE["E"] * v["layers"]
    assert round(ffn_total / 1e9) == v["ffn_params_billions"]
    assert abs(ffn_total / 1e9 + v["other_params_billions"] - v["total_params_billions"]) < 0.15
    active = 3 * per_proj * MIXTRAL_SHAPE["k"] * v["layers"] + v["other_params_billions"] * 1e9
    assert abs(active / 1e9 - v["active_params_billions"]) < 0.1
    assert MIXTRAL_SHAPE["k"] / MIXTRAL_SHAPE["E"] == v["fraction_active"]


# ---------------------------------------------------------------------------
# Backward (gradients of sum(dout * layer(x)), for training).  Pinned to the
# forward itself by finite differences, to torch's autograd on the layer with
# the oracle's expert choice held fixed, and to properties of the softmax.
# ---------------------------------------------------------------------------

def _loss(o, x, Wg, W1, W3, W2, k, dout):
    """sum(dout * exact layer output) and the expert choice, from the forward."""
    _, _, idx, _, ex = o.moe_forward(x, Wg, W1, W3, W2, k, exact=True)
    return float((ex * dout.astype(np.float64)).sum()), idx


def pin_backward_finite_differences(o):
    """For each input (x, W_g, all W1, all W3, all W2) and a random direction
    R: L(P + hR) - L(P - hR) equals <grad, (P + hR) - (P - hR)> up to third-
    order terms (L from the forward's exact output; the expert choice stays
    the same under the perturbation)."""
    rng = _rng(101)
    T, d, ffn, E, k = 5, 12, 20, 4, 2
    x, Wg, W1, W3, W2 = _rand_layer(rng, T, d, ffn, E)
    dout = rng.standard_normal((T, d)).astype(np.float32)
    g = o.moe_backward(x, Wg, W1, W3, W2, k, dout)
    grads = dict(x=g["dx"], Wg=g["dWg"], W1=np.stack(g["dW1"]), W3=np.stack(g["dW3"]),
                 W2=np.stack(g["dW2"]))
    params = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2)
    _, idx0 = _loss(o, x, Wg, W1, W3, W2, k, dout)
    # W_g acts only through the logits, which the forward stores as fp32: the
    # difference sees that rounding (~6e-8 absolute per logit), so it takes a
    # larger step and a looser bound than the other inputs
    steps = dict(x=(1e-3, 1e-5), Wg=(1e-2, 2e-4), W1=(1e-3, 1e-5), W3=(1e-3, 1e-5),
                 W2=(1e-3, 1e-5))
    for name, P in params.items():
        R = rng.standard_normal(P.shape).astype(np.float32)
        h, tol = steps[name]
        Pp = (P + np.float32(h) * R).astype(np.float32)
        Pm = (P - np.float32(h) * R).astype(np.float32)
        lp, idxp = _loss(o, **{**params, name: Pp}, k=k, dout=dout)
        lm, idxm = _loss(o, **{**params, name: Pm}, k=k, dout=dout)
        assert np.array_equal(idxp, idx0) and np.array_equal(idxm, idx0), name
        fd = lp - lm
        an = float((grads[name] * (Pp.astype(np.float64) - Pm.astype(np.float64))).sum())
        assert abs(fd - an) <= tol * abs(an) + 1e-10, (name, fd, an)


def pin_backward_matches_autograd(o):
    """torch float64 autograd of the layer written with torch ops (logits,
    softmax over the oracle's kept experts, SwiGLU experts, weighted sum)
    gives the same gradients for every input."""
    rng = _rng(102)
    T, d, ffn, E, k = 7, 10, 16, 5, 2
    x, Wg, W1, W3, W2 = _rand_layer(rng, T, d, ffn, E)
    dout = rng.standard_normal((T, d)).astype(np.float32)
    g = o.moe_backward(x, Wg, W1, W3, W2, k, dout)
    _, _, idx, _ = o.moe_forward(x, Wg, W1, W3, W2, k)
    tx, tg, t1, t3, t2 = (torch.tensor(a, dtype=torch.float64, requires_grad=True)
                          for a in (x, Wg, W1, W3, W2))
    logits = tx @ tg.T
    sel = torch.tensor(idx, dtype=torch.long)
    gates = torch.softmax(torch.gather(logits, 1, sel), dim=1)
    out = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            hid = torch.nn.functional.silu(t1[e] @ tx[t]) * (t3[e] @ tx[t])
            out[t] = out[t] + gates[t, j] * (t2[e] @ hid)
    (out * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    # the oracle's logits carry one fp32 rounding: agree to ~1e-7 relative
    for got, ref in ((g["dx"], tx.grad), (g["dWg"], tg.grad), (np.stack(g["dW1"]), t1.grad),
                     (np.stack(g["dW3"]), t3.grad), (np.stack(g["dW2"]), t2.grad)):
        ref = ref.numpy()
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-7 * np.abs(ref).max()), \
            float(np.abs(got - ref).max())


def pin_backward_router_properties(o):
    """The kept gates always sum to 1, so the logit gradients of a token sum
    to 0 and sum_e dW_g[e] = 0; with one expert and k = 1 the gate is the
    constant 1 and dW_g = 0; gradients are linear in dout (doubling dout
    doubles every gradient exactly)."""
    rng = _rng(103)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 9, 8, 12, 6)
    dout = rng.standard_normal((9, 8)).astype(np.float32)
    g = o.moe_backward(x, Wg, W1, W3, W2, 2, dout)
    assert np.abs(g["dWg"].sum(axis=0)).max() <= 1e-12 * max(1.0, np.abs(g["dWg"]).max())
    g2 = o.moe_backward(x, Wg, W1, W3, W2, 2, (2 * dout).astype(np.float32))
    for key in ("dx", "dWg"):
        assert np.array_equal(g2[key], 2 * g[key])
    for key in ("dW1", "dW3", "dW2"):
        assert all(np.array_equal(a, 2 * b) for a, b in zip(g2[key], g[key]))
    x1, Wg1, W11, W31, W21 = _rand_layer(rng, 6, 8, 12, 1)
    g1 = o.moe_backward(x1, Wg1, W11, W31, W21, 1, dout[:6])
    assert np.all(g1["dWg"] == 0.0)


def pin_backward_dtype_and_windows(o):
    """bf16 inputs give the same gradients as their exact fp32 copies; the
    weight-gradient row windows are slices of the full gradients."""
    rng = _rng(104)
    x, Wg, W1, W3, W2 = _rand_layer(rng, 6, 16, 24, 4)
    dout = rng.standard_normal((6, 16)).astype(np.float32)
    to_bf = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    to_f32 = lambda b: bf16_bits_to_f64(b).astype(np.float32)
    bx, bg, b1, b3, b2, bd = (to_bf(a) for a in (x, Wg, W1, W3, W2, dout))
    gb = o.moe_backward(bx, bg, list(b1), list(b3), list(b2), 2, bd)
    gf = o.moe_backward(to_f32(bx), to_f32(bg), list(to_f32(b1)), list(to_f32(b3)),
                        list(to_f32(b2)), 2, to_f32(bd))
    for key in ("dx", "dWg"):
        assert np.array_equal(gb[key], gf[key])
    for key in ("dW1", "dW3", "dW2"):
        assert all(np.array_equal(a, b) for a, b in zip(gb[key], gf[key]))
    gw = o.moe_backward(x, Wg, W1, W3, W2, 2, dout, rows1=(5, 11), rows2=(3, 9))
    gfull = o.moe_backward(x, Wg, W1, W3, W2, 2, dout)
    for e in range(4):
        assert np.array_equal(gw["dW1"][e], gfull["dW1"][e][5:11])
        assert np.array_equal(gw["dW3"][e], gfull["dW3"][e][5:11])
        assert np.array_equal(gw["dW2"][e], gfull["dW2"][e][3:9])


ALL = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
