"""Randomised parity: seeded layers of random shape (tokens 1..3000, hidden
and expert widths, 2..64 experts, top-1..8, both gatings, bf16 and fp32) run
through moe_forward under random tile plans (CTA pairs on or off, token tile
heights and slots, contraction splits, gate/up halves, the two-box or
interleaved gate/up layout, balanced grids, the streaming router, the folded
combine, one- or two-kernel grouping), each against the oracle, and each
called twice (the second call through the launch-graph cache) with the same
bits."""
import numpy as np
import pytest
import torch

import helpers
import oracle
from sparse_mixture_experts_58_b300 import inputs

pytestmark = pytest.mark.gpu

N_CASES = 160


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from sparse_mixture_experts_58_b300 import moe as m
    return m


@pytest.fixture(autouse=True)
def _status_clean(moe):
    moe.device_status(clear=True)
    yield
    assert moe.device_status(clear=True) == 0, "a kernel's bounded wait expired"


def _case(i):
    """The i-th random configuration: shape, routing and plan switches."""
    rng = np.random.default_rng(1000 + i)
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    band = rng.random()
    T = int(rng.integers(1, 9) if band < 0.25 else
            rng.integers(9, 201) if band < 0.5 else
            rng.integers(201, 1201) if band < 0.85 else rng.integers(1201, 3001))
    if dtype == "bf16":
        d = 64 * int(rng.integers(1, 17))
        ffn = 64 * int(rng.integers(1, 13))
    else:
        d = 4 * int(rng.integers(8, 65))
        ffn = 4 * int(rng.integers(8, 129))
    E = int(rng.integers(2, 17)) if rng.random() < 0.85 else int(rng.integers(17, 65))
    k = 2 if rng.random() < 0.6 else int(rng.integers(1, min(E, 8) + 1))
    gating = 1 if rng.random() < 0.25 else 0
    knobs = {}
    for name, values in (("MOE_PLAN_PAIR", ("0", "1")),
                         ("MOE_PLAN_BM", tuple(str(8 * j) for j in range(1, 17))),
                         ("MOE_PLAN_SPLITS", ("1", "2", "3", "4")),
                         ("MOE_PLAN_GSPLIT", ("0", "1")),
                         ("MOE_ROUTER_WIDE", ("0", "1")),
                         ("MOE_FUSE_COMBINE", ("0",)),
                         ("MOE_ROUTE_SMALL", ("0", "1")),
                         ("MOE_PAIR_IL", ("0",)),
                         ("MOE_PAIR_BALANCE", ("0",)),
                         ("MOE_TC_NARROW", ("0",))):
        if rng.random() < 0.35:
            knobs[name] = str(rng.choice(values))
    return dict(T=T, d=d, ffn=ffn, E=E, k=k, dtype=dtype, gating=gating, knobs=knobs,
                seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_layer_against_oracle(moe, monkeypatch, i):
    c = _case(i)
    for name, v in c["knobs"].items():
        monkeypatch.setenv(name, v)
    T, d, ffn, E, k, dtype = c["T"], c["d"], c["ffn"], c["E"], c["k"], c["dtype"]
    x, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=c["seed"], device="cuda")
    outs = [moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias,
                        gating=c["gating"]).clone() for _ in range(2)]
    torch.cuda.synchronize()
    view = torch.int16 if dtype == "bf16" else torch.int32
    label = f"case {i}: {c}"
    assert torch.equal(outs[0].view(view), outs[1].view(view)), label
    Wg, W1, W3, W2, bias = inputs.layer_to_host(layer)
    _, rl, _, _, exact = oracle.load().moe_forward(inputs.to_host(x), Wg, W1, W3, W2, k,
                                                   bias=bias, exact=True, gating=c["gating"])
    keep = ~helpers.near_tie_mask(rl, k)
    err = helpers.rel_error(inputs.to_host(outs[0])[keep], exact[keep], dtype)
    print(f"PARITY {label}: gated {err:.3e} over {keep.sum()} tokens, {(~keep).sum()} near ties")
    assert keep.mean() > 0.8, label
    assert err <= helpers.tol(dtype), (label, err)


EPS = 1e-5


@pytest.mark.parametrize("i", range(48))
def test_random_block_equals_unfused_chain(moe, monkeypatch, i):
    """The pre-norm block x <- x + MoE(RMSNorm(x)) (moe_block_forward: the
    RMSNorm fused into the router and the grouping, the residual into the
    combine) against the same block from the separate entry points
    (add_rmsnorm, forward, add_rmsnorm), bit for bit, over random shapes,
    routings and tile plans."""
    c = _case(10_000 + i)
    for name, v in c["knobs"].items():
        monkeypatch.setenv(name, v)
    T, d, ffn, E, k, dtype = c["T"], c["d"], c["ffn"], c["E"], c["k"], c["dtype"]
    x0, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=c["seed"], device="cuda")
    a, b = x0.clone(), x0.clone()
    xn = moe.add_rmsnorm(a, eps=EPS)
    out = moe.forward(xn, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias,
                      gating=c["gating"])
    moe.add_rmsnorm(a, out, eps=EPS)
    moe.block_forward(b, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias, eps=EPS,
                      gating=c["gating"])
    torch.cuda.synchronize()
    view = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(a.view(view), b.view(view)), f"case {10_000 + i}: {c}"


@pytest.mark.parametrize("i", range(24))
def test_random_host_io_equals_device_path(moe, i):
    """moe_forward_host_io with page-locked host tokens and output (the router
    reading the rows over the bus below 1536 tokens, the last kernel writing
    the output into host memory) gives the device path's bits, over random
    shapes, dtypes and expert counts, on repeated calls."""
    c = _case(20_000 + i)
    T, d, ffn, E, k, dtype = c["T"], c["d"], c["ffn"], c["E"], c["k"], c["dtype"]
    x, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=c["seed"], device="cuda")
    ref = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias).cpu()
    xh = x.cpu().pin_memory()
    view = torch.int16 if dtype == "bf16" else torch.int32
    for _ in range(2):
        oh = torch.empty_like(xh, pin_memory=True)
        oh.fill_(0)
        moe.forward_host_io(xh, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias,
                            out_host=oh)
        torch.cuda.synchronize()
        assert torch.equal(oh.view(view), ref.view(view)), f"case {20_000 + i}: {c}"
