"""Pre-norm MoE block (moe_block_forward): x <- x + MoE(RMSNorm(x)) with the
RMSNorm fused into the router and the grouping pass and the residual add into
the combine.  Checked bit for bit against the unfused chain (moe_add_rmsnorm,
moe_forward / moe_forward_ex, moe_add_rmsnorm), which computes the same
values in separate kernels, and against the oracle (needs a GPU)."""
import numpy as np
import pytest
import torch

import helpers
import oracle
from sparse_mixture_experts_58_b300 import inputs

pytestmark = pytest.mark.gpu

EPS = 1e-5


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


def unfused_block(moe, x, layer, k, **kw):
    """x <- x + MoE(RMSNorm(x)) from the separate entry points, in place."""
    xn = moe.add_rmsnorm(x, eps=EPS)
    out = moe.forward(xn, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias, **kw)
    moe.add_rmsnorm(x, out, eps=EPS)
    return x


def bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("T,d,ffn,E,k,dtype", [
    (1, 128, 448, 8, 2, "bf16"),
    (16, 256, 448, 8, 2, "bf16"),
    (37, 192, 320, 5, 2, "bf16"),      # odd token count: a router block with one token
    (300, 256, 512, 8, 2, "bf16"),
    (700, 192, 384, 8, 2, "bf16"),     # CTA-pair expert GEMMs
    (1500, 128, 192, 4, 3, "bf16"),
    (65, 128, 448, 8, 2, "f32"),
    (33, 64, 96, 3, 1, "f32"),
])
def test_block_equals_unfused_chain(moe, T, d, ffn, E, k, dtype):
    x0, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=T + 11, device="cuda")
    a, b = x0.clone(), x0.clone()
    unfused_block(moe, a, layer, k)
    moe.block_forward(b, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias, eps=EPS)
    torch.cuda.synchronize()
    assert not torch.equal(bits(a), bits(x0))
    assert torch.equal(bits(a), bits(b))


@pytest.mark.parametrize("kw", [
    dict(gating=1),
    dict(capacity=40, drop_policy=0),
    dict(capacity=40, drop_policy=1),
], ids=["softmax_then_topk", "capacity_lose", "capacity_renorm"])
def test_block_routing_variants_equal_unfused_chain(moe, kw):
    T, d, ffn, E, k = 200, 256, 512, 8, 2
    x0, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=5, device="cuda",
                                     bias=inputs.SKEW_BIAS)
    a, b = x0.clone(), x0.clone()
    unfused_block(moe, a, layer, k, **kw)
    moe.block_forward(b, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias, eps=EPS,
                      **kw)
    torch.cuda.synchronize()
    assert torch.equal(bits(a), bits(b))


def test_block_stack_equals_unfused_chain(moe):
    """The token-count sweep's stack (32 layers of the Mixtral shape with
    independent weights, T = 32) through fused blocks gives the unfused
    chain's residual stream bit for bit after every layer."""
    cfg = inputs.WORKLOADS["sweep"]
    T, d, ffn, E, k = 32, cfg["d"], cfg["ffn"], cfg["E"], cfg["k"]
    x0 = inputs.sweep_tokens(T, d, device="cuda")
    a, b = x0.clone(), x0.clone()
    for l in range(cfg["layers"]):
        layer = inputs.sweep_layer(l, d, ffn, E, device="cuda")
        unfused_block(moe, a, layer, k)
        moe.block_forward(b, layer.Wg, layer.W1, layer.W3, layer.W2, k, eps=EPS)
        torch.cuda.synchronize()
        assert torch.equal(bits(a), bits(b)), f"layer {l}"
        del layer


def test_block_against_oracle(moe):
    """The fused block against the oracle's RMSNorm, layer and residual add on
    every token: the error beyond the block's two roundings (the layer output,
    then the sum, half an ulp each) is within the layer's bf16 tolerance of
    the layer output's RMS."""
    T, d, ffn, E, k = 48, 256, 512, 8, 2
    x0, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=21, device="cuda")
    o = oracle.load()
    xh = inputs.to_host(x0)
    xn_ref = o.rmsnorm(xh, EPS)
    exact, rl, _, _ = helpers.oracle_on_rows(inputs.from_host(xn_ref, "cuda"), layer, k)
    x = x0.clone()
    moe.block_forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, eps=EPS)
    torch.cuda.synchronize()
    got = helpers.host_f64(inputs.to_host(x))
    ref = helpers.host_f64(xh) + exact
    excess = np.abs(got - ref) - helpers.bf16_half_ulp(got) - helpers.bf16_half_ulp(exact)
    keep = ~helpers.near_tie_mask(rl, k)
    err = max(float(excess[keep].max()), 0.0) / float(np.sqrt((exact ** 2).mean()))
    print(f"block vs oracle: {err:.3e} over {keep.sum()} tokens")
    assert keep.mean() > 0.9
    assert err <= helpers.TOL_BF16
