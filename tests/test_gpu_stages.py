"""Stage-by-stage parity of the CUDA path through the C ABI (needs a GPU).

Router and grouping against the oracle; the grouped expert GEMMs against a
plain torch fp32 evaluation of the same rows (a debugging aid: the layer
tests compare everything against the oracle)."""
import numpy as np
import pytest
import torch

import helpers
import oracle
from sparse_mixture_experts_58_b300 import inputs

pytestmark = pytest.mark.gpu


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


def _logits_with_ties(T, E, seed):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[::3] = (np.round(l[::3] * 2) / 2).astype(np.float32)   # many exact ties
    l[5::7, :] = 0.0                                           # all-equal rows
    return l


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (16, 8, 2), (17, 8, 2), (300, 8, 2), (4096, 8, 2),
                                   (1000, 3, 1), (257, 32, 2), (64, 2, 2), (50, 1, 1),
                                   (16384, 8, 2),
                                   (20000, 64, 8)])   # chunk counts too large for shared memory
def test_route_from_logits_bit_exact(moe, T, E, k):
    l = _logits_with_ties(T, E, seed=T * 31 + E)
    idx, gates, counts, offsets, perm, inv = moe.route_from_logits(torch.from_numpy(l).cuda(), k)
    torch.cuda.synchronize()
    o = oracle.load()
    ridx, rg, rcounts, roffsets, rperm, rinv = o.route(l, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.array_equal(counts.cpu().numpy(), rcounts)
    assert np.array_equal(offsets.cpu().numpy(), roffsets)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.allclose(gates.cpu().numpy(), rg, rtol=0, atol=2e-7)


def test_route_empty(moe):
    idx, gates, counts, offsets, perm, inv = moe.route_from_logits(
        torch.zeros(0, 8, device="cuda"), 2)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and offsets.abs().sum().item() == 0


@pytest.mark.parametrize("name,T", [("tiny", 64), ("decode", 16), ("prefill", 512)])
def test_router_matches_oracle(moe, name, T):
    x, layer = inputs.make_named(name, device="cuda", T=T)
    k = layer.meta["k"]
    logits, idx, gates = moe.router(x, layer.Wg, k, layer.bias)
    torch.cuda.synchronize()
    o = oracle.load()
    rl, ridx, rg = o.router(inputs.to_host(x), inputs.to_host(layer.Wg), k)
    assert np.allclose(logits.cpu().numpy(), rl, rtol=1e-5, atol=1e-5)
    keep = ~helpers.near_tie_mask(rl, k)
    assert np.array_equal(idx.cpu().numpy()[keep], ridx[keep])
    assert np.allclose(gates.cpu().numpy()[keep], rg[keep], atol=2e-5)


@pytest.mark.parametrize("E,k,Ts", [(8, 2, (1, 16, 1500, 2400, 4096)), (64, 8, (3, 16, 1200))])
def test_router_logits_do_not_depend_on_batch(moe, E, k, Ts):
    """A token's logits, selection and gates are the same bits whether it is
    routed alone, in a small batch or in a large one: the router takes 2, 4
    or 8 tokens per block by batch size but sums every token's products in
    the same order."""
    x, layer = inputs.make_workload(max(Ts), 4096, 64, E, k, "bf16", seed=E, device="cuda")
    full = moe.router(x, layer.Wg, k)
    for T in Ts:
        part = moe.router(x[:T].contiguous(), layer.Wg, k)
        torch.cuda.synchronize()
        for a, b in zip(full, part):
            assert torch.equal(a[:T], b), T


def test_router_skew_bias(moe):
    x, layer = inputs.make_named("skewed", device="cuda", T=1024)
    logits, idx, gates = moe.router(x, layer.Wg, 2, layer.bias)
    torch.cuda.synchronize()
    o = oracle.load()
    rl, ridx, rg = o.router(inputs.to_host(x), inputs.to_host(layer.Wg), 2,
                            bias=layer.bias.cpu().numpy())
    keep = ~helpers.near_tie_mask(rl, 2)
    assert np.array_equal(idx.cpu().numpy()[keep], ridx[keep])
    share = np.bincount(ridx.ravel(), minlength=8) / ridx.size
    assert share[0] > 0.3 and share[7] < 0.01      # experts 0-1 get most rows


@pytest.mark.parametrize("dtype,d", [("bf16", 4096), ("f32", 128), ("bf16", 64)])
def test_permute_exact(moe, dtype, d):
    T, k = 37, 2
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(T, d, device="cuda", generator=g).to(inputs.TORCH_DTYPE[dtype])
    perm = torch.randperm(T * k, device="cuda", generator=g).to(torch.int32)
    xp = moe.permute(x, perm, k)
    torch.cuda.synchronize()
    ref = x[(perm.long() // k)]
    assert torch.equal(xp.view(torch.int16 if dtype == "bf16" else torch.int32),
                       ref.view(torch.int16 if dtype == "bf16" else torch.int32))


def _grouped_case(T, d, ffn, E, dtype, seed, skew=False):
    x, layer = inputs.make_workload(T, d, ffn, E, 2, dtype, seed, "cuda",
                                    bias=(inputs.SKEW_BIAS if skew else None))
    return x, layer


def _torch_swiglu_rows(x_perm, offsets, W1, W3):
    xp = x_perm.float()
    h = torch.empty(xp.shape[0], W1.shape[1], device=xp.device)
    off = offsets.cpu().tolist()
    for e in range(W1.shape[0]):
        a, b = off[e], off[e + 1]
        if b > a:
            u = xp[a:b] @ W1[e].float().T
            v = xp[a:b] @ W3[e].float().T
            h[a:b] = torch.nn.functional.silu(u) * v
    return h


@pytest.mark.parametrize("T,d,ffn,E,skew", [
    (16, 256, 448, 8, False),      # narrow tiles, ragged last column tile
    (200, 128, 256, 4, False),     # 100 rows per expert: narrow, several row tiles
    (700, 192, 384, 8, False),     # wide tiles (175 rows/expert), ragged rows
    (1024, 256, 512, 8, True),     # skewed: one expert with many row tiles
    (5, 64, 64, 8, False),         # several experts empty
    (2300, 192, 320, 8, False),    # pairs: several token tiles per expert, ragged features
])
@pytest.mark.parametrize("pair", [None, "0", "1"], ids=["auto", "one_cta", "pair"])
def test_grouped_gemms_against_torch(moe, monkeypatch, T, d, ffn, E, skew, pair):
    """Both expert GEMMs against torch on the GPU's own permuted rows, under
    the automatic tile plan and with the CTA-pair kernel forced off and on."""
    if pair is not None:
        monkeypatch.setenv("MOE_PLAN_PAIR", pair)
    x, layer = _grouped_case(T, d, ffn, E, "bf16", seed=T, skew=skew)
    logits, idx, gates = moe.router(x, layer.Wg, 2, layer.bias)
    idx2, gates2, counts, offsets, perm, inv = moe.route_from_logits(logits, 2)
    xp = moe.permute(x, perm, 2)
    h = moe.expert_swiglu(xp, offsets, layer.W1, layer.W3)
    y = moe.expert_down(h, offsets, layer.W2, T, 2)
    out = moe.combine(y, gates2, inv, T, 2, torch.bfloat16)
    torch.cuda.synchronize()
    href = _torch_swiglu_rows(xp, offsets, layer.W1, layer.W3)
    scale = href.pow(2).mean().sqrt().item()
    # h is stored in bf16: each element is within half a bf16 ulp (2^-9
    # relative) of its fp32 value, plus accumulation-order differences
    bound = href.abs() * 2.0 ** -8 + 1e-3 * scale
    assert ((h.float() - href).abs() <= bound).all(), (h.float() - href).abs().max().item()
    # down projection from the GPU's own h
    yref = torch.empty(h.shape[0], d, device="cuda")
    off = offsets.cpu().tolist()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            yref[a:b] = h[a:b].float() @ layer.W2[e].float().T
    ysum = y.sum(0)
    yscale = yref.pow(2).mean().sqrt().item()
    assert (ysum - yref).abs().max().item() <= 1e-3 * yscale + 1e-6
    oref = torch.zeros(T, d, device="cuda")
    for j in range(2):
        oref += gates2[:, j:j + 1] * ysum[inv.view(T, 2)[:, j].long()]
    obound = oref.abs() * 2.0 ** -8 + 1e-4 * oref.pow(2).mean().sqrt().item()
    assert ((out.float() - oref).abs() <= obound).all()


def test_wait_timeout_selftest(moe):
    """A bounded wait that nothing satisfies gives up, reports, and leaves the
    context usable."""
    moe.selftest_wait_timeout(2_000_000)
    assert moe.device_status(clear=True) == 5
    a = torch.ones(1024, device="cuda")
    assert a.sum().item() == 1024.0
    assert moe.device_status(clear=True) == 0


@pytest.mark.parametrize("T,d,E", [(7, 4096, 8), (600, 512, 3), (1500, 4096, 8),
                                   (4096, 4096, 8), (2500, 1024, 5), (3001, 2048, 8),
                                   (16383, 4096, 8)])
def test_wide_router_same_bits(moe, monkeypatch, T, d, E):
    """The streaming large-batch router (each compute thread's slices of the
    router rows in registers, groups of four token rows brought in by bulk
    copies through a ring of stages by one warp, the eight compute warps'
    sums selected by another, products as packed fp32x2 FMAs) sums in
    router_kernel's order: the same logits, choices and gates bit for bit,
    and the same pre-norm block (the fused RMSNorm's scales included).  The
    shapes cover fewer groups than SMs, a ragged last group and many trips
    around the ring."""
    x, layer = inputs.make_workload(T, d, 128, E, 2, "bf16", seed=T, device="cuda",
                                    bias=inputs.SKEW_BIAS[:E] if E == 8 else None)
    res = {}
    for wide in ("0", "1"):
        monkeypatch.setenv("MOE_ROUTER_WIDE", wide)
        lg, idx, g = moe.router(x, layer.Wg, 2, layer.bias)
        xb = x.clone()
        moe.block_forward(xb, layer.Wg, layer.W1, layer.W3, layer.W2, 2, bias=layer.bias)
        torch.cuda.synchronize()
        res[wide] = (lg.clone(), idx.clone(), g.clone(), xb)
    a, b = res["0"], res["1"]
    assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32))
    assert torch.equal(a[1], b[1])
    assert torch.equal(a[2].view(torch.int32), b[2].view(torch.int32))
    assert torch.equal(a[3].view(torch.int16), b[3].view(torch.int16))


@pytest.mark.parametrize("E,k,gating", [(8, 1, 0), (8, 3, 0), (8, 8, 0), (8, 2, 1), (4, 3, 1),
                                        (6, 2, 0)])
def test_wide_router_selection_variants(moe, monkeypatch, E, k, gating):
    """The streaming router's selection (one lane per (token, expert) adds the
    warps' sums and the bias; the token's logits, gathered in registers, go
    through the same top-k and gate arithmetic as router_kernel's) for k from
    1 to 8 and both gatings (softmax over the kept logits, or over all E):
    the same logits, choices, gates and layer output bit for bit."""
    T, d, ffn = 650, 256, 128   # 650 tokens: the last group of four holds two
    bias = inputs.SKEW_BIAS[:E] if E == 8 else None
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=10 * E + k, device="cuda",
                                    bias=bias)
    res = {}
    for wide in ("0", "1"):
        monkeypatch.setenv("MOE_ROUTER_WIDE", wide)
        routed = None
        if gating == 0:
            lg, idx, g = moe.router(x, layer.Wg, k, layer.bias)
            routed = (lg.clone(), idx.clone(), g.clone())
        out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias,
                          gating=gating)
        torch.cuda.synchronize()
        res[wide] = (routed, out.clone())
    (ra, oa), (rb, ob) = res["0"], res["1"]
    if ra is not None:
        assert torch.equal(ra[0].view(torch.int32), rb[0].view(torch.int32))
        assert torch.equal(ra[1], rb[1])
        assert torch.equal(ra[2].view(torch.int32), rb[2].view(torch.int32))
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert moe.device_status(clear=True) == 0
