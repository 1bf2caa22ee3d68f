"""Whole-layer parity: moe_forward (CUDA, through the C ABI) against the CPU
oracle on the same seeded inputs (needs a GPU).

Small shapes are compared element by element on every token; the Mixtral
shapes at their full token counts, in the launch configuration the benchmark
times, are compared on every token (decode) or on a seeded sample of tokens
the oracle computes one by one (prefill, skewed, stacked layers).  Tokens
whose top-(k+1) oracle logits are within 1e-3 of each other are left out and
counted."""
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


def check_layer(moe, x, layer, k, rows=None, dtype=None, label="", exclude_ties=True):
    dtype = dtype or layer.meta["dtype"]
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias)
    torch.cuda.synchronize()
    ref, rl, ridx, _ = helpers.oracle_on_rows(x, layer, k, rows)
    got = inputs.to_host(out if rows is None else
                         out[torch.as_tensor(rows, device=out.device, dtype=torch.long)])
    keep = ~helpers.near_tie_mask(rl, k) if exclude_ties else np.ones(len(rl), bool)
    err = helpers.rel_error(got[keep], ref[keep], dtype)
    raw = helpers.raw_rel_error(got[keep], ref[keep])
    print(f"PARITY {label}: gated {err:.3e} raw max|d|/rms {raw:.3e} over {keep.sum()} tokens, "
          f"{(~keep).sum()} near ties")
    assert err <= helpers.tol(dtype), (label, err)
    assert keep.mean() > 0.9
    return out, ref, keep


# ---- small shapes, every token --------------------------------------------

def test_tiny_fp32_config(moe):
    """T=64, d=128, ffn=448, E=8, top-2, fp32."""
    x, layer = inputs.make_named("tiny", device="cuda")
    check_layer(moe, x, layer, 2, label="tiny")


@pytest.mark.parametrize("T,d,ffn,E,k,dtype", [
    (1, 128, 448, 8, 2, "bf16"),
    (3, 256, 192, 8, 2, "bf16"),
    (16, 256, 448, 8, 2, "bf16"),
    (37, 192, 320, 5, 2, "bf16"),
    (129, 128, 256, 8, 2, "bf16"),      # first size with 128-row tiles
    (700, 192, 384, 8, 2, "bf16"),      # wide tiles, ragged row and column tiles
    (600, 128, 256, 8, 1, "bf16"),      # k = 1
    (256, 128, 192, 2, 2, "bf16"),      # E = k = 2: every token uses both experts
    (100, 64, 64, 1, 1, "bf16"),        # E = 1: one dense SwiGLU FFN
    (65, 128, 448, 8, 2, "f32"),
    (33, 64, 96, 3, 1, "f32"),
    (256, 64, 64, 32, 2, "bf16"),       # 32 experts, many nearly empty
])
def test_small_layers(moe, T, d, ffn, E, k, dtype):
    x, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=T + d, device="cuda")
    check_layer(moe, x, layer, k, dtype=dtype, label=f"T{T} d{d} ffn{ffn} E{E} k{k} {dtype}")


@pytest.mark.parametrize("T,d,ffn,E,k", [
    (16, 256, 448, 8, 2),
    (129, 128, 256, 8, 2),
    (700, 192, 384, 8, 2),
    (1500, 128, 192, 4, 3),
])
@pytest.mark.parametrize("pair", ["0", "1"], ids=["one_cta", "pair"])
def test_small_layers_forced_tile_plan(moe, monkeypatch, T, d, ffn, E, k, pair):
    """The whole layer with the CTA-pair GEMMs forced off and on, on shapes
    the automatic plan sends to the other kernel as well."""
    monkeypatch.setenv("MOE_PLAN_PAIR", pair)
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=T + 7, device="cuda")
    check_layer(moe, x, layer, k, dtype="bf16", label=f"T{T} E{E} k{k} pair={pair}")


@pytest.mark.parametrize("splits", ["2", "3", "4", "8", "16"])
@pytest.mark.parametrize("pair", ["0", "1"], ids=["one_cta", "pair"])
def test_forced_down_splits(moe, monkeypatch, splits, pair):
    """Split-K down projection with every combine shape (2, 3-4 and more
    partials per row, and two batches of 8) on both GEMM kernels."""
    monkeypatch.setenv("MOE_PLAN_PAIR", pair)
    monkeypatch.setenv("MOE_PLAN_SPLITS", splits)
    T, d, ffn, E, k = 300, 256, 1024, 8, 2
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=int(splits), device="cuda")
    assert moe.down_splits(T, d, ffn, E, k, moe.BF16) == int(splits)
    check_layer(moe, x, layer, k, dtype="bf16", label=f"splits={splits} pair={pair}")


@pytest.mark.parametrize("bm", ["8", "16", "24", "32", "64", "72", "96", "128"])
def test_forced_token_tile(moe, monkeypatch, bm):
    """The one-CTA GEMMs at every token tile height (token slots of 16, 32, 64,
    96 and 128 rows in shared memory), on a batch whose experts span several
    tiles at the small heights."""
    monkeypatch.setenv("MOE_PLAN_BM", bm)
    T, d, ffn, E, k = 150, 256, 448, 8, 2
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=int(bm), device="cuda")
    check_layer(moe, x, layer, k, dtype="bf16", label=f"token tile {bm}")


@pytest.mark.parametrize("T,d,ffn,E,k", [
    (1, 256, 448, 8, 2),
    (2, 256, 448, 8, 2),
    (3, 128, 320, 8, 2),        # ffn = 320: the last 56-feature tile holds 40
    (3, 512, 1024, 4, 2),
    (1, 4096, 14336, 8, 2),     # Mixtral shape, one token
])
@pytest.mark.parametrize("gsplit", ["0", "1"], ids=["whole", "halves"])
def test_gate_up_halves_for_the_smallest_batches(moe, monkeypatch, T, d, ffn, E, k, gsplit):
    """The gate/up contraction in two halves for the smallest batches (fp32
    partial sums; the later half of each tile adds them in split order and
    applies the SwiGLU) and whole, against the oracle; repeated calls give
    the same bits whichever half of a tile finishes last."""
    monkeypatch.setenv("MOE_PLAN_GSPLIT", gsplit)
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=T + 31, device="cuda")
    check_layer(moe, x, layer, k, dtype="bf16", label=f"T{T} d{d} ffn{ffn} gsplit={gsplit}")
    outs = [moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert moe.device_status(clear=True) == 0


def test_empty_batch(moe):
    x, layer = inputs.make_workload(0, 128, 256, 8, 2, "bf16", 0, "cuda")
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    torch.cuda.synchronize()
    assert out.shape == (0, 128)


def test_zero_router_picks_first_two(moe):
    """W_g = 0: every logit ties, so experts 0 and 1 with gates 1/2 each."""
    x, layer = inputs.make_workload(40, 128, 256, 8, 2, "bf16", 5, "cuda")
    layer.Wg.zero_()
    logits, idx, gates = moe.router(x, layer.Wg, 2)
    torch.cuda.synchronize()
    assert (idx[:, 0] == 0).all() and (idx[:, 1] == 1).all()
    assert (gates == 0.5).all()
    # exact ties: both sides apply the same rule, nothing to exclude
    check_layer(moe, x, layer, 2, dtype="bf16", label="zero router", exclude_ties=False)


def test_identical_experts_equal_dense_ffn(moe):
    x, layer = inputs.make_workload(64, 128, 256, 8, 2, "f32", 6, "cuda")
    layer.W1[:] = layer.W1[0]
    layer.W3[:] = layer.W3[0]
    layer.W2[:] = layer.W2[0]
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    torch.cuda.synchronize()
    u = x.double() @ layer.W1[0].double().T
    v = x.double() @ layer.W3[0].double().T
    dense = (torch.nn.functional.silu(u) * v) @ layer.W2[0].double().T
    err = (out.double() - dense).abs().max() / dense.abs().max()
    assert err.item() <= 1e-4


def test_duplicates_and_permutation(moe):
    """Duplicated tokens give bit-identical rows; permuting tokens permutes
    the output rows bit for bit."""
    x, layer = inputs.make_workload(300, 128, 256, 8, 2, "bf16", 7, "cuda")
    x[10] = x[200]
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    p = torch.randperm(300, device="cuda")
    outp = moe.forward(x[p].contiguous(), layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    torch.cuda.synchronize()
    assert torch.equal(out[10].view(torch.int16), out[200].view(torch.int16))
    assert torch.equal(outp.view(torch.int16), out[p].view(torch.int16))


def test_deterministic(moe):
    x, layer = inputs.make_workload(500, 128, 256, 8, 2, "bf16", 8, "cuda")
    a = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    b = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_host_io_matches_device_path(moe):
    x, layer = inputs.make_workload(48, 256, 512, 8, 2, "bf16", 9, "cuda")
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    xh = x.cpu().pin_memory()
    oh = moe.forward_host_io(xh, layer.Wg, layer.W1, layer.W3, layer.W2, 2)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), out.cpu().view(torch.int16))


# ---- the Mixtral shape (hidden 4096, expert width 14336, 8 experts, top-2) --

@pytest.fixture(scope="module")
def decode_case():
    return inputs.make_named("decode", device="cuda")


def test_decode_config_all_tokens(moe, decode_case):
    x, layer = decode_case
    check_layer(moe, x, layer, 2, label="decode T=16")


@pytest.mark.parametrize("T", [1, 3, 4, 5])
def test_decode_weights_few_tokens(moe, decode_case, T):
    """The decode layer's weights with 1, 3, 4 and 5 tokens: two to ten expert
    rows, most experts idle, token tiles of 8 rows (the gate/up contraction
    in halves where the kernel takes them: one token, two busy experts)."""
    x, layer = decode_case
    check_layer(moe, x[:T].contiguous(), layer, 2, label=f"decode weights T={T}")


def _layout_sample(x, layer, k, per_expert, seed, must=(), row_tiles=()):
    """Tokens to compare, chosen from the oracle's grouping of the whole
    batch: every expert's first and last grouped rows, the edges and CTA
    halves of its token tiles, and at least `per_expert` rows per expert."""
    host = inputs.layer_to_host(layer)
    _, idx, offsets, perm = helpers.oracle_layout(inputs.to_host(x), host, k)
    rows = helpers.layout_rows(idx, offsets, perm, k, per_expert=per_expert, seed=seed,
                               must=must, row_tiles=row_tiles)
    return rows, host, idx


def test_prefill_config_sampled(moe):
    """Prefill T=4096: the tokens at every expert's grouped-layout edges and
    tile edges, and at least 32 rows per expert."""
    x, layer = inputs.make_named("prefill", device="cuda")
    rows, host, idx = _layout_sample(x, layer, 2, per_expert=32, seed=1)
    for e in range(layer.E):
        assert (idx[rows] == e).any(1).sum() >= 32
    check_layer(moe, x, layer, 2, rows=rows, label=f"prefill T=4096 ({len(rows)} layout rows)")
    del x, layer
    torch.cuda.empty_cache()


def test_mixtral_shape_96_row_token_tiles(moe):
    """T=256 at the Mixtral shape: 64 rows per expert on average, at most
    about 80, so the one-CTA GEMMs take 96-row token tiles (8 ring stages);
    every expert's layout edges and at least 16 rows per expert."""
    T = 256
    x, layer = inputs.make_workload(T, 4096, 14336, 8, 2, "bf16", seed=T, device="cuda")
    assert moe.down_splits(T, 4096, 14336, 8, 2, moe.BF16) == 1
    rows, host, idx = _layout_sample(x, layer, 2, per_expert=16, seed=3)
    check_layer(moe, x, layer, 2, rows=rows, label=f"T=256 ({len(rows)} layout rows)")
    del x, layer
    torch.cuda.empty_cache()


def test_skewed_config_sampled(moe):
    """Skewed routing T=8192: layout edges of every expert (expert 0 holds
    about 43% of the rows, expert 7 a handful), duplicate pairs, and at least
    16 rows per expert (all of them for the rarest)."""
    x, layer = inputs.make_named("skewed", device="cuda")
    dst, src = layer.meta["dups"]
    must = list(dst[:12]) + list(src[:12])
    rows, host, idx = _layout_sample(x, layer, 2, per_expert=16, seed=2, must=must)
    out, ref, keep = check_layer(moe, x, layer, 2, rows=rows,
                                 label=f"skewed T=8192 ({len(rows)} layout rows)")
    # exact duplicates give bit-identical outputs
    o = out[torch.as_tensor(dst, device="cuda")].view(torch.int16)
    s = out[torch.as_tensor(src, device="cuda")].view(torch.int16)
    assert torch.equal(o, s)
    counts = np.bincount(idx.flatten(), minlength=8)
    assert counts[0] > 5 * counts[2] and counts.sum() == 2 * 8192
    for e in range(8):
        assert (idx[rows] == e).any(1).sum() >= min(16, counts[e])
    del x, layer
    torch.cuda.empty_cache()


def test_stacked_layers_sampled(moe):
    """Token-count sweep workload: x <- x + MoE(RMSNorm(x)) through 32 layers
    with independent weights.  Per layer, the GPU's own layer input is given
    to the oracle for a few sampled tokens (T = 32, every layer); the RMSNorm
    and residual steps are checked against the oracle too."""
    cfg = inputs.WORKLOADS["sweep"]
    T, d, ffn, E, k = 32, cfg["d"], cfg["ffn"], cfg["E"], cfg["k"]
    o = oracle.load()
    x = inputs.sweep_tokens(T, d, device="cuda")
    rows = helpers.sample_rows(T, 3, seed=3)
    worst = 0.0
    for l in range(cfg["layers"]):
        layer = inputs.sweep_layer(l, d, ffn, E, device="cuda")
        x_before = x.clone()
        xn = moe.add_rmsnorm(x)
        out = moe.forward(xn, layer.Wg, layer.W1, layer.W3, layer.W2, k)
        torch.cuda.synchronize()
        assert torch.equal(x.view(torch.int16), x_before.view(torch.int16))
        ref_xn = o.rmsnorm(inputs.to_host(x), 1e-5)
        assert helpers.rel_error(inputs.to_host(xn), ref_xn, "bf16") <= 1e-2
        ref, rl, _, _ = helpers.oracle_on_rows(xn, layer, k, rows)
        got = inputs.to_host(out[torch.as_tensor(rows, device="cuda")])
        keep = ~helpers.near_tie_mask(rl, k)
        if keep.any():
            err = helpers.rel_error(got[keep], ref[keep], "bf16")
            worst = max(worst, err)
            assert err <= helpers.TOL_BF16, (l, err)
        # residual: x <- x + out, checked against the oracle's add
        x_host, out_host = inputs.to_host(x), inputs.to_host(out)
        moe.add_rmsnorm(x, out)
        torch.cuda.synchronize()
        assert np.array_equal(inputs.to_host(x).view(np.uint16), o.add(x_host, out_host)) or \
            helpers.rel_error(inputs.to_host(x), o.add(x_host, out_host), "bf16") <= 1e-2
        del layer
    print(f"stacked layers: worst per-layer rel err {worst:.3e}")


# Token-count sweep at the Mixtral shape: the layers each token count is
# checked at (the chain runs all 32).
SWEEP_CHECK = {1: (0, 1, 15, 31), 1024: (0, 1, 31), 16384: (0, 31)}
EPS = 1e-5


def test_sweep_blocks_mixtral_shape(moe):
    """The token-count sweep workload as the benchmark times it: 32 pre-norm
    blocks x <- x + MoE(RMSNorm(x)) (moe_block_forward, RMSNorm fused into the
    router and the grouping, residual into the combine) with independent
    weights at hidden 4096, expert width 14336, 8 experts, top-2, for T = 1,
    1024 and 16384.  At the checked layers the oracle gets the GPU's own
    layer input: its RMSNorm, its layer (every token at T = 1, layout rows
    otherwise) and the residual add.  The error beyond the block's two
    roundings (the layer output, then the sum: half an ulp each) must be
    within the bf16 bar of the layer output's RMS."""
    cfg = inputs.WORKLOADS["sweep"]
    d, ffn, E, k, L = cfg["d"], cfg["ffn"], cfg["E"], cfg["k"], cfg["layers"]
    o = oracle.load()
    xs = {T: inputs.sweep_tokens(T, d, device="cuda") for T in SWEEP_CHECK}
    ws = moe.Workspace("cuda")
    worst = {T: (0.0, 0.0) for T in SWEEP_CHECK}
    for l in range(L):
        layer = inputs.sweep_layer(l, d, ffn, E, device="cuda", seed0=cfg["layer_seed0"])
        host = None
        for T, x in xs.items():
            check = l in SWEEP_CHECK[T]
            x_before = inputs.to_host(x) if check else None
            moe.block_forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, eps=EPS,
                              workspace=ws)
            if not check:
                continue
            torch.cuda.synchronize()
            if host is None:
                host = inputs.layer_to_host(layer)
            xn = o.rmsnorm(x_before, EPS)
            if T <= 64:
                rows = np.arange(T)
            else:
                _, idx, offsets, perm = helpers.oracle_layout(xn, host, k)
                rows = helpers.layout_rows(idx, offsets, perm, k, per_expert=16,
                                           seed=l + T, halves=T <= 4096,
                                           row_tiles=(128,) if T <= 1024 else ())
            out, rl, _, _, exact = o.moe_forward(xn[rows], *host[:4], k, exact=True)
            got = helpers.host_f64(inputs.to_host(x)[rows])
            ref = helpers.host_f64(x_before[rows]) + exact
            keep = ~helpers.near_tie_mask(rl, k)
            assert keep.mean() > 0.9 or T == 1
            if not keep.any():
                continue
            rms = float(np.sqrt((exact[keep] ** 2).mean()))
            excess = (np.abs(got - ref) - helpers.bf16_half_ulp(got)
                      - helpers.bf16_half_ulp(exact))[keep]
            err = max(float(excess.max()), 0.0) / rms
            raw = float(np.abs(got - ref)[keep].max()) / rms
            print(f"PARITY sweep T={T} layer {l}: gated {err:.3e} raw max|d|/rms {raw:.3e} "
                  f"over {keep.sum()} tokens, {(~keep).sum()} near ties")
            worst[T] = (max(worst[T][0], err), max(worst[T][1], raw))
            assert err <= helpers.TOL_BF16, (T, l, err)
        del layer, host
    assert moe.device_status(clear=True) == 0
    for T, (g, r) in worst.items():
        print(f"PARITY sweep T={T} worst: gated {g:.3e} raw {r:.3e}")


@pytest.mark.parametrize("fuse", ["0", "1"], ids=["combine_pass", "combine_in_down"])
@pytest.mark.parametrize("T,d,ffn,E,k,gating", [
    (700, 192, 384, 8, 2, 0),
    (2300, 192, 320, 8, 2, 0),     # several token tiles per expert, ragged features
    (1500, 128, 192, 4, 1, 0),     # one slot per token
    (900, 256, 256, 8, 2, 1),      # gates from the full softmax (not renormalised)
])
def test_combine_in_down_epilogue(moe, monkeypatch, fuse, T, d, ffn, E, k, gating):
    """The CTA-pair down projection with the gated combine in its epilogue
    (fp32 additions of gate x output into a zeroed row per token, then one
    rounding) against the separate combine pass: both against the oracle,
    and the fused form gives the same bits on every call (at most two
    additions into zero per element)."""
    monkeypatch.setenv("MOE_PLAN_PAIR", "1")
    monkeypatch.setenv("MOE_PLAN_SPLITS", "1")
    monkeypatch.setenv("MOE_FUSE_COMBINE", fuse)
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=T + 3, device="cuda")
    kw = dict(gating=gating) if gating else {}
    out = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, **kw)
    out2 = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    o = oracle.load()
    Wg, W1, W3, W2, bias = inputs.layer_to_host(layer)
    _, rl, _, _, exact = o.moe_forward(inputs.to_host(x), Wg, W1, W3, W2, k, exact=True,
                                       gating=gating)
    keep = ~helpers.near_tie_mask(rl, k)
    got = inputs.to_host(out)
    err = helpers.rel_error(got[keep], exact[keep], "bf16")
    print(f"PARITY combine fuse={fuse} T{T} k{k} gating{gating}: gated {err:.3e} raw "
          f"{helpers.raw_rel_error(got[keep], exact[keep]):.3e} over {keep.sum()} tokens")
    assert err <= helpers.TOL_BF16


@pytest.mark.parametrize("T,d,ffn,E,k,dtype,cap", [
    (1, 256, 448, 8, 2, "bf16", 0),
    (16, 256, 448, 8, 2, "bf16", 0),
    (37, 192, 320, 5, 2, "bf16", 0),
    (64, 128, 256, 64, 8, "bf16", 0),     # 512 selections over 64 experts
    (100, 64, 64, 8, 2, "bf16", 20),      # capacity: dropped selections get no row
    (65, 128, 448, 8, 2, "f32", 0),
    (500, 64, 64, 8, 2, "bf16", 0),       # 1000 selections: every warp several chunks
])
def test_small_batch_grouping_kernel_equals_two_kernels(moe, monkeypatch, T, d, ffn, E, k,
                                                        dtype, cap):
    """Grouping a small batch in one kernel (counts, scan over 32-selection
    chunks, ranks from matching lanes, row copies) gives the bits of the
    two-kernel grouping (chunk counts + scan, then ranks and copies), for
    the layer and for the pre-norm block (rows scaled on the way)."""
    x, layer = inputs.make_workload(T, d, ffn, E, k, dtype, seed=T + 13, device="cuda")
    kw = dict(capacity=cap) if cap else {}
    outs, blocks = {}, {}
    for r in ("0", "1"):
        monkeypatch.setenv("MOE_ROUTE_SMALL", r)
        outs[r] = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, **kw)
        xb = x.clone()
        moe.block_forward(xb, layer.Wg, layer.W1, layer.W3, layer.W2, k, **kw)
        blocks[r] = xb
    torch.cuda.synchronize()
    view = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(outs["0"].view(view), outs["1"].view(view))
    assert torch.equal(blocks["0"].view(view), blocks["1"].view(view))
    if not cap:
        check_layer(moe, x, layer, k, dtype=dtype, label=f"small grouping T{T} E{E} k{k}")


@pytest.mark.parametrize("order", ["w1_first", "w3_first", "mixed"])
@pytest.mark.parametrize("T,d,ffn,E,k", [
    (700, 192, 384, 8, 2),
    (2300, 192, 320, 8, 2),        # ffn = 5 x 64: the last pair tile is half outside
    (1500, 128, 192, 4, 3),
])
def test_interleaved_gate_up_rows_equal_two_boxes(moe, monkeypatch, order, T, d, ffn, E, k):
    """The CTA-pair gate/up GEMM loading W1[e] and W3[e] as one 4-D box that
    interleaves them in 16-row groups (gate and up of a feature 16 lanes
    apart, swapped by shuffle; seven ring stages) gives the bits of the
    two-box layout (exchange through shared memory, six stages): the same
    rows reach the same MMAs.  W3 is placed after W1 in memory, before it,
    or alternately per expert (the map then starts at the lower matrix)."""
    monkeypatch.setenv("MOE_PLAN_PAIR", "1")
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=T + 17, device="cuda")
    buf = torch.empty(2, E, ffn, d, dtype=torch.bfloat16, device="cuda")
    W1, W3 = [], []
    for e in range(E):
        first = 0 if order == "w1_first" else 1 if order == "w3_first" else e % 2
        buf[first, e] = layer.W1[e]
        buf[1 - first, e] = layer.W3[e]
        W1.append(buf[first, e])
        W3.append(buf[1 - first, e])
    outs = {}
    for il in ("0", "1"):
        monkeypatch.setenv("MOE_PAIR_IL", il)
        outs[il] = moe.forward(x, layer.Wg, W1, W3, layer.W2, k)
    torch.cuda.synchronize()
    assert torch.equal(outs["0"].view(torch.int16), outs["1"].view(torch.int16))
    ref = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), outs["1"].view(torch.int16))


@pytest.mark.parametrize("pinned_in", [True, False], ids=["pinned_in", "pageable_in"])
@pytest.mark.parametrize("pinned_out", [True, False], ids=["pinned_out", "pageable_out"])
@pytest.mark.parametrize("direct", ["1", "0"], ids=["direct", "copy"])
def test_host_io_paths(moe, monkeypatch, pinned_in, pinned_out, direct):
    """moe_forward_host_io delivers the device path's bits to out_host
    whether the router reads page-locked x_host itself (leaving the rows in
    x_dev) or a copy to x_dev comes first, and whether the last kernel writes
    page-locked out_host directly or a copy from out_dev follows (pageable
    buffers, or the direct paths turned off), on repeated calls (launch-graph
    replays)."""
    monkeypatch.setenv("MOE_HOSTIO_DIRECT", direct)
    x, layer = inputs.make_workload(48, 256, 512, 8, 2, "bf16", 19, "cuda")
    ref = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, 2).cpu()
    xh = x.cpu().pin_memory() if pinned_in else x.cpu()
    for _ in range(3):
        oh = torch.empty_like(xh, pin_memory=pinned_out)
        oh.fill_(0)
        moe.forward_host_io(xh, layer.Wg, layer.W1, layer.W3, layer.W2, 2, out_host=oh)
        torch.cuda.synchronize()
        assert torch.equal(oh.view(torch.int16), ref.view(torch.int16))
