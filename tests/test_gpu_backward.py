"""Backward of the layer (moe_backward, through the C ABI) against the oracle's
backward on the same seeded inputs (needs a GPU).

The GPU keeps the recomputed gate/up projections U, V and the hidden
gradients dU, dV and g*H in bf16 (as the forward keeps h; the last three are
bf16 tensor-core operands), accumulates in fp32 and returns dx in bf16 and the
weight gradients in fp32; the oracle works in double.  The bar is derived from
those roundings: an exact emulation of just them (float64 otherwise) differs
from the oracle by 2.4e-3 to 3.1e-3 normwise (||a - b|| / ||b||) and, where an
expert has only a few rows to sum over, by up to 1.1e-1 of the RMS on single
elements.  So for every gradient: normwise error <= 1e-2 and max error <=
2.5e-1 * RMS.  (A kernel mistake such as a dropped term or factor moves the
normwise error to 1e-1 or more.)  Tokens whose oracle top-(k+1) logits lie
within 1e-3 of each other get a zero upstream gradient on both sides, so a
rounding-dependent expert choice cannot enter the comparison."""
import numpy as np
import pytest
import torch

import helpers
import oracle
from sparse_mixture_experts_58_b300 import inputs

pytestmark = pytest.mark.gpu

TOL_NORM = 1e-2
TOL_MAX = 2.5e-1


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


def _case(T, d, ffn, E, k, seed, bias=None):
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=seed, device="cuda", bias=bias)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dout = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    o = oracle.load()
    logits, _, _ = o.router(inputs.to_host(x), inputs.to_host(layer.Wg), k,
                            None if layer.bias is None else layer.bias.cpu().numpy())
    ties = helpers.near_tie_mask(logits, k)
    dout[torch.as_tensor(ties, device="cuda")] = 0
    return x, layer, dout, ties


def _errs(got, ref):
    """(normwise error, max error / RMS) of got against ref."""
    got = helpers.host_f64(np.asarray(got)) if np.asarray(got).dtype == np.uint16 \
        else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = max(float(np.sqrt((ref ** 2).mean())), 1e-30)
    diff = got - ref
    return float(np.sqrt((diff ** 2).mean())) / rms, float(np.abs(diff).max()) / rms


def _compare(moe, x, layer, dout, k, label, rows1=None, rows2=None):
    E = layer.E
    got = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout, k, bias=layer.bias)
    torch.cuda.synchronize()
    Wg, W1, W3, W2, bias = inputs.layer_to_host(layer)
    ref = oracle.load().moe_backward(inputs.to_host(x), Wg, W1, W3, W2, k, inputs.to_host(dout),
                                     bias=bias, rows1=rows1, rows2=rows2)
    errs = {"dx": _errs(inputs.to_host(got["dx"]), ref["dx"]),
            "dWg": _errs(got["dWg"].cpu().numpy(), ref["dWg"])}
    c0, c1 = rows1 if rows1 else (0, layer.ffn)
    n0, n1 = rows2 if rows2 else (0, layer.d)
    for key, sl in (("dW1", slice(c0, c1)), ("dW3", slice(c0, c1)), ("dW2", slice(n0, n1))):
        errs[key] = _errs(got[key][:, sl].cpu().numpy(), np.stack(ref[key]))
    print(f"{label}: " + ", ".join(f"{k_} {n:.2e}/{m:.2e}" for k_, (n, m) in errs.items()))
    for key, (n, m) in errs.items():
        assert n <= TOL_NORM and m <= TOL_MAX, (label, key, n, m)
    return got


@pytest.mark.parametrize("T,d,ffn,E,k", [
    (16, 256, 448, 8, 2),       # decode-sized: one token tile per expert
    (37, 128, 192, 8, 2),
    (5, 128, 128, 8, 2),        # most experts empty: their weight gradients are zero
    (300, 256, 512, 8, 2),
    (700, 192, 384, 8, 2),      # several token tiles per expert, ragged features
    (64, 128, 128, 4, 1),
    (100, 64, 64, 1, 1),        # one expert: a dense SwiGLU FFN, no router gradient
    (256, 128, 256, 16, 3),
])
def test_backward_against_oracle(moe, T, d, ffn, E, k):
    x, layer, dout, ties = _case(T, d, ffn, E, k, seed=T + d + E)
    got = _compare(moe, x, layer, dout, k, f"T{T} d{d} ffn{ffn} E{E} k{k}")
    if E == 1:
        assert torch.count_nonzero(got["dWg"]) == 0


def test_backward_skewed_router_bias(moe):
    """The skewed benchmark's per-expert bias: one expert takes most rows."""
    x, layer, dout, _ = _case(400, 128, 256, 8, 2, seed=9, bias=inputs.SKEW_BIAS)
    _compare(moe, x, layer, dout, 2, "skewed T400")


def test_backward_mixtral_shape_decode(moe):
    """The Mixtral shape (hidden 4096, expert width 14336, 8 experts, top-2)
    at T = 16: dx and dW_g in full, the weight gradients on a window of 64
    rows of each expert."""
    x, layer, dout, _ = _case(16, 4096, 14336, 8, 2, seed=0)
    _compare(moe, x, layer, dout, 2, "Mixtral shape T16", rows1=(1000, 1064), rows2=(2000, 2064))


def test_backward_exact_properties(moe):
    """Deterministic (two calls agree bit for bit), exactly linear in dout
    (doubling dout doubles every gradient: scaling by 2 is exact in bf16 and
    fp32), zero for a zero dout, and all zeros for an empty batch."""
    x, layer, dout, _ = _case(300, 256, 512, 8, 2, seed=3)
    a = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout, 2)
    b = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout, 2)
    c = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout * 2, 2)
    z = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, torch.zeros_like(dout), 2)
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key
        assert torch.equal(c[key].float(), 2 * a[key].float()), key
        assert torch.count_nonzero(z[key]) == 0, key
    e = moe.backward(x[:0], layer.Wg, layer.W1, layer.W3, layer.W2, dout[:0], 2,
                     grads={key: torch.full_like(v, 7.0) if key != "dx" else v[:0]
                            for key, v in a.items()})
    torch.cuda.synchronize()
    for key in ("dWg", "dW1", "dW3", "dW2"):
        assert torch.count_nonzero(e[key]) == 0, key


@pytest.mark.parametrize("T,d,ffn,E,k", [(37, 128, 192, 8, 2), (700, 192, 384, 8, 2)])
def test_backward_matches_rounding_emulation(moe, T, d, ffn, E, k):
    """Against torch (fp32 matmuls) with the GPU's rounding points emulated:
    U, V, dU, dV and g*H rounded to bf16, sums in fp32.  What remains is
    summation order and the odd intermediate landing on the other side of a
    bf16 rounding, so the normwise error is far below the oracle bar."""
    x, layer, dout, _ = _case(T, d, ffn, E, k, seed=T + d + E)
    got = moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout, k)
    _, idx, gates = moe.router(x, layer.Wg, k)
    torch.cuda.synchronize()
    bf = lambda t: t.to(torch.bfloat16).float()
    xf, df = x.float(), dout.float()
    ref = {key: torch.zeros_like(got[key], dtype=torch.float32) for key in ("dW1", "dW3", "dW2")}
    dx = torch.zeros(T, d, device="cuda")
    for e in range(E):
        sel = (idx == e).nonzero()
        if len(sel) == 0:
            continue
        t, j = sel[:, 0], sel[:, 1]
        X, G, gg = xf[t], df[t], gates[t, j][:, None]
        U, V = bf(X @ layer.W1[e].float().T), bf(X @ layer.W3[e].float().T)
        s = torch.sigmoid(U)
        dh = gg * (G @ layer.W2[e].float())
        dU, dV, gH = bf(dh * V * (s + U * s * (1 - s))), bf(dh * U * s), bf(gg * U * s * V)
        ref["dW1"][e], ref["dW3"][e], ref["dW2"][e] = dU.T @ X, dV.T @ X, G.T @ gH
        dx.index_add_(0, t, dU @ layer.W1[e].float() + dV @ layer.W3[e].float())
    for key in ("dW1", "dW3", "dW2"):
        n = ((got[key] - ref[key]).norm() / ref[key].norm()).item()
        assert n <= 1e-3, (key, n)


def _random_backward_case(i):
    """The i-th seeded random backward shape: tokens 1..800, hidden and
    expert widths in 64-wide steps, 1..16 experts, top-1..4."""
    rng = np.random.default_rng(5000 + i)
    band = rng.random()
    T = int(rng.integers(1, 17) if band < 0.3 else rng.integers(17, 801))
    d = 64 * int(rng.integers(1, 7))
    ffn = 64 * int(rng.integers(1, 9))
    E = int(rng.integers(1, 17))
    k = int(rng.integers(1, min(E, 4) + 1))
    return T, d, ffn, E, k, int(rng.integers(0, 1 << 30))


@pytest.mark.parametrize("i", range(32))
def test_random_backward_against_oracle(moe, i):
    """Seeded random shapes (ragged token tiles, empty experts, one expert,
    top-1 to top-4) against the oracle's backward with the same bars."""
    T, d, ffn, E, k, seed = _random_backward_case(i)
    x, layer, dout, ties = _case(T, d, ffn, E, k, seed=seed)
    if ties.all():
        pytest.skip("every token near a tie")
    _compare(moe, x, layer, dout, k, f"random {i}: T{T} d{d} ffn{ffn} E{E} k{k}")
