"""moe_forward_static_scratch: the layer for callers that cannot allocate
device memory where they run it (an engine plugin handed fixed buffers, a
process whose memory budget was reserved up front).  Its
scratch is a fixed array inside the library, so the caller passes only the
tokens, the weights and the output.

Checked through the C ABI against moe_forward (the entry point with a caller
workspace), on two calls in a row that share the library's scratch.  Runs
last (file name) and works alone in a fresh process or after the others."""
import ctypes

import pytest
import torch

import helpers
from sparse_mixture_experts_58_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from sparse_mixture_experts_58_b300 import moe as m
    return m


def _call_static(moe, x, layer, k, out):
    T, d = x.shape
    E, ffn = layer.E, layer.ffn
    rc = moe.lib().moe_forward_static_scratch(
        x.data_ptr(), layer.Wg.data_ptr(),
        None if layer.bias is None else layer.bias.data_ptr(),
        moe._expert_ptrs(layer.W1, E), moe._expert_ptrs(layer.W3, E),
        moe._expert_ptrs(layer.W2, E), T, d, ffn, E, k, moe._dt(x), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("name,T,seed", [("decode", 16, None), ("small", 40, 21),
                                         ("one_token", 1, None), ("four_tokens", 4, None)])
def test_static_scratch_matches_workspace_entry_point(moe, name, T, seed):
    """Equal to moe_forward (its own workspace) at decode, at a small shape,
    and at one and four tokens of the Mixtral shape, where the plan also
    carves the gate/up halves' partial sums and counters out of the array."""
    if name == "decode":
        x, layer = inputs.make_named("decode", device="cuda")
    elif seed is None:
        x, layer = inputs.make_named("decode", device="cuda")
        x = x[:T].contiguous()
    else:
        x, layer = inputs.make_workload(T, 256, 448, 8, 2, "bf16", seed, "cuda")
    k = 2
    ref = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias)
    # a second batch, so the two static-scratch calls in a row differ
    x2 = torch.flip(x, dims=[0]).contiguous()
    ref2 = moe.forward(x2, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=layer.bias)
    out1 = torch.empty_like(x)
    out2 = torch.empty_like(x)
    assert _call_static(moe, x, layer, k, out1) == 0
    assert _call_static(moe, x2, layer, k, out2) == 0
    torch.cuda.synchronize()
    assert moe.device_status(clear=True) == 0
    for got, want in ((out1, ref), (out2, ref2)):
        err = helpers.rel_error(inputs.to_host(got), helpers.host_f64(inputs.to_host(want)),
                                "bf16")
        assert err <= helpers.TOL_BF16, err
        # same kernels, same plan: identical bits in practice
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_static_scratch_rejects_oversize(moe):
    """A batch whose scratch would exceed the fixed array is refused before
    anything runs."""
    T, d, ffn, E, k = 512, 4096, 14336, 8, 2
    assert moe.workspace_bytes(T, d, ffn, E, k, moe.BF16) > moe.STATIC_SCRATCH_BYTES
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros(E, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, 1, dtype=torch.bfloat16, device="cuda")   # never touched
    ptrs = (ctypes.c_void_p * E)(*([w.data_ptr()] * E))
    out = torch.empty_like(x)
    rc = moe.lib().moe_forward_static_scratch(x.data_ptr(), Wg.data_ptr(), None, ptrs, ptrs,
                                              ptrs, T, d, ffn, E, k, moe.BF16, out.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    assert rc == moe.ERR_WORKSPACE


def test_static_scratch_repeated_identical_calls_allocate_nothing(moe):
    """Three calls in a row with the same pointers (the case where the
    workspace entry points would start replaying a captured launch graph):
    after a first call, the device's free memory does not move across the
    repeated calls, and every output equals moe_forward's."""
    x, layer = inputs.make_workload(24, 256, 448, 8, 2, "bf16", 31, "cuda")
    k = 2
    ref = moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k)
    out = torch.empty_like(x)
    assert _call_static(moe, x, layer, k, out) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        out.fill_(0)
        assert _call_static(moe, x, layer, k, out) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert moe.device_status(clear=True) == 0
