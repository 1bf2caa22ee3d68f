"""Launch graphs: a forward entry point called again with the same arguments
replays a CUDA graph of its launches (the second call captures it).  The
graph holds the same kernels with the same parameters, so every result must
equal the bits of direct launches (MOE_GRAPHS=0) on the same data, whatever
the data were when the graph was captured (needs a GPU)."""
import pytest
import torch

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


def _inputs(T, d, ffn, E, k, seed):
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 99)
    xs = [x.clone()] + [torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
                        for _ in range(2)]
    return x, layer, xs


def _sequence(moe, call, x, xs, reps):
    """Run call() after loading each batch of xs into x, reps times over."""
    outs = []
    for _ in range(reps):
        for xi in xs:
            x.copy_(xi)
            outs.append(call().clone())
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("T,d,ffn,E,k", [(16, 256, 448, 8, 2), (700, 192, 384, 8, 2)])
def test_repeated_forward_equals_direct_launches(moe, monkeypatch, T, d, ffn, E, k):
    """Same tensors, new contents per call: direct call, capture, replays."""
    x, layer, xs = _inputs(T, d, ffn, E, k, seed=T)
    out = torch.empty_like(x)
    ws = moe.Workspace(x.device)

    def call():
        return moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, out=out, workspace=ws)

    monkeypatch.setenv("MOE_GRAPHS", "0")
    ref = _sequence(moe, call, x, xs, 1)
    monkeypatch.setenv("MOE_GRAPHS", "1")
    got = _sequence(moe, call, x, xs, 3)
    for i, o in enumerate(got):
        assert torch.equal(o, ref[i % len(xs)]), i


def test_repeated_host_io_equals_direct_launches(moe, monkeypatch):
    """moe_forward_host_io: the copies are part of the graph, so each replay
    reads the pinned input as it is at launch and writes the pinned output."""
    T, d, ffn, E, k = 16, 256, 448, 8, 2
    x, layer, xs = _inputs(T, d, ffn, E, k, seed=5)
    x_host = x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    x_dev, out_dev = torch.empty_like(x), torch.empty_like(x)
    ws = moe.Workspace(x.device)

    def run(reps):
        outs = []
        for _ in range(reps):
            for xi in xs:
                x_host.copy_(xi.cpu())
                moe.forward_host_io(x_host, layer.Wg, layer.W1, layer.W3, layer.W2, k,
                                    out_host=out_host, x_dev=x_dev, out_dev=out_dev, workspace=ws)
                torch.cuda.synchronize()
                outs.append(out_host.clone())
        return outs

    monkeypatch.setenv("MOE_GRAPHS", "0")
    ref = run(1)
    monkeypatch.setenv("MOE_GRAPHS", "1")
    got = run(3)
    for i, o in enumerate(got):
        assert torch.equal(o, ref[i % len(xs)]), i
    dev_out = moe.forward(xs[-1], layer.Wg, layer.W1, layer.W3, layer.W2, k)
    torch.cuda.synchronize()
    assert torch.equal(got[-1], dev_out.cpu())


def test_repeated_block_forward_equals_direct_launches(moe, monkeypatch):
    """The in-place pre-norm block: each replay updates x from its current
    contents, exactly as direct launches do."""
    T, d, ffn, E, k = 64, 256, 448, 8, 2
    x, layer, xs = _inputs(T, d, ffn, E, k, seed=11)
    ws = moe.Workspace(x.device)

    def chain():
        x.copy_(xs[0])
        outs = []
        for _ in range(4):
            moe.block_forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, workspace=ws)
            outs.append(x.clone())
        torch.cuda.synchronize()
        return outs

    monkeypatch.setenv("MOE_GRAPHS", "0")
    ref = chain()
    monkeypatch.setenv("MOE_GRAPHS", "1")
    for _ in range(2):
        got = chain()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_plan_change_with_same_tensors_gets_its_own_graph(moe, monkeypatch):
    """The plan is part of the key: forcing another split count on the same
    tensors must not replay the graph captured under the first plan."""
    T, d, ffn, E, k = 300, 256, 1024, 8, 2
    x, layer, _ = _inputs(T, d, ffn, E, k, seed=3)
    out = torch.empty_like(x)
    ws = moe.Workspace(x.device)

    def call():
        moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, out=out, workspace=ws)
        torch.cuda.synchronize()
        return out.clone()

    ref = {}
    monkeypatch.setenv("MOE_GRAPHS", "0")
    for splits in ("2", "5"):
        monkeypatch.setenv("MOE_PLAN_SPLITS", splits)
        ref[splits] = call()
    assert not torch.equal(ref["2"], ref["5"])  # fp32 partial sums in another order
    monkeypatch.setenv("MOE_GRAPHS", "1")
    for splits in ("2", "5", "2", "5", "2", "5"):
        monkeypatch.setenv("MOE_PLAN_SPLITS", splits)
        assert torch.equal(call(), ref[splits]), splits


def test_call_inside_a_caller_capture(moe):
    """On a stream that is being captured the kernels go into the caller's
    graph; replaying it gives the direct result."""
    T, d, ffn, E, k = 16, 256, 448, 8, 2
    x, layer, xs = _inputs(T, d, ffn, E, k, seed=21)
    out = torch.empty_like(x)
    ws = moe.Workspace(x.device)
    for _ in range(3):  # the library's own graph exists before the capture
        moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, out=out, workspace=ws)
    for xi in xs:
        x.copy_(xi)
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        ref = moe.forward(xi, layer.Wg, layer.W1, layer.W3, layer.W2, k)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_graph_cache_counts_and_evicts_least_recent(moe, monkeypatch):
    """The cache's counters: first call direct, second a capture, then
    replays; more than 64 argument sets evict the least recently used one,
    whose next call starts over (direct), with the same bits as before."""
    monkeypatch.setenv("MOE_GRAPHS", "1")
    T, d, ffn, E, k = 8, 128, 256, 8, 2
    x, layer = inputs.make_workload(T, d, ffn, E, k, "bf16", seed=41, device="cuda")
    ws = moe.Workspace(x.device)
    outs = [torch.empty_like(x) for _ in range(70)]   # one argument set per output buffer
    moe.graph_cache_stats(reset=True)

    def call(i):
        return moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, out=outs[i],
                           workspace=ws)

    call(0)
    call(0)
    call(0)
    torch.cuda.synchronize()
    st = moe.graph_cache_stats()
    assert (st["direct_calls"], st["captures"], st["replays"]) == (1, 1, 1)
    ref = outs[0].clone()
    for i in range(1, 70):
        call(i)
    torch.cuda.synchronize()
    st = moe.graph_cache_stats()
    assert st["entries"] == 64
    assert st["evictions"] >= 6
    # set 0 was the least recently used: gone, so it runs directly again
    before = st["direct_calls"]
    outs[0].zero_()
    call(0)
    torch.cuda.synchronize()
    assert moe.graph_cache_stats()["direct_calls"] == before + 1
    assert torch.equal(outs[0].view(torch.int16), ref.view(torch.int16))
    for i in range(70):
        assert torch.equal(outs[i].view(torch.int16), ref.view(torch.int16))
