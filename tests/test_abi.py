"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, sizes workspaces, and rejects bad arguments before touching
the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    from sparse_mixture_experts_58_b300 import build
    build.build()
    from sparse_mixture_experts_58_b300 import moe as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert "moe_forward" in names and "moe_route_from_logits" in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(moe):
    lib = moe.lib()
    for name in declared_functions():
        assert hasattr(lib, name), f"libmoe.so does not export {name}"
    # the binding wraps every declared entry point
    assert sorted(moe.EXPORTED) == declared_functions()


def test_strerror_and_version(moe):
    assert moe.strerror(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert moe.strerror(code) != "unknown status"
    assert moe.lib().moe_version() >= 100


def test_workspace_sizes(moe):
    # Mixtral decode/prefill shapes: scratch holds the grouped rows, the hidden
    # activations and the fp32 partial outputs
    for T in (1, 16, 4096, 8192, 16384):
        n = moe.workspace_bytes(T, 4096, 14336, 8, 2, moe.BF16)
        S = moe.down_splits(T, 4096, 14336, 8, 2, moe.BF16)
        rows = 2 * T
        assert n >= rows * 4096 * 2 + rows * 14336 * 2 + S * rows * 4096 * 4
        assert n % 256 == 0
        assert 1 <= S <= 14336 // 64
    assert moe.workspace_bytes(0, 4096, 14336, 8, 2, moe.BF16) >= 0
    assert moe.down_splits(4096, 4096, 14336, 8, 2, moe.BF16) == 1
    assert moe.down_splits(16, 4096, 14336, 8, 2, moe.BF16) > 1


def test_down_split_plan(moe):
    """The split of the down projection's contraction (host-side plan, Mixtral
    shape): measured best choices are kept -- two splits for one token (two
    busy experts, 128 units on 148 SMs), four at decode (1024 units, the last
    wave 136 of 148 SMs), none once the fp32 partial sums outweigh the wave
    fill (one-CTA tiles from T=200, CTA pairs up to 1024 rows), two for pairs
    at T=1024..2048; always a whole number of 64-deep blocks per split."""
    S = lambda T, E=8, k=2: moe.down_splits(T, 4096, 14336, E, k, moe.BF16)
    assert S(1) == 2
    assert S(16) == 4
    assert all(S(T) == 1 for T in (200, 256, 400, 511, 512, 3072, 4096, 16384))
    assert S(1024) == 2 and S(2048) == 2
    for T in (1, 2, 3, 4, 8, 16, 32, 64, 128, 199, 300, 1024, 8192):
        s = S(T)
        kps = -(-224 // s)
        assert 1 <= s <= 28 and -(-224 // kps) == s, (T, s)
    for E, k in ((4, 1), (4, 2), (16, 3), (64, 8)):
        for T in (1, 7, 16, 300):
            assert 1 <= S(T, E, k) <= 28
    # decode batches group in one kernel (5 launches); larger ones in two
    assert moe.forward_launches(16, 4096, 14336, 8, 2, moe.BF16) == 5
    assert moe.forward_launches(32, 4096, 14336, 8, 2, moe.BF16) == 5
    assert moe.forward_launches(33, 4096, 14336, 8, 2, moe.BF16) == 6
    assert moe.forward_launches(4096, 4096, 14336, 8, 2, moe.BF16) == 6
    assert moe.forward_launches(0, 4096, 14336, 8, 2, moe.BF16) == 0


@pytest.mark.parametrize("args,code", [
    ((16, 4096, 14336, 16, 9, 1), -2),     # top-k above 8
    ((16, 4096, 14336, 2, 3, 1), -1),      # k > E
    ((-1, 4096, 14336, 8, 2, 1), -1),      # negative T
    ((16, 4096, 14336, 65, 2, 1), -2),     # more than 64 experts
    ((16, 4000, 14336, 8, 2, 1), -2),      # bf16 needs d % 64 == 0
    ((16, 4096, 14300, 8, 2, 1), -2),      # bf16 needs ffn % 64 == 0
    ((16, 130, 448, 8, 2, 0), -2),         # fp32 needs d % 4 == 0
    ((16, 4096, 14336, 8, 2, 7), -1),      # unknown dtype
])
def test_workspace_rejects_bad_shapes(moe, args, code):
    n = ctypes.c_size_t()
    assert moe.lib().moe_workspace_bytes(*args, ctypes.byref(n)) == code


def _forward_call(moe, **over):
    E = over.get("E", 8)
    arr = ctypes.c_void_p * E
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first
    w = arr(*([0x10000] * E))
    a = dict(x=fake, Wg=fake, bias=None, W1=w, W3=w, W2=w, T=16, d=256, ffn=512, E=E, k=2,
             dt=moe.BF16, out=fake, ws=None, ws_bytes=0, stream=None)
    a.update(over)
    return moe.lib().moe_forward(a["x"], a["Wg"], a["bias"], a["W1"], a["W3"], a["W2"], a["T"],
                                 a["d"], a["ffn"], a["E"], a["k"], a["dt"], a["out"], a["ws"],
                                 a["ws_bytes"], a["stream"])


def test_forward_validates_before_launch(moe):
    assert _forward_call(moe, k=9, E=16) == -2
    assert _forward_call(moe, x=None) == -1
    assert _forward_call(moe, W1=None) == -1
    assert _forward_call(moe, ws=None) == -3                       # no workspace
    assert _forward_call(moe, ws=ctypes.c_void_p(0x10000), ws_bytes=16) == -3
    assert _forward_call(moe, x=ctypes.c_void_p(0x10008)) == -2    # misaligned tensor
    assert _forward_call(moe, T=0) == 0                            # empty batch: no-op


def test_fault_injection_fails_before_launch(moe, monkeypatch):
    monkeypatch.setenv("MOE_FAULT_INJECT", "workspace")
    assert _forward_call(moe) == -3
    monkeypatch.setenv("MOE_FAULT_INJECT", "cuda")
    assert _forward_call(moe) == -4
    monkeypatch.setenv("MOE_FAULT_INJECT", "arg")
    assert _forward_call(moe) == -1
    monkeypatch.delenv("MOE_FAULT_INJECT")


def test_binding_module_requires_library(tmp_path):
    """Importing the binding without the built library raises (no fallback)."""
    import subprocess
    import sys
    import shutil
    pkg = os.path.join(ROOT, "sparse_mixture_experts_58_b300")
    dst = tmp_path / "sparse_mixture_experts_58_b300"
    dst.mkdir()
    for f in ("__init__.py", "moe.py", "inputs.py"):
        shutil.copy(os.path.join(pkg, f), dst / f)
    code = ("import sys; sys.path.insert(0, %r)\n"
            "try:\n    import sparse_mixture_experts_58_b300.moe\n"
            "except ImportError as e:\n    print('raised', e); sys.exit(0)\n"
            "sys.exit(1)\n") % str(tmp_path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "not built" in r.stdout


def test_capacity_helper(moe):
    assert moe.capacity(1.0, 4096, 2, 8) == 1024
    assert moe.capacity(1.25, 4096, 2, 8) == 1280
    assert moe.capacity(1.1, 10, 2, 8) == 3          # ceil(2.75)
    assert moe.capacity(0.0, 4096, 2, 8) == 0        # no limit


def test_forward_ex_rejects_bad_options(moe):
    E = 8
    arr = ctypes.c_void_p * E
    fake = ctypes.c_void_p(0x10000)
    w = arr(*([0x10000] * E))
    for opt in (moe.Options(2, 0, 0), moe.Options(0, 10, 5)):
        rc = moe.lib().moe_forward_ex(fake, fake, None, w, w, w, 16, 256, 512, E, 2, moe.BF16,
                                      ctypes.byref(opt), fake, None, 0, None)
        assert rc == -1


def test_block_forward_validates_before_launch(moe):
    """moe_block_forward checks its arguments on the host like moe_forward_ex
    (negative eps, null or misaligned x, missing workspace, bad options)."""
    E = 8
    arr = ctypes.c_void_p * E
    fake = ctypes.c_void_p(0x10000)
    w = arr(*([0x10000] * E))
    lib = moe.lib()

    def call(x=fake, T=16, eps=1e-5, ws=fake, ws_bytes=1 << 30, opt=None):
        return lib.moe_block_forward(x, fake, None, w, w, w, T, 256, 512, E, 2, moe.BF16, eps,
                                     opt, ws, ws_bytes, None)

    assert call(eps=-1.0) == -1
    assert call(eps=float("nan")) == -1
    assert call(x=None) == -1
    assert call(x=ctypes.c_void_p(0x10008)) == -2
    assert call(ws=None) == -3
    assert call(opt=ctypes.byref(moe.Options(2, 0, 0))) == -1
    assert call(T=0) == 0


def test_backward_validates_before_launch(moe):
    """moe_backward checks its arguments on the host: fp32 is not supported,
    null and misaligned tensors and a missing workspace are rejected."""
    E = 8
    arr = ctypes.c_void_p * E
    fake = ctypes.c_void_p(0x10000)
    w = arr(*([0x10000] * E))
    lib = moe.lib()

    def call(x=fake, dt=moe.BF16, dWg=fake, ws=fake, ws_bytes=1 << 34, gW=w, dx=fake, d=256):
        return lib.moe_backward(x, fake, None, w, w, w, 16, d, 512, E, 2, dt, fake, dx, dWg,
                                gW, gW, gW, ws, ws_bytes, None)

    assert call(dt=moe.F32) == -2
    assert call(d=96) == -2
    assert call(x=None) == -1
    assert call(dx=None) == -1
    assert call(dWg=None) == -1
    assert call(gW=arr(*([0] * E))) == -1
    assert call(x=ctypes.c_void_p(0x10008)) == -2
    assert call(ws=None) == -3
    n = ctypes.c_size_t()
    assert lib.moe_backward_workspace_bytes(16, 256, 512, E, 2, moe.BF16, ctypes.byref(n)) == 0
    assert n.value > 0
    assert lib.moe_backward_workspace_bytes(16, 256, 512, E, 2, moe.F32, ctypes.byref(n)) == -2


def test_gate_up_halves_scratch_in_workspace(moe):
    """Batches of up to 8 expert rows (T <= 4 at top-2) reserve the gate/up
    halves' scratch: fp32 partial sums [2][rows][2 ffn] and the arrival
    counters; T = 5 (10 rows) does not, and shrinks below T = 4 despite the
    larger batch."""
    d, ffn = 4096, 14336
    ws = {T: moe.workspace_bytes(T, d, ffn, 8, 2, moe.BF16) for T in range(1, 7)}
    for T in range(1, 5):
        assert ws[T] >= 2 * (2 * T) * 2 * ffn * 4
    assert ws[5] < ws[4]
    assert ws[5] < 2 * 10 * 2 * ffn * 4


def test_static_scratch_limit_stated_in_header():
    """The header's statement of the fixed scratch array's reach: at the
    Mixtral shape every batch of up to 81 tokens fits, 82 does not, and a
    larger batch can fit again (the fit follows the tile plan)."""
    from sparse_mixture_experts_58_b300 import moe
    hdr = re.sub(r"\s*\n\s*\*\s*", " ", open(HEADER).read())
    assert "every batch of up to 81 tokens fits" in hdr
    fits = [moe.workspace_bytes(T, 4096, 14336, 8, 2, moe.BF16) <= moe.STATIC_SCRATCH_BYTES
            for T in range(1, 200)]
    assert all(fits[:81]) and not fits[81]
    assert any(fits[82:])


def test_graph_cache_stats_without_device_work():
    """The cache counters are readable with no GPU work (all zero before any
    forward call in this process); a null pointer is an argument error."""
    from sparse_mixture_experts_58_b300 import moe
    st = moe.graph_cache_stats()
    assert set(st) == {"entries", "replays", "captures", "direct_calls", "evictions"}
    assert all(v >= 0 for v in st.values())
    assert moe.lib().moe_graph_cache_stats(None, 0) == moe.ERR_ARG
