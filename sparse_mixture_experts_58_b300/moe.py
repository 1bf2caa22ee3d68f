"""Python binding over libmoe.so (include/moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; torch supplies
device memory and the current stream.  Importing this module without the
built library raises -- there is no fallback.

Tensors: x / out [T, d]; W_g [E, d]; W1, W3 [E, ffn, d]; W2 [E, d, ffn]
(one contiguous tensor per projection, or a list of E per-expert tensors);
bf16 or fp32, CUDA, contiguous.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libmoe.so is not built ({LIB_PATH}); run "
        "`python -m sparse_mixture_experts_58_b300.build` (there is no fallback path)")

_lib = ctypes.CDLL(LIB_PATH)

F32, BF16 = 0, 1
OK, ERR_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = 0, -1, -2, -3, -4, -5
MAX_EXPERTS = 64

_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_P = ctypes.POINTER


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("moe_strerror", ctypes.c_char_p, _i)
_sig("moe_version", _i)
_sig("moe_workspace_bytes", _i, _i, _i, _i, _i, _i, _i, _P(_sz))
_sig("moe_forward", _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp)
_sig("moe_forward_host_io", _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
     _i, _i, _i, _i, _i, _i, _vp, _sz, _vp)
_sig("moe_router", _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp)
_sig("moe_route_workspace_bytes", _i, _i, _i, _i, _P(_sz))
_sig("moe_route_from_logits", _i, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp)
_sig("moe_permute", _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp)
_sig("moe_expert_swiglu", _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp)
_sig("moe_down_splits", _i, _i, _i, _i, _i, _i, _i, _P(_i))
_sig("moe_expert_down", _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp)
_sig("moe_combine", _i, _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp)
_sig("moe_add_rmsnorm", _i, _vp, _vp, _vp, _i, _i, ctypes.c_float, _i, _vp)
_sig("moe_device_status", _i, _vp, _P(_i), _i)
_sig("moe_selftest_wait_timeout", _i, ctypes.c_uint, _vp)
_sig("moe_forward_launches", _i, _i, _i, _i, _i, _i, _i, _P(_i))
_sig("moe_forward_static_scratch", _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
     _vp, _vp)
STATIC_SCRATCH_BYTES = 16 << 20


class GraphStats(ctypes.Structure):
    """moe_graph_stats: the launch-graph cache's counters."""
    _fields_ = [("entries", ctypes.c_longlong), ("replays", ctypes.c_longlong),
                ("captures", ctypes.c_longlong), ("direct_calls", ctypes.c_longlong),
                ("evictions", ctypes.c_longlong)]


_sig("moe_graph_cache_stats", _i, _P(GraphStats), _i)


class Options(ctypes.Structure):
    """moe_options: gating (0 softmax over kept, 1 full softmax then top-k),
    capacity (rows per expert, 0 = no limit), drop_policy (0 lose, 1
    renormalise)."""
    _fields_ = [("gating", ctypes.c_int), ("capacity", ctypes.c_int),
                ("drop_policy", ctypes.c_int)]


GATING_TOPK_SOFTMAX, GATING_SOFTMAX_TOPK = 0, 1
DROP_LOSE, DROP_RENORMALIZE = 0, 1
MAX_TOPK = 8

_sig("moe_forward_ex", _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _P(Options),
     _vp, _vp, _sz, _vp)
_sig("moe_capacity", _i, ctypes.c_double, _i, _i, _i, _P(_i))
_sig("moe_block_forward", _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_float,
     _P(Options), _vp, _sz, _vp)
_sig("moe_backward_workspace_bytes", _i, _i, _i, _i, _i, _i, _i, _P(_sz))
_sig("moe_backward", _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
     _vp, _vp, _vp, _sz, _vp)
_sig("moe_route_from_logits_ex", _i, _vp, _i, _i, _i, _P(Options), _vp, _vp, _vp, _vp, _vp, _vp,
     _vp, _sz, _vp)

EXPORTED = [
    "moe_strerror", "moe_version", "moe_workspace_bytes", "moe_forward", "moe_forward_host_io",
    "moe_router", "moe_route_workspace_bytes", "moe_route_from_logits", "moe_permute",
    "moe_expert_swiglu", "moe_down_splits", "moe_expert_down", "moe_combine",
    "moe_add_rmsnorm", "moe_device_status", "moe_selftest_wait_timeout", "moe_forward_launches",
    "moe_forward_static_scratch", "moe_forward_ex", "moe_capacity", "moe_route_from_logits_ex",
    "moe_block_forward", "moe_backward_workspace_bytes", "moe_backward",
    "moe_graph_cache_stats",
]


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


def strerror(code: int) -> str:
    return _lib.moe_strerror(code).decode()


def _check(code, where):
    if code != OK:
        raise MoeError(code, where)


def lib():
    return _lib


def graph_cache_stats(reset=False) -> dict:
    """The launch-graph cache's counters (moe_graph_cache_stats)."""
    st = GraphStats()
    _check(_lib.moe_graph_cache_stats(ctypes.byref(st), int(bool(reset))),
           "moe_graph_cache_stats")
    return {name: getattr(st, name) for name, _ in GraphStats._fields_}


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _expert_ptrs(W, E):
    if isinstance(W, (list, tuple)):
        assert len(W) == E
        return (ctypes.c_void_p * E)(*[w.data_ptr() for w in W])
    assert W.shape[0] == E and W.is_contiguous()
    step = W[0].numel() * W.element_size()
    base = W.data_ptr()
    return (ctypes.c_void_p * E)(*[base + e * step for e in range(E)])


def _shape(x, Wg, W1):
    T, d = x.shape
    E = Wg.shape[0]
    ffn = (W1[0] if isinstance(W1, (list, tuple)) else W1[0]).shape[0]
    return T, d, ffn, E


def workspace_bytes(T, d, ffn, E, k, dtype) -> int:
    n = ctypes.c_size_t()
    _check(_lib.moe_workspace_bytes(T, d, ffn, E, k, dtype, ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def forward_launches(T, d, ffn, E, k, dtype) -> int:
    n = ctypes.c_int()
    _check(_lib.moe_forward_launches(T, d, ffn, E, k, dtype, ctypes.byref(n)), "moe_forward_launches")
    return n.value


def down_splits(T, d, ffn, E, k, dtype) -> int:
    n = ctypes.c_int()
    _check(_lib.moe_down_splits(T, d, ffn, E, k, dtype, ctypes.byref(n)), "moe_down_splits")
    return n.value


def alloc_workspace(T, d, ffn, E, k, dtype, device="cuda") -> torch.Tensor:
    return torch.empty(max(workspace_bytes(T, d, ffn, E, k, dtype), 256), dtype=torch.uint8,
                       device=device)


class Workspace:
    """Reusable device scratch, grown on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def capacity(factor, T, k, E) -> int:
    """ceil(factor * T * k / E) through moe_capacity (0 for factor <= 0)."""
    c = ctypes.c_int()
    _check(_lib.moe_capacity(float(factor), T, k, E, ctypes.byref(c)), "moe_capacity")
    return c.value


def forward(x, Wg, W1, W3, W2, k=2, bias=None, out=None, workspace=None, stream=None,
            gating=0, capacity=0, drop_policy=0):
    """out = MoE(x) through moe_forward, or moe_forward_ex when a routing
    option is set (gating, capacity in rows per expert, drop_policy)."""
    T, d, ffn, E = _shape(x, Wg, W1)
    dt = _dt(x)
    if out is None:
        out = torch.empty_like(x)
    need = workspace_bytes(T, d, ffn, E, k, dt)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    p1, p3, p2 = _expert_ptrs(W1, E), _expert_ptrs(W3, E), _expert_ptrs(W2, E)
    if gating or capacity or drop_policy:
        opt = Options(int(gating), int(capacity), int(drop_policy))
        _check(_lib.moe_forward_ex(_ptr(x), _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn, E, k, dt,
                                   ctypes.byref(opt), _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_forward_ex")
        return out
    _check(_lib.moe_forward(_ptr(x), _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn, E, k, dt,
                            _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_forward")
    return out


def block_forward(x, Wg, W1, W3, W2, k=2, bias=None, eps=1e-5, workspace=None, stream=None,
                  gating=0, capacity=0, drop_policy=0):
    """x <- x + MoE(RMSNorm(x)) in place through moe_block_forward (RMSNorm
    fused into the router and the grouping, the residual add into the
    combine); returns x."""
    T, d, ffn, E = _shape(x, Wg, W1)
    dt = _dt(x)
    need = workspace_bytes(T, d, ffn, E, k, dt)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    p1, p3, p2 = _expert_ptrs(W1, E), _expert_ptrs(W3, E), _expert_ptrs(W2, E)
    opt = Options(int(gating), int(capacity), int(drop_policy))
    _check(_lib.moe_block_forward(_ptr(x), _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn, E, k, dt,
                                  float(eps), ctypes.byref(opt), _ptr(ws), ws.numel(),
                                  _stream(stream)), "moe_block_forward")
    return x


def backward_workspace_bytes(T, d, ffn, E, k, dtype) -> int:
    n = ctypes.c_size_t()
    _check(_lib.moe_backward_workspace_bytes(T, d, ffn, E, k, dtype, ctypes.byref(n)),
           "moe_backward_workspace_bytes")
    return n.value


def backward(x, Wg, W1, W3, W2, dout, k=2, bias=None, workspace=None, stream=None, grads=None):
    """Gradients of sum(dout * layer(x)) through moe_backward: returns dict
    dx [T,d] (x's dtype), dWg [E,d], dW1, dW3 [E,ffn,d] and dW2 [E,d,ffn]
    (fp32).  ``grads`` may pass that dict to be overwritten."""
    T, d, ffn, E = _shape(x, Wg, W1)
    dt = _dt(x)
    dev = x.device
    if grads is None:
        grads = dict(dx=torch.empty_like(x),
                     dWg=torch.empty(E, d, dtype=torch.float32, device=dev),
                     dW1=torch.empty(E, ffn, d, dtype=torch.float32, device=dev),
                     dW3=torch.empty(E, ffn, d, dtype=torch.float32, device=dev),
                     dW2=torch.empty(E, d, ffn, dtype=torch.float32, device=dev))
    need = backward_workspace_bytes(T, d, ffn, E, k, dt)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    p1, p3, p2 = _expert_ptrs(W1, E), _expert_ptrs(W3, E), _expert_ptrs(W2, E)
    g1, g3, g2 = (_expert_ptrs(grads[key], E) for key in ("dW1", "dW3", "dW2"))
    _check(_lib.moe_backward(_ptr(x), _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn, E, k, dt,
                             _ptr(dout), _ptr(grads["dx"]), _ptr(grads["dWg"]), g1, g3, g2,
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_backward")
    return grads


def forward_host_io(x_host, Wg, W1, W3, W2, k=2, bias=None, out_host=None, x_dev=None,
                    out_dev=None, workspace=None, stream=None):
    """Tokens and result in (pinned) host memory; copies are enqueued by the
    library on the stream.  Synchronise before reading ``out_host``."""
    T, d, ffn, E = _shape(x_host, Wg, W1)
    dt = _dt(x_host)
    dev = Wg.device
    if out_host is None:
        out_host = torch.empty_like(x_host, pin_memory=True)
    if x_dev is None:
        x_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
    if out_dev is None:
        out_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
    need = workspace_bytes(T, d, ffn, E, k, dt)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    p1, p3, p2 = _expert_ptrs(W1, E), _expert_ptrs(W3, E), _expert_ptrs(W2, E)
    _check(_lib.moe_forward_host_io(_ptr(x_host), _ptr(out_host), _ptr(x_dev), _ptr(out_dev),
                                    _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn, E, k, dt,
                                    _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward_host_io")
    return out_host


def router(x, Wg, k=2, bias=None, stream=None):
    T, d = x.shape
    E = Wg.shape[0]
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device)
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    gates = torch.empty(T, k, dtype=torch.float32, device=x.device)
    _check(_lib.moe_router(_ptr(x), _ptr(Wg), _ptr(bias), T, d, E, k, _dt(x), _ptr(logits),
                           _ptr(idx), _ptr(gates), _stream(stream)), "moe_router")
    return logits, idx, gates


def route_from_logits(logits, k=2, stream=None, gating=0, capacity=0):
    """(idx, gates, counts, offsets, perm, inv); with a capacity, counts are
    the kept counts, perm has offsets[E] valid rows, inv is -1 when dropped."""
    T, E = logits.shape
    dev = logits.device
    n = ctypes.c_size_t()
    _check(_lib.moe_route_workspace_bytes(T, E, k, ctypes.byref(n)), "moe_route_workspace_bytes")
    ws = torch.empty(max(n.value, 256), dtype=torch.uint8, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    gates = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    if gating or capacity:
        opt = Options(int(gating), int(capacity), 0)
        _check(_lib.moe_route_from_logits_ex(_ptr(logits), T, E, k, ctypes.byref(opt), _ptr(idx),
                                             _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(perm),
                                             _ptr(inv), _ptr(ws), ws.numel(), _stream(stream)),
               "moe_route_from_logits_ex")
    else:
        _check(_lib.moe_route_from_logits(_ptr(logits), T, E, k, _ptr(idx), _ptr(gates),
                                          _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                                          _ptr(ws), ws.numel(), _stream(stream)),
               "moe_route_from_logits")
    return idx, gates, counts, offsets, perm[:T * k], inv[:T * k]


def permute(x, perm, k=2, rows=None, stream=None):
    """x_perm[r] = x[perm[r] // k] for r < rows (default T*k; the kept count
    under a capacity limit).  x_perm has T*k rows."""
    T, d = x.shape
    rows = T * k if rows is None else int(rows)
    x_perm = torch.empty(T * k, d, dtype=x.dtype, device=x.device)
    _check(_lib.moe_permute(_ptr(x), _ptr(perm), rows, T, d, k, _dt(x), _ptr(x_perm),
                            _stream(stream)), "moe_permute")
    return x_perm


def expert_swiglu(x_perm, offsets, W1, W3, stream=None):
    rows, d = x_perm.shape
    E = offsets.numel() - 1
    ffn = (W1[0] if isinstance(W1, (list, tuple)) else W1[0]).shape[0]
    h = torch.empty(rows, ffn, dtype=x_perm.dtype, device=x_perm.device)
    _check(_lib.moe_expert_swiglu(_ptr(x_perm), _ptr(offsets), _expert_ptrs(W1, E),
                                  _expert_ptrs(W3, E), rows, d, ffn, E, _dt(x_perm), _ptr(h),
                                  _stream(stream)), "moe_expert_swiglu")
    return h


def expert_down(h, offsets, W2, T, k=2, stream=None):
    rows, ffn = h.shape
    E = offsets.numel() - 1
    d = (W2[0] if isinstance(W2, (list, tuple)) else W2[0]).shape[0]
    S = down_splits(T, d, ffn, E, k, _dt(h))
    y = torch.empty(S, rows, d, dtype=torch.float32, device=h.device)
    _check(_lib.moe_expert_down(_ptr(h), _ptr(offsets), _expert_ptrs(W2, E), T, d, ffn, E, k,
                                _dt(h), _ptr(y), _stream(stream)), "moe_expert_down")
    return y


def combine(y_partial, gates, inv, T, k=2, dtype=torch.bfloat16, stream=None):
    S, rows, d = y_partial.shape
    out = torch.empty(T, d, dtype=dtype, device=y_partial.device)
    _check(_lib.moe_combine(_ptr(y_partial), S, _ptr(gates), _ptr(inv), T, d, k,
                            BF16 if dtype == torch.bfloat16 else F32, _ptr(out), _stream(stream)),
           "moe_combine")
    return out


def add_rmsnorm(x, add=None, xn=None, eps=1e-5, stream=None):
    """x <- x + add (in place, if add is given); returns RMSNorm(x) (gain 1)."""
    T, d = x.shape
    if xn is None:
        xn = torch.empty_like(x)
    _check(_lib.moe_add_rmsnorm(_ptr(x), _ptr(add), _ptr(xn), T, d, float(eps), _dt(x),
                                _stream(stream)), "moe_add_rmsnorm")
    return xn


def device_status(clear=True, stream=None) -> int:
    v = ctypes.c_int()
    _check(_lib.moe_device_status(_stream(stream), ctypes.byref(v), 1 if clear else 0),
           "moe_device_status")
    return v.value


def selftest_wait_timeout(limit_ns=1_000_000, stream=None):
    _check(_lib.moe_selftest_wait_timeout(int(limit_ns), _stream(stream)), "moe_selftest_wait_timeout")


def forward_static_scratch(x, Wg, W1, W3, W2, k=2, bias=None, out=None, stream=None):
    """out = MoE(x) through moe_forward_static_scratch: no workspace, the
    library's fixed per-device scratch instead (see include/moe.h)."""
    T, d, ffn, E = _shape(x, Wg, W1)
    if out is None:
        out = torch.empty_like(x)
    p1, p3, p2 = _expert_ptrs(W1, E), _expert_ptrs(W3, E), _expert_ptrs(W2, E)
    _check(_lib.moe_forward_static_scratch(_ptr(x), _ptr(Wg), _ptr(bias), p1, p3, p2, T, d, ffn,
                                           E, k, _dt(x), _ptr(out), _stream(stream)),
           "moe_forward_static_scratch")
    return out
