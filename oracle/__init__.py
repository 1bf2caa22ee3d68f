"""CPU oracle for the Mixtral sparse mixture-of-experts feed-forward layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and
its ``--impl reference`` arm) may.  It wraps ``moe_oracle.c`` (plain C, double
accumulation, compiled with gcc) through ctypes and shares no code with the
CUDA library.

Arrays are numpy: fp32 tensors as ``float32``, bf16 tensors as ``uint16`` bit
patterns.  Layouts: x [T,d], W_g [E,d], W1/W3 [E,ffn,d], W2 [E,d,ffn].

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
closed forms, brute force and invariants that the pages fix; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1

# No -ffast-math and no FMA contraction: the arithmetic is the source's, in order.
CFLAGS = ["-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
          "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra"]


def build(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc; returns the shared-object path."""
    cmd = ["gcc", *CFLAGS, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _declare(lib):
    c_void_p, c_int = ctypes.c_void_p, ctypes.c_int
    lib.oracle_moe_forward.argtypes = [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
        c_int, c_int, c_int, c_int, c_int, c_int,
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int]
    lib.oracle_moe_forward.restype = c_int
    lib.oracle_moe_forward_ex.argtypes = [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
        c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int]
    lib.oracle_moe_forward_ex.restype = c_int
    lib.oracle_router.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_int,
                                  c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]
    lib.oracle_router.restype = c_int
    lib.oracle_route.argtypes = [c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.oracle_route.restype = c_int
    lib.oracle_rmsnorm.argtypes = [c_void_p, c_int, c_int, ctypes.c_double, c_int, c_void_p]
    lib.oracle_rmsnorm.restype = c_int
    lib.oracle_add.argtypes = [c_void_p, c_void_p, ctypes.c_size_t, c_int, c_void_p]
    lib.oracle_add.restype = c_int
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = c_int
    lib.oracle_moe_backward.argtypes = [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
        c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
        c_int, c_int, c_int]
    lib.oracle_moe_backward.restype = c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` selects
    another build of the same source (the mutation tests use this)."""
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB) or
                     os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
            if stale:
                build()
            _lib = Oracle(_declare(ctypes.CDLL(_LIB)))
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _dt_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {a.dtype}")


class Oracle:
    """Thin ctypes marshalling over one build of ``moe_oracle.c``."""

    def __init__(self, lib):
        self.lib = lib

    def max_threads(self) -> int:
        return self.lib.oracle_max_threads()

    def moe_forward(self, x, Wg, W1, W3, W2, k, bias=None, threads=0, exact=False,
                    gating=0, capacity=0, drop_renorm=0):
        """Whole layer.  Returns (out, logits fp32 [T,E], idx int32 [T,k],
        gates float64 [T,k] before any drop); ``out`` has x's element type.
        With ``exact=True`` a fifth item is the float64 result before
        rounding.  gating 0: softmax over the kept logits; 1: softmax over all
        logits, kept ones not renormalised.  capacity: selections each expert
        keeps, in token order (0: all); drop_renorm: dropped slots' gate mass
        lost (0) or spread over the token's kept slots (1)."""
        x = np.ascontiguousarray(x)
        dt = _dt_code(x)
        T, d = x.shape
        E = Wg.shape[0]
        Wg = np.ascontiguousarray(Wg)
        W1 = [np.ascontiguousarray(w) for w in W1]
        W3 = [np.ascontiguousarray(w) for w in W3]
        W2 = [np.ascontiguousarray(w) for w in W2]
        ffn = W1[0].shape[0]
        assert len(W1) == len(W3) == len(W2) == E
        for w in (Wg, *W1, *W3, *W2):
            assert w.dtype == x.dtype
        assert Wg.shape == (E, d)
        assert all(w.shape == (ffn, d) for w in W1 + W3)
        assert all(w.shape == (d, ffn) for w in W2)
        arr = ctypes.c_void_p * E
        p1 = arr(*[w.ctypes.data for w in W1])
        p3 = arr(*[w.ctypes.data for w in W3])
        p2 = arr(*[w.ctypes.data for w in W2])
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        out = np.empty_like(x)
        logits = np.empty((T, E), np.float32)
        idx = np.empty((T, k), np.int32)
        gates = np.empty((T, k), np.float64)
        ex = np.empty((T, d), np.float64) if exact else None
        rc = self.lib.oracle_moe_forward_ex(
            _ptr(x), _ptr(Wg), _ptr(b), p1, p3, p2, T, d, ffn, E, k, dt, int(gating),
            int(capacity), int(drop_renorm), _ptr(out), _ptr(logits), _ptr(idx), _ptr(gates),
            _ptr(ex), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_moe_forward failed: {rc}")
        if exact:
            return out, logits, idx, gates, ex
        return out, logits, idx, gates

    def moe_backward(self, x, Wg, W1, W3, W2, k, dout, bias=None, threads=0, rows1=None,
                     rows2=None, weights=True):
        """Gradients of sum(dout * layer(x)) (gating 0, no capacity limit), in
        float64: returns dict(dx [T,d], dWg [E,d], dW1, dW3 (lists of E arrays
        [c1-c0, d]) and dW2 (list of [n1-n0, ffn])).  rows1 = (c0, c1) and
        rows2 = (n0, n1) restrict the weight-gradient rows (default: all);
        weights=False skips dW1/dW3/dW2."""
        x = np.ascontiguousarray(x)
        dt = _dt_code(x)
        T, d = x.shape
        E = Wg.shape[0]
        Wg = np.ascontiguousarray(Wg)
        W1 = [np.ascontiguousarray(w) for w in W1]
        W3 = [np.ascontiguousarray(w) for w in W3]
        W2 = [np.ascontiguousarray(w) for w in W2]
        dout = np.ascontiguousarray(dout)
        ffn = W1[0].shape[0]
        assert dout.shape == (T, d) and dout.dtype == x.dtype
        for w in (Wg, *W1, *W3, *W2):
            assert w.dtype == x.dtype
        c0, c1 = rows1 if rows1 is not None else (0, ffn)
        n0, n1 = rows2 if rows2 is not None else (0, d)
        arr = ctypes.c_void_p * E
        p1 = arr(*[w.ctypes.data for w in W1])
        p3 = arr(*[w.ctypes.data for w in W3])
        p2 = arr(*[w.ctypes.data for w in W2])
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        dx = np.empty((T, d), np.float64)
        dWg = np.empty((E, d), np.float64)
        g1 = [np.empty((c1 - c0, d), np.float64) for _ in range(E)] if weights else []
        g3 = [np.empty((c1 - c0, d), np.float64) for _ in range(E)] if weights else []
        g2 = [np.empty((n1 - n0, ffn), np.float64) for _ in range(E)] if weights else []
        q1 = arr(*[a.ctypes.data for a in g1]) if weights else None
        q3 = arr(*[a.ctypes.data for a in g3]) if weights else None
        q2 = arr(*[a.ctypes.data for a in g2]) if weights else None
        rc = self.lib.oracle_moe_backward(
            _ptr(x), _ptr(Wg), _ptr(b), p1, p3, p2, T, d, ffn, E, k, dt, _ptr(dout), _ptr(dx),
            _ptr(dWg), q1, q3, q2, int(c0), int(c1), int(n0), int(n1), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_moe_backward failed: {rc}")
        return dict(dx=dx, dWg=dWg, dW1=g1, dW3=g3, dW2=g2)

    def router(self, x, Wg, k, bias=None, gating=0):
        x = np.ascontiguousarray(x)
        dt = _dt_code(x)
        T, d = x.shape
        E = Wg.shape[0]
        Wg = np.ascontiguousarray(Wg)
        assert Wg.dtype == x.dtype and Wg.shape == (E, d)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        logits = np.empty((T, E), np.float32)
        idx = np.empty((T, k), np.int32)
        gates = np.empty((T, k), np.float64)
        rc = self.lib.oracle_router(_ptr(x), _ptr(Wg), _ptr(b), T, d, E, k, dt, int(gating),
                                    _ptr(logits), _ptr(idx), _ptr(gates))
        if rc != 0:
            raise RuntimeError(f"oracle_router failed: {rc}")
        return logits, idx, gates

    def route(self, logits, k, gating=0, capacity=0):
        """Grouping from given fp32 logits: (idx, gates, counts, offsets, perm,
        inv); with a capacity, only kept selections get rows (perm holds
        offsets[E] valid entries, inv is -1 for dropped ones)."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        gates = np.empty((T, k), np.float64)
        counts = np.empty(E, np.int32)
        offsets = np.empty(E + 1, np.int32)
        perm = np.full(T * k, -1, np.int32)
        inv = np.empty(T * k, np.int32)
        rc = self.lib.oracle_route(_ptr(logits), T, E, k, int(gating), int(capacity), _ptr(idx),
                                   _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(perm),
                                   _ptr(inv))
        if rc != 0:
            raise RuntimeError(f"oracle_route failed: {rc}")
        return idx, gates, counts, offsets, perm[:int(offsets[-1])], inv

    def rmsnorm(self, x, eps=1e-5):
        x = np.ascontiguousarray(x)
        dt = _dt_code(x)
        T, d = x.shape
        y = np.empty_like(x)
        rc = self.lib.oracle_rmsnorm(_ptr(x), T, d, float(eps), dt, _ptr(y))
        if rc != 0:
            raise RuntimeError(f"oracle_rmsnorm failed: {rc}")
        return y

    def add(self, a, b):
        a = np.ascontiguousarray(a)
        b = np.ascontiguousarray(b)
        assert a.dtype == b.dtype and a.shape == b.shape
        z = np.empty_like(a)
        rc = self.lib.oracle_add(_ptr(a), _ptr(b), a.size, _dt_code(a), _ptr(z))
        if rc != 0:
            raise RuntimeError(f"oracle_add failed: {rc}")
        return z

    def to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_double_to_bf16(float(v)))

    def from_bf16(self, h: int) -> float:
        return float(self.lib.oracle_bf16_to_double(int(h)))


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
