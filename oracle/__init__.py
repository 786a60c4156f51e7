"""Reference oracle for causal attention with grouped KV heads (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (libxattn and its binding in
``bwd_xattn_fwd_gb300``) neither imports it nor shares code with it.

Two independent formulations live here:

* ``OracleLib`` wraps ``xattn_oracle.c``: the plain fp64 definition, row by row
  (xtrain "演进总览" / docs/evolution.md, phase table rows T14 and T15).
* ``composed`` evaluates the same function the way the pages' composed path does
  (materialised causal scores, row softmax, matmul with V; full softmax Jacobian in
  the backward; GQA by literally repeating K/V): xtrain "Known Issues & Perf
  Backlog" (docs/known-issues.md), KI-1 fix, and evolution.md row T15.

Both take numpy float64 arrays in row-major [B, S, heads, hd].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()


def lib_path(mutation: int = 0) -> str:
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP) into oracle/_build/. Returns the path."""
    out = lib_path(mutation)
    with _lock:
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
            return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               f"-DORACLE_MUTATION={int(mutation)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_dbl_p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dbl_p)


class OracleLib:
    """ctypes handle on one build of the C oracle."""

    def __init__(self, mutation: int = 0):
        self.mutation = mutation
        self._lib = ctypes.CDLL(build(mutation))
        for name in ("xo_fwd", "xo_bwd", "xo_decode"):
            getattr(self._lib, name).restype = None
        self._lib.xo_mutation.restype = ctypes.c_int
        assert self._lib.xo_mutation() == mutation

    @staticmethod
    def _shape(q, k):
        B, S, nh, hd = q.shape
        Bk, Sk, nkv, hdk = k.shape
        if (Bk, Sk, hdk) != (B, S, hd) or nkv <= 0 or nh % nkv != 0:
            raise ValueError(f"bad shapes q{q.shape} k{k.shape}")
        return B, S, nh, nkv, hd

    def fwd(self, q, k, v, scale):
        """Returns (o [B,S,nh,hd], lse [B,S,nh]) in float64."""
        q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
        B, S, nh, nkv, hd = self._shape(q, k)
        o = np.empty_like(q)
        lse = np.empty((B, S, nh), dtype=np.float64)
        self._lib.xo_fwd(_ptr(q), _ptr(k), _ptr(v), B, S, nh, nkv, hd,
                         ctypes.c_double(scale), _ptr(o), _ptr(lse))
        return o, lse

    def bwd(self, q, k, v, dO, scale):
        """Returns (dq, dk, dv) in float64 for the loss sum(dO * O)."""
        q, k, v, dO = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, dO))
        B, S, nh, nkv, hd = self._shape(q, k)
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        self._lib.xo_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), B, S, nh, nkv, hd,
                         ctypes.c_double(scale), _ptr(dq), _ptr(dk), _ptr(dv))
        return dq, dk, dv


    def decode(self, q, k, v, scale):
        """One query per sequence against its T cached keys/values.

        q [B, nh, hd], k, v [B, T, nkv, hd] -> (o [B, nh, hd], lse [B, nh]) in float64.
        """
        q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
        B, nh, hd = q.shape
        Bk, T, nkv, hdk = k.shape
        if (Bk, hdk) != (B, hd) or v.shape != k.shape or T <= 0 or nkv <= 0 or nh % nkv != 0:
            raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
        o = np.empty_like(q)
        lse = np.empty((B, nh), dtype=np.float64)
        self._lib.xo_decode(_ptr(q), _ptr(k), _ptr(v), B, T, nh, nkv, hd, ctypes.c_double(scale),
                            _ptr(o), _ptr(lse))
        return o, lse


_default = None


def default() -> OracleLib:
    """The unmutated oracle (built on first use)."""
    global _default
    if _default is None:
        _default = OracleLib(0)
    return _default


def unit_slices(q, k, v, dO, b: int, kvh: int):
    """The independent sub-problem of batch b and kv head kvh.

    One (b, kv head) unit is itself an attention problem with B=1, nkv=1 and
    nh=group: its query heads read only that kv head, and its K/V gradients receive
    only that group's contributions.
    """
    nh, nkv = q.shape[2], k.shape[2]
    g = nh // nkv
    sl = slice(kvh * g, (kvh + 1) * g)
    return (q[b:b + 1, :, sl], k[b:b + 1, :, kvh:kvh + 1], v[b:b + 1, :, kvh:kvh + 1],
            dO[b:b + 1, :, sl])
