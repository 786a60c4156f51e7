"""ctypes binding of libxattn (include/xattn.h).

Argument marshalling only: tensors become device pointers, the current torch CUDA
stream becomes the ``stream`` argument, and a non-OK status raises ``XattnError``.
Every step of the attention runs in libxattn's kernels; there is no fallback. If
the library has not been built, importing this module raises at once.

The functions named like the C entry points (``xattn_fwd``, ``xattn_bwd``, ...)
take the same arguments in the same order; tensor arguments may be torch tensors
or raw integer addresses. ``attention_fwd`` / ``attention_bwd`` allocate the
outputs with torch and call them.
"""
from __future__ import annotations

import ctypes
import enum
import os

from . import build as _build

# XATTN_LIBRARY may name another build of libxattn (for example an instrumented one).
_LIB_PATH = os.environ.get("XATTN_LIBRARY") or _build.LIB

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libxattn is not built ({_LIB_PATH} missing): run "
        "`python -c 'import __graft_entry__ as g; g.build()'` or "
        "`python bwd_xattn_fwd_gb300/build.py` first")

_lib = ctypes.CDLL(_LIB_PATH)


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL_PTR = 1
    ERR_BAD_SHAPE = 2
    ERR_GROUP = 3
    ERR_UNSUPPORTED_HD = 4
    ERR_MISALIGNED = 5
    ERR_CUDA = 6
    ERR_NO_DEVICE_SUPPORT = 7
    ERR_DEVICE_TIMEOUT = 8
    ERR_BAD_SCALE = 9
    ERR_WORKSPACE = 10
    ERR_SCRATCH_LIMIT = 11


class XattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name} ({status_string(status)})")


_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "xattn_fwd": [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp],
    "xattn_bwd": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp],
    "xattn_bwd_noalloc": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp],
    "xattn_bwd_preprocess": [_vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _sz, _vp],
    "xattn_bwd_main": [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _sz, _vp],
    "xattn_bwd_dq_convert": [_i, _i, _i, _i, _f, _vp, _vp, _sz, _vp],
    "xattn_bwd_deterministic": [_vp] * 5 + [_vp] + [_i] * 5 + [_f] + [_vp] * 4,
    "xattn_fwd_f32": [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp],
    "xattn_bwd_f32": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp],
    "xattn_decode": [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp],
    "xattn_check_device_status": [_vp],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
_lib.xattn_status_string.argtypes = [ctypes.c_int]
_lib.xattn_status_string.restype = ctypes.c_char_p
_lib.xattn_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i]
_lib.xattn_bwd_workspace_bytes.restype = ctypes.c_size_t
_lib.xattn_bwd_dq_mode.argtypes = [_i, _i, _i, _i, _i]
_lib.xattn_bwd_dq_mode.restype = ctypes.c_int
_lib.xattn_decode_runs.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.xattn_decode_runs.restype = ctypes.c_int
_lib.xattn_build_flags.argtypes = []
_lib.xattn_build_flags.restype = ctypes.c_int
_lib.xattn_selftest_bounds_check.argtypes = [_vp]
_lib.xattn_selftest_bounds_check.restype = ctypes.c_int

BWD_FUSED_DQ, BWD_RESIDENT_DQ, BWD_QUERY_DQ = 0, 1, 2
BUILD_DEVICE_CHECKS = 1             # xattn_build_flags bit: on-device bounds checks compiled in
ERR_DEVICE_TIMEOUT, ERR_DEVICE_BOUNDS = 8, 12


def lib_path() -> str:
    return _LIB_PATH


def status_string(status: int) -> str:
    return _lib.xattn_status_string(int(status)).decode()


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    rc = getattr(_lib, name)(*args)
    if rc != 0:
        raise XattnError(rc, name)


# ---- the C entry points, same names and argument order -------------------------------

def xattn_fwd(q, k, v, B, S, nh, nkv, hd, scale, o, lse, stream=None):
    _call("xattn_fwd", _addr(q), _addr(k), _addr(v), B, S, nh, nkv, hd, scale, _addr(o),
          _addr(lse), _stream(stream))


def xattn_bwd(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream=None):
    _call("xattn_bwd", _addr(q), _addr(k), _addr(v), _addr(o), _addr(dO), _addr(lse), B, S, nh,
          nkv, hd, scale, _addr(dq), _addr(dk), _addr(dv), _stream(stream))


def xattn_bwd_deterministic(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream=None):
    """xattn_bwd with a bit-reproducible dQ (query-stationary dQ recompute, no atomics)."""
    _call("xattn_bwd_deterministic", _addr(q), _addr(k), _addr(v), _addr(o), _addr(dO), _addr(lse),
          B, S, nh, nkv, hd, scale, _addr(dq), _addr(dk), _addr(dv), _stream(stream))


def xattn_bwd_noalloc(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream=None):
    """xattn_bwd using the library's fixed device scratch array instead of allocating
    (for callers that may not allocate device memory). Sizes whose scratch exceeds
    NOALLOC_SCRATCH_BYTES raise ERR_SCRATCH_LIMIT; overlapping calls race on the array."""
    _call("xattn_bwd_noalloc", _addr(q), _addr(k), _addr(v), _addr(o), _addr(dO), _addr(lse), B,
          S, nh, nkv, hd, scale, _addr(dq), _addr(dk), _addr(dv), _stream(stream))


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024   # XATTN_NOALLOC_SCRATCH_BYTES in xattn.h


def xattn_bwd_workspace_bytes(B, S, nh, hd) -> int:
    return int(_lib.xattn_bwd_workspace_bytes(B, S, nh, hd))


def xattn_decode_runs(B, T, nh, nkv, hd, num_sms) -> int:
    """Key runs per (sequence, kv head) that xattn_decode uses on num_sms SMs (-1: rejected)."""
    return int(_lib.xattn_decode_runs(B, T, nh, nkv, hd, num_sms))


def xattn_bwd_dq_mode(S, nh, nkv, hd, deterministic=False) -> int:
    """Which backward xattn_bwd (or, with deterministic, xattn_bwd_deterministic) runs for
    these sizes (BWD_FUSED_DQ, BWD_RESIDENT_DQ, BWD_QUERY_DQ), or -1 for sizes it rejects."""
    return int(_lib.xattn_bwd_dq_mode(S, nh, nkv, hd, int(bool(deterministic))))


def xattn_bwd_preprocess(o, dO, lse, B, S, nh, hd, scale, workspace, workspace_bytes, stream=None):
    _call("xattn_bwd_preprocess", _addr(o), _addr(dO), _addr(lse), B, S, nh, hd, scale,
          _addr(workspace), workspace_bytes, _stream(stream))


def xattn_bwd_main(q, k, v, dO, B, S, nh, nkv, hd, scale, dk, dv, workspace, workspace_bytes,
                   stream=None):
    _call("xattn_bwd_main", _addr(q), _addr(k), _addr(v), _addr(dO), B, S, nh, nkv, hd, scale,
          _addr(dk), _addr(dv), _addr(workspace), workspace_bytes, _stream(stream))


def xattn_bwd_dq_convert(B, S, nh, hd, scale, dq, workspace, workspace_bytes, stream=None):
    _call("xattn_bwd_dq_convert", B, S, nh, hd, scale, _addr(dq), _addr(workspace), workspace_bytes,
          _stream(stream))


def xattn_fwd_f32(q, k, v, B, S, nh, nkv, hd, scale, o, lse, stream=None):
    _call("xattn_fwd_f32", _addr(q), _addr(k), _addr(v), B, S, nh, nkv, hd, scale, _addr(o),
          _addr(lse), _stream(stream))


def xattn_bwd_f32(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream=None):
    _call("xattn_bwd_f32", _addr(q), _addr(k), _addr(v), _addr(o), _addr(dO), _addr(lse), B, S,
          nh, nkv, hd, scale, _addr(dq), _addr(dk), _addr(dv), _stream(stream))


def xattn_decode(q, k_cache, v_cache, B, T, nh, nkv, hd, scale, o, lse, stream=None):
    _call("xattn_decode", _addr(q), _addr(k_cache), _addr(v_cache), B, T, nh, nkv, hd, scale, _addr(o),
          _addr(lse), _stream(stream))


def xattn_selftest_wait_timeout(limit_ns, stream=None):
    fn = _lib.xattn_selftest_wait_timeout
    fn.argtypes = [ctypes.c_ulonglong, _vp]
    fn.restype = ctypes.c_int
    st = fn(int(limit_ns), _stream(stream))
    if st != 0:
        raise XattnError(st, "xattn_selftest_wait_timeout")


def xattn_build_flags() -> int:
    """Bit BUILD_DEVICE_CHECKS is set in a debug build (on-device bounds checks)."""
    return int(_lib.xattn_build_flags())


def xattn_selftest_bounds_check(stream=None):
    st = _lib.xattn_selftest_bounds_check(_stream(stream))
    if st != 0:
        raise XattnError(st, "xattn_selftest_bounds_check")


def xattn_status_string(status: int) -> str:
    return status_string(status)


def xattn_check_device_status(stream=None) -> int:
    """Synchronises the stream; returns the device status (0 = OK) and clears it."""
    return int(_lib.xattn_check_device_status(_stream(stream)))


# ---- tensor-level helpers ---------------------------------------------------------------

def _dims(q, k):
    B, S, nh, hd = q.shape
    nkv = k.shape[2]
    return int(B), int(S), int(nh), int(nkv), int(hd)


def attention_fwd(q, k, v, scale=None, stream=None):
    """(o, lse) for contiguous CUDA tensors q [B,S,nh,hd], k/v [B,S,nkv,hd] (bf16 or fp32)."""
    import torch
    B, S, nh, nkv, hd = _dims(q, k)
    scale = float(hd ** -0.5 if scale is None else scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, S, nh), dtype=torch.float32, device=q.device)
    if q.dtype == torch.bfloat16:
        xattn_fwd(q, k, v, B, S, nh, nkv, hd, scale, o, lse, stream)
    elif q.dtype == torch.float32:
        xattn_fwd_f32(q, k, v, B, S, nh, nkv, hd, scale, o, lse, stream)
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    return o, lse


def attention_bwd(q, k, v, o, dO, lse, scale=None, stream=None, deterministic=False):
    """(dq, dk, dv) for the tensors of attention_fwd and the output gradient dO.
    deterministic (bf16): dQ bit-reproducible as well, at the cost of a second recompute."""
    import torch
    B, S, nh, nkv, hd = _dims(q, k)
    scale = float(hd ** -0.5 if scale is None else scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if q.dtype == torch.bfloat16:
        fn = xattn_bwd_deterministic if deterministic else xattn_bwd
        fn(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream)
    elif q.dtype == torch.float32:
        xattn_bwd_f32(q, k, v, o, dO, lse, B, S, nh, nkv, hd, scale, dq, dk, dv, stream)
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    return dq, dk, dv


def attention_decode(q, k_cache, v_cache, scale=None, stream=None):
    """(o [B,nh,hd], lse [B,nh]) for one new query per sequence: q [B,nh,hd] against the
    cached k/v [B,T,nkv,hd] (bf16, contiguous CUDA tensors)."""
    import torch
    B, nh, hd = (int(x) for x in q.shape)
    T, nkv = int(k_cache.shape[1]), int(k_cache.shape[2])
    scale = float(hd ** -0.5 if scale is None else scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, nh), dtype=torch.float32, device=q.device)
    xattn_decode(q, k_cache, v_cache, B, T, nh, nkv, hd, scale, o, lse, stream)
    return o, lse
