"""libxattn's C ABI without a GPU: the library loads, exports every entry point that
include/xattn.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xattn.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xattn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from bwd_xattn_fwd_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("xattn_fwd", "xattn_bwd", "xattn_fwd_f32", "xattn_bwd_f32", "xattn_status_string",
              "xattn_check_device_status"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_binding_exposes_the_same_names():
    from bwd_xattn_fwd_gb300 import xattn
    missing = [s for s in declared_symbols() if not callable(getattr(xattn, s, None))]
    assert not missing, missing


def test_status_strings(lib):
    lib.xattn_status_string.restype = ctypes.c_char_p
    seen = set()
    for code in range(0, 13):
        s = lib.xattn_status_string(code).decode()
        assert s and s != "unknown xattn status"
        seen.add(s)
    assert len(seen) == 13
    assert lib.xattn_status_string(99).decode() == "unknown xattn status"


def test_release_build_has_no_device_checks(lib):
    """The default build compiles the on-device bounds checks out (bit 0 of the flags);
    the debug build (build(debug=True)) is a separate library."""
    lib.xattn_build_flags.restype = ctypes.c_int
    assert lib.xattn_build_flags() == 0


def test_debug_build_compiles_and_reports_its_checks():
    """The debug build (XATTN_DEBUG) builds without a GPU and says so in its flags."""
    from bwd_xattn_fwd_gb300 import build
    dbg = ctypes.CDLL(build.build(debug=True))
    dbg.xattn_build_flags.restype = ctypes.c_int
    assert dbg.xattn_build_flags() == 1


def _fwd(lib, q=16, k=32, v=48, B=1, S=4, nh=2, nkv=1, hd=64, scale=0.125, o=64, lse=80):
    f = lib.xattn_fwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 3
    return f(q, k, v, B, S, nh, nkv, hd, scale, o, lse, None)


def test_fwd_argument_checks(lib):
    # None of these reach the device: each is rejected by the host checks first.
    assert _fwd(lib, q=None) == 1                      # NULL pointer
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, B=0) == 2                         # bad shape
    assert _fwd(lib, S=-1) == 2
    assert _fwd(lib, nh=3, nkv=2) == 3                 # nh % nkv != 0
    assert _fwd(lib, hd=48) == 4                       # unsupported head dim for bf16
    assert _fwd(lib, hd=256) == 4
    assert _fwd(lib, q=18) == 5                        # not 16-byte aligned
    assert _fwd(lib, scale=float("nan")) == 9
    assert _fwd(lib, scale=float("inf")) == 9


def _bwd(lib, scale):
    f = lib.xattn_bwd
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_float]
                  + [ctypes.c_void_p] * 4)
    return f(16, 32, 48, 64, 80, 96, 1, 4, 2, 1, 64, scale, 112, 128, 144, None)


def test_bwd_scale_checks(lib):
    # The bf16 backward adds -LSE/scale inside a tensor-core product: it takes scale == 0
    # exactly and rejects a nonzero |scale| below 2^-64 on the host.
    assert _bwd(lib, float("nan")) == 9
    assert _bwd(lib, 1e-30) == 9
    assert _bwd(lib, -1e-30) == 9
    import torch
    if not torch.cuda.is_available():
        assert _bwd(lib, 0.0) == 6                     # accepted; fails only for want of a GPU
        assert _bwd(lib, 2.0 ** -64) == 6


def test_head_dim_128(lib):
    """bf16 hd = 128 passes the host checks of the forward and of both backwards; the
    backward's stage calls and the no-allocation backward (fused dQ only) reject it."""
    import torch
    bwd_types = ([ctypes.c_void_p] * 5 + [ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_float]
                 + [ctypes.c_void_p] * 4)
    args = (16, 32, 48, 64, 80, 96, 1, 4, 2, 1, 128, 0.1, 112, 128, 144, None)
    for name in ("xattn_bwd", "xattn_bwd_deterministic", "xattn_bwd_noalloc"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = bwd_types
        if name == "xattn_bwd_noalloc":
            assert f(*args) == 4
        elif not torch.cuda.is_available():
            assert f(*args) == 6                       # accepted; fails only for want of a GPU
    if not torch.cuda.is_available():
        assert _fwd(lib, hd=128) == 6
    f = lib.xattn_bwd_main
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert f(16, 32, 48, 64, 1, 4, 2, 1, 128, 0.1, 80, 96, 256, 1 << 20, None) == 4


def test_f32_head_dim_limit(lib):
    f = lib.xattn_fwd_f32
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 3
    assert f(16, 32, 48, 1, 4, 2, 1, 129, 0.1, 64, 80, None) == 4


def test_workspace_checks(lib):
    lib.xattn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.xattn_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 4
    n = lib.xattn_bwd_workspace_bytes(2, 200, 4, 64)
    # Auxiliary rows padded to 256 (=2 tiles): 2*4*256 rows of 16 bf16; D: 2*200*4 fp32;
    # dQ accumulator: 2*200*4*64 fp32.
    assert n == 2 * 4 * 256 * 16 * 2 + 2 * 200 * 4 * 4 + 2 * 200 * 4 * 64 * 4
    assert lib.xattn_bwd_workspace_bytes(0, 200, 4, 64) == 0
    f = lib.xattn_bwd_dq_convert
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p]
    assert f(2, 200, 4, 64, 0.125, 256, None, n, None) == 10          # NULL workspace
    assert f(2, 200, 4, 64, 0.125, 256, 4096 + 16, n, None) == 10     # not 256-byte aligned
    assert f(2, 200, 4, 64, 0.125, 256, 4096, n - 1, None) == 10      # too small
    assert f(2, 200, 4, 64, float("nan"), 256, 4096, n, None) == 9    # non-finite scale


def test_no_device_is_a_cuda_error(lib):
    """With valid arguments and no usable GPU, the call fails with XATTN_ERR_CUDA
    (it never silently does nothing or falls back to the CPU)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib) == 6


def _decode(lib, q=16, k=32, v=48, B=2, T=5, nh=4, nkv=2, hd=64, scale=0.125, o=64, lse=80):
    f = lib.xattn_decode
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 3
    return f(q, k, v, B, T, nh, nkv, hd, scale, o, lse, None)


def test_decode_argument_checks(lib):
    assert _decode(lib, k=None) == 1                    # NULL pointer
    assert _decode(lib, lse=None) == 1
    assert _decode(lib, T=0) == 2                       # bad shape
    assert _decode(lib, B=-2) == 2
    assert _decode(lib, nh=6, nkv=4) == 3               # nh % nkv != 0
    assert _decode(lib, nh=34, nkv=2) == 3              # group above 16
    assert _decode(lib, hd=48) == 4                     # head dims 32, 64, 128 only
    assert _decode(lib, hd=256) == 4
    assert _decode(lib, v=56) == 5                      # not 16-byte aligned
    assert _decode(lib, lse=82) == 5                    # lse not 4-byte aligned
    assert _decode(lib, scale=float("nan")) == 9
    import torch
    if not torch.cuda.is_available():
        assert _decode(lib, hd=128, nh=32, nkv=2) == 6  # accepted; no GPU here


def test_selftest_limit_checks(lib):
    f = lib.xattn_selftest_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    assert f(0, None) == 2
    assert f(20 * 10**9, None) == 2


def test_decode_runs(lib):
    """How the decode splits the caches (a pure function of the sizes and the SM count)."""
    f = lib.xattn_decode_runs
    f.restype = ctypes.c_int
    # 64 sequences x 4 kv heads fill 152 SMs in one wave: one CTA per (sequence, kv head)
    assert f(64, 4096, 16, 4, 64, 152) == 1
    assert f(40, 1000, 16, 4, 128, 152) == 1
    # 32 pairs: as many runs as fill one wave, each run non-empty (12 chunks of 256 keys)
    assert f(8, 3000, 16, 4, 64, 152) == 12
    assert f(1, 1, 2, 1, 64, 152) == 1
    # more pairs than resident CTAs: a count between 1 and the chunk count
    r = f(128, 700, 32, 8, 64, 152)
    assert 1 <= r <= 3
    for bad in [(0, 10, 4, 2, 64, 152), (1, 10, 6, 4, 64, 152), (1, 10, 4, 2, 48, 152), (1, 10, 34, 2, 64, 152),
                (1, 10, 4, 2, 64, 0)]:
        assert f(*bad) == -1, bad


def test_bwd_dq_mode(lib):
    """The backward that xattn_bwd / xattn_bwd_deterministic pick, by sizes: xattn_bwd runs
    the fused-dQ backward at hd 32 and 64 and the query-stationary one at hd 128; the
    deterministic backward keeps dQ in tensor memory when a head's dQ tiles fit its 64
    free columns, else it runs the query-stationary dQ."""
    f = lib.xattn_bwd_dq_mode
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5
    assert f(256, 12, 12, 32, 0) == 0 and f(2048, 8, 2, 64, 0) == 0 and f(4096, 16, 4, 128, 0) == 2
    assert f(256, 12, 12, 32, 1) == 1         # one head, two query tiles at hd 32
    assert f(128, 4, 2, 32, 1) == 1           # group 2, one tile
    assert f(129, 4, 2, 32, 1) == 2           # group 2, two tiles: 128 columns
    assert f(128, 2, 2, 64, 1) == 1 and f(129, 2, 2, 64, 1) == 2
    assert f(2048, 8, 2, 64, 1) == 2 and f(4096, 16, 4, 128, 1) == 2
    assert f(256, 6, 4, 32, 0) == -1 and f(0, 2, 2, 32, 1) == -1 and f(256, 2, 2, 48, 0) == -1
