"""bf16 forward and backward at head dim 128 against the oracle. Each tile is two
64-column swizzled sub-tiles; the forward keeps one Q buffer and two K/V stages and
writes P over its own scores in TMEM; the backward runs the key-stationary dK / dV
kernel (P^T over S^T, dS^T over dP^T) and the query-stationary dQ kernel. Shapes cover
S = 1, partial tiles, one-tile and many-tile sequences with and without a second query
tile per unit, and groups 1 to 8; scales zero, negative and large."""
import numpy as np
import pytest
import torch

import oracle
from bwd_xattn_fwd_gb300 import workloads as W
from gpu_path import (TOL_BF16, TOL_LSE, compare, compare_every_unit, oracle_full, rel_err,
                      run_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _fwd(w, x, scale):
    from bwd_xattn_fwd_gb300 import xattn
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = xattn.attention_fwd(q, k, v, scale)
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0
    return W.as_f64(o), W.as_f64(lse)


def _check(w, x, scale, label):
    o, lse = _fwd(w, x, scale)
    ro, rlse = oracle.default().fwd(*(W.as_f64(x[n]) for n in ("q", "k", "v")), scale)
    eo, el = rel_err(o, ro), float(np.abs(lse - rlse).max())
    assert eo <= TOL_BF16 and el <= TOL_LSE, f"{label}: o {eo:.3e} lse {el:.3e}"


SHAPES = [
    # (B, S, nh, nkv): S = 1; partial tile; exactly one tile; a unit without tile B;
    # two units per head; many tiles with group 8
    (1, 1, 2, 1),
    (2, 77, 4, 2),
    (1, 128, 2, 2),
    (1, 300, 4, 1),
    (2, 513, 6, 3),
    (1, 1024, 4, 4),
    (1, 2048, 8, 1),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_S%d_nh%d_nkv%d" % s)
def test_fwd_hd128_shapes(shape):
    B, S, nh, nkv = shape
    w = W.Workload("hd128", B, S, nh, nkv, 128, "bf16", qkv_scale=0.5)
    _check(w, W.make_inputs(w, seed=11), w.scale, str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.3, 0.5], ids=lambda s: "scale=%g" % s)
def test_fwd_hd128_scales(scale):
    w = W.Workload("hd128", 2, 300, 4, 2, 128, "bf16", qkv_scale=0.5)
    _check(w, W.make_inputs(w, seed=13), scale, "scale=%g" % scale)


def test_fwd_hd128_matches_fp32_path_rows():
    """The bf16 forward and the fp32 CUDA-core forward on the same (bf16-exact) inputs
    agree within the bf16 output rounding."""
    from bwd_xattn_fwd_gb300 import xattn
    w = W.Workload("hd128", 1, 640, 4, 2, 128, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=17)
    o, lse = _fwd(w, x, w.scale)
    q, k, v = (x[n].cuda().float() for n in ("q", "k", "v"))
    o32, lse32 = xattn.attention_fwd(q, k, v, w.scale)
    torch.cuda.synchronize()
    assert rel_err(o, W.as_f64(o32)) <= TOL_BF16
    assert float(np.abs(lse - W.as_f64(lse32)).max()) <= TOL_LSE


# ---- backward at hd = 128: the key-stationary dK / dV kernel with P^T over S^T and
# dS^T over dP^T in TMEM, and the query-stationary dQ kernel; xattn_bwd takes that path
# (every output reproducible) ----
BWD_SHAPES = [(1, 1, 2, 1), (2, 77, 4, 2), (1, 300, 4, 1), (2, 513, 6, 3), (1, 1024, 4, 4)]


@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "B%d_S%d_nh%d_nkv%d" % s)
def test_bwd_hd128_shapes(shape):
    B, S, nh, nkv = shape
    w = W.Workload("hd128", B, S, nh, nkv, 128, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=19)
    compare(run_gpu(w, x), oracle_full(w, x), "bf16", str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.3], ids=lambda s: "scale=%g" % s)
def test_bwd_hd128_scales(scale):
    w = W.Workload("hd128", 2, 300, 4, 2, 128, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=23)
    compare(run_gpu(w, x, scale=scale), oracle_full(w, x, scale=scale), "bf16", "scale=%g" % scale)


def test_bwd_hd128_long_every_unit():
    """A long-sequence GQA problem at hd = 128 (4 x 4096, 16 query heads on 4 kv heads),
    compared element by element with the oracle on all 16 (batch, kv head) units."""
    w = W.Workload("hd128_long", 4, 4096, 16, 4, 128, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=29)
    out = run_gpu(w, x)
    ref = oracle_full(w, x)
    compare(out, ref, "bf16", "hd128_long")
    print(compare_every_unit(w, out, ref, "hd128_long"))


def test_bwd_hd128_reproducible_and_same_as_deterministic():
    w = W.Workload("hd128", 2, 700, 8, 2, 128, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=31)
    a = run_gpu(w, x)
    b = run_gpu(w, x)
    c = run_gpu(w, x, deterministic=True)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[n], b[n]) and np.array_equal(a[n], c[n]), n
