"""bf16 forward at head dim 128 against the oracle: each tile is two 64-column swizzled
sub-tiles, one Q buffer and two K/V stages, and P written over its own scores in TMEM.
Shapes cover S = 1, partial tiles, one-tile and many-tile sequences with and without a
second query tile per unit, and groups 1 to 8; scales zero, negative and large."""
import numpy as np
import pytest
import torch

import oracle
from bwd_xattn_fwd_gb300 import workloads as W
from gpu_path import TOL_BF16, TOL_LSE, rel_err

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
