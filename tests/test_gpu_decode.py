"""Decode attention (one new query per sequence against its cached K/V) through the C
ABI against the oracle's decode, element by element, on edge shapes and on the full
decode workload; and against the last row of the library's own causal forward.
Tolerances as for the bf16 path: max|err|/max|ref| <= 2e-2 for O, LSE absolute <= 1e-3."""
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
    from bwd_xattn_fwd_gb300 import xattn  # noqa: F401  (fails loudly if not built)


def _run(x, scale, device="cuda"):
    from bwd_xattn_fwd_gb300 import xattn
    q, k, v = (x[n].to(device) for n in ("q", "k", "v"))
    o, lse = xattn.attention_decode(q, k, v, scale)
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0
    return W.as_f64(o), W.as_f64(lse)


def _check(x, scale, label, sel=slice(None)):
    o, lse = _run(x, scale)
    q, k, v = (W.as_f64(x[n][sel]) for n in ("q", "k", "v"))
    ro, rlse = oracle.default().decode(q, k, v, scale)
    eo, el = rel_err(o[sel], ro), float(np.abs(lse[sel] - rlse).max())
    assert eo <= TOL_BF16 and el <= TOL_LSE, f"{label}: o {eo:.3e} lse {el:.3e}"
    return eo, el


SHAPES = [
    # (B, T, nh, nkv, hd): one key; chunk and tile edges (chunks of 512, 256, 128 keys at
    # hd 32, 64, 128; last chunks with tiles wholly past T); long caches; groups 1..16
    # (each padded width of the query tile at each head dim); head dims 32, 64, 128
    (1, 1, 2, 1, 64),
    (3, 255, 8, 2, 64),
    (2, 256, 4, 4, 32),
    (2, 257, 16, 1, 128),
    (1, 1000, 12, 12, 64),
    (2, 777, 32, 2, 64),
    (4, 2049, 8, 1, 32),
    (1, 5000, 4, 2, 128),
    (2, 600, 16, 1, 32),
    (2, 1300, 16, 2, 64),
    # one CTA per (sequence, kv head) streaming a ragged cache (no combine), at each head
    # dim; and more (sequence, kv head) pairs than resident CTAs (several waves of runs)
    (40, 1000, 16, 4, 64),
    (40, 1000, 16, 4, 128),
    (40, 1500, 8, 4, 32),
    (128, 700, 32, 8, 64),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_T%d_nh%d_nkv%d_hd%d" % s)
def test_decode_edge_shapes(shape):
    B, T, nh, nkv, hd = shape
    w = W.DecodeWorkload("edge", B=B, T=T, nh=nh, nkv=nkv, hd=hd)
    _check(W.make_decode_inputs(w, seed=3), w.scale, str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.4, 2.0], ids=lambda s: f"scale={s}")
def test_decode_scales(scale):
    w = W.DecodeWorkload("edge", B=2, T=300, nh=8, nkv=2, hd=64, qkv_scale=1.0)
    _check(W.make_decode_inputs(w, seed=4), scale, f"scale {scale}")


def test_decode_workload():
    """The full decode workload (64 sequences x 4096 cached positions), every sequence; on
    a GB300 (152 SMs) it runs as one CTA per (sequence, kv head)."""
    from bwd_xattn_fwd_gb300 import xattn
    w = W.DECODE_WORKLOADS["decode"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms >= 128:
        assert xattn.xattn_decode_runs(w.B, w.T, w.nh, w.nkv, w.hd, sms) == 1
    eo, el = _check(W.make_decode_inputs(w), w.scale, "decode workload")
    print("decode workload: o", eo, "lse", el)


def test_decode_is_last_row_of_forward():
    """Decode equals the last row of the library's own causal forward when the query is
    placed at position T-1 (the pages' gate for decode attention)."""
    from bwd_xattn_fwd_gb300 import xattn
    w = W.Workload("rows", B=2, S=333, nh=8, nkv=2, hd=64, dtype="bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o_full, lse_full = xattn.attention_fwd(q, k, v, w.scale)
    o_dec, lse_dec = xattn.attention_decode(q[:, -1].contiguous(), k, v, w.scale)
    torch.cuda.synchronize()
    of, od = W.as_f64(o_full[:, -1]), W.as_f64(o_dec)
    assert rel_err(od, of) <= TOL_BF16
    assert float(np.abs(W.as_f64(lse_dec) - W.as_f64(lse_full[:, -1])).max()) <= TOL_LSE


def test_decode_is_bit_reproducible():
    w = W.DecodeWorkload("rep", B=8, T=3000, nh=16, nkv=4, hd=64)
    x = W.make_decode_inputs(w, seed=6)
    a, b = _run(x, w.scale), _run(x, w.scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
