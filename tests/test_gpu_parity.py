"""Parity of the CUDA path (through the C ABI) with the oracle, on the seeded workloads
and on edge shapes. Tolerances: bf16 max|err|/max|ref| <= 2e-2, fp32 <= 1e-4 (O, dQ,
dK, dV), LSE absolute <= 1e-3."""
import numpy as np
import pytest
import torch

from bwd_xattn_fwd_gb300 import workloads as W
from gpu_path import (TOL_BF16, compare, compare_every_unit, oracle_full, run_gpu, tol_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bwd_xattn_fwd_gb300 import xattn  # noqa: F401  (fails loudly if not built)


# Oracle outputs of the seeded full-size workloads (seed 0), computed once per session:
# the default and the deterministic backward are both compared with them.
_ORACLE_CACHE = {}


def _workload_oracle(name):
    if name not in _ORACLE_CACHE:
        w = W.WORKLOADS[name]
        x = W.make_inputs(w)
        _ORACLE_CACHE[name] = (x, oracle_full(w, x))
    return _ORACLE_CACHE[name]


@pytest.mark.parametrize("name", ["tiny", "dim384"])
def test_workload_full(name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w)
    out = run_gpu(w, x)
    ref = oracle_full(w, x)
    print(name, compare(out, ref, w.dtype, name))


@pytest.mark.parametrize("name", ["dim768", "gqa", "long"])
def test_workload_every_unit(name):
    """The full-size workloads, in the launch configuration the benchmark times, compared
    element by element with the oracle on every (batch, kv head) unit: 384 units of
    dim768, 16 of gqa and 16 of long."""
    w = W.WORKLOADS[name]
    x, ref = _workload_oracle(name)
    out = run_gpu(w, x)
    compare(out, ref, w.dtype, name)
    print(name, compare_every_unit(w, out, ref, name))


EDGE = [
    # (B, S, nh, nkv, hd) -- partial tiles, S = 1, one tile, group > 1, hd 32 and 64
    (1, 1, 2, 1, 64),
    (2, 77, 4, 2, 64),
    (1, 128, 2, 2, 32),
    (1, 129, 3, 1, 64),
    (2, 200, 6, 3, 32),
    (1, 300, 4, 1, 64),
    (1, 513, 2, 2, 64),
    # several units per CTA with a ragged last tile: query groups (dK from dS^T in TMEM,
    # dQ staged in the dS tiles across unit boundaries) and one query head per kv head,
    # at hd 64 and 32
    (48, 300, 8, 2, 64),
    (48, 200, 6, 3, 32),
    (40, 300, 4, 4, 64),
]


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "B%d_S%d_nh%d_nkv%d_hd%d" % s)
def test_edge_shapes_bf16(shape):
    B, S, nh, nkv, hd = shape
    w = W.Workload("edge", B, S, nh, nkv, hd, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=3)
    compare(run_gpu(w, x), oracle_full(w, x), "bf16", str(shape))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("scale", [0.0, 1.0, -0.3, 2.0 ** -40], ids=lambda s: "scale=%g" % s)
def test_scale_values(scale, dtype):
    """Scales other than 1/sqrt(hd): zero (uniform attention over the causal prefix; dQ
    and dK vanish), large, negative (the row maximum of the scaled scores is the scaled
    minimum of the raw ones) and tiny. The bf16 backward adds -LSE/scale to the scores
    inside a tensor-core product, with scale == 0 taken as its own case."""
    w = W.Workload("scale", 2, 200, 4, 2, 64 if dtype == "bf16" else 32, dtype, qkv_scale=0.5)
    x = W.make_inputs(w, seed=7)
    compare(run_gpu(w, x, scale=scale), oracle_full(w, x, scale=scale), dtype, "scale=%g" % scale)


EDGE_F32 = [(1, 1, 1, 1, 8), (2, 37, 6, 3, 24), (1, 150, 4, 2, 128), (1, 64, 2, 1, 1)]


@pytest.mark.parametrize("shape", EDGE_F32, ids=lambda s: "B%d_S%d_nh%d_nkv%d_hd%d" % s)
def test_edge_shapes_f32(shape):
    B, S, nh, nkv, hd = shape
    w = W.Workload("edge32", B, S, nh, nkv, hd, "f32")
    x = W.make_inputs(w, seed=4)
    compare(run_gpu(w, x), oracle_full(w, x), "f32", str(shape))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_equals_repeated_mha(dtype):
    """GQA on (K, V) equals MHA on K/V repeated per group, with dK/dV summed per group
    (the broadcast and its backward of xtrain docs/evolution.md, row T15). The forward
    is bit-identical: each query head reads the same K/V values either way."""
    w = W.Workload("g", 2, 256, 8, 2, 64 if dtype == "bf16" else 32, dtype, qkv_scale=0.5)
    x = W.make_inputs(w, seed=5)
    g = w.group
    xr = dict(x)
    xr["k"] = x["k"].repeat_interleave(g, dim=2).contiguous()
    xr["v"] = x["v"].repeat_interleave(g, dim=2).contiguous()
    wr = w.with_(nkv=w.nh)
    a = run_gpu(w, x)
    r = run_gpu(wr, xr)
    assert np.array_equal(a["o"], r["o"]) and np.array_equal(a["lse"], r["lse"])
    tol = tol_for(dtype)
    for name in ("dk", "dv"):
        summed = r[name].reshape(w.B, w.S, w.nkv, g, w.hd).sum(axis=3)
        e = np.abs(a[name] - summed).max() / np.abs(summed).max()
        assert e <= tol, (name, e)
    e = np.abs(a["dq"] - r["dq"]).max() / np.abs(r["dq"]).max()
    assert e <= tol, ("dq", e)


def test_reproducible():
    """O, LSE, dK and dV are bit-identical run to run; dQ (fp32 reduce-adds across key
    tiles, in no fixed order) agrees within the bf16 tolerance."""
    w = W.WORKLOADS["gqa"].with_(B=2)
    x = W.make_inputs(w, seed=6)
    a, b = run_gpu(w, x), run_gpu(w, x)
    for name in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[name], b[name]), name
    assert np.abs(a["dq"] - b["dq"]).max() <= TOL_BF16 * np.abs(a["dq"]).max()


DET_EDGE = [(1, 1, 2, 1, 64), (2, 77, 4, 2, 64), (2, 200, 6, 3, 32), (1, 513, 2, 2, 64)]


@pytest.mark.parametrize("shape", DET_EDGE, ids=lambda s: "B%d_S%d_nh%d_nkv%d_hd%d" % s)
def test_deterministic_edge_shapes(shape):
    """The deterministic backward (query-stationary dQ recompute) against the oracle."""
    B, S, nh, nkv, hd = shape
    w = W.Workload("det", B, S, nh, nkv, hd, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=8)
    compare(run_gpu(w, x, deterministic=True), oracle_full(w, x), "bf16", "det " + str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.3], ids=lambda s: "scale=%g" % s)
def test_deterministic_scales(scale):
    w = W.Workload("det", 2, 200, 4, 2, 64, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=7)
    compare(run_gpu(w, x, scale=scale, deterministic=True), oracle_full(w, x, scale=scale), "bf16",
            "det scale=%g" % scale)


@pytest.mark.parametrize("name", ["gqa", "dim768"])
def test_deterministic_workload_every_unit(name):
    w = W.WORKLOADS[name]
    x, ref = _workload_oracle(name)
    out = run_gpu(w, x, deterministic=True)
    compare(out, ref, "bf16", "det " + name)
    print(name, compare_every_unit(w, out, ref, "det " + name))


def test_deterministic_is_bit_reproducible():
    """Every output of the deterministic backward is bit-identical run to run, and its dK
    and dV equal the default backward's (the same key-stationary recompute)."""
    w = W.WORKLOADS["gqa"].with_(B=2)
    x = W.make_inputs(w, seed=6)
    a, b = run_gpu(w, x, deterministic=True), run_gpu(w, x, deterministic=True)
    for name in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[name], b[name]), name
    c = run_gpu(w, x)
    for name in ("dk", "dv"):
        assert np.array_equal(a[name], c[name]), name
    assert np.abs(a["dq"] - c["dq"]).max() <= TOL_BF16 * np.abs(c["dq"]).max()


def test_stage_calls_match_bwd():
    """xattn_bwd equals its three steps run with a caller-owned workspace."""
    from bwd_xattn_fwd_gb300 import xattn
    w = W.Workload("s", 2, 384, 4, 2, 64, "bf16", qkv_scale=0.5)
    x = {n: t.cuda() for n, t in W.make_inputs(w, seed=7).items()}
    o, lse = xattn.attention_fwd(x["q"], x["k"], x["v"], w.scale)
    dq, dk, dv = xattn.attention_bwd(x["q"], x["k"], x["v"], o, x["dO"], lse, w.scale)
    nbytes = xattn.xattn_bwd_workspace_bytes(w.B, w.S, w.nh, w.hd)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    xattn.xattn_bwd_preprocess(o, x["dO"], lse, w.B, w.S, w.nh, w.hd, w.scale, ws, nbytes)
    xattn.xattn_bwd_main(x["q"], x["k"], x["v"], x["dO"], w.B, w.S, w.nh, w.nkv, w.hd, w.scale,
                         dk2, dv2, ws, nbytes)
    xattn.xattn_bwd_dq_convert(w.B, w.S, w.nh, w.hd, w.scale, dq2, ws, nbytes)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.float() - dq2.float()).abs().max() <= TOL_BF16 * dq.float().abs().max()
    assert xattn.xattn_check_device_status() == 0


def test_right_padded_ragged_batch():
    """Ragged sequences right-padded to one length (xtrain "演进总览", milestone M2d: under
    causal masking the real rows never see the padding, so a padded batch needs no
    per-sequence lengths). The pad rows' inputs are garbage and their output gradient is
    zero (the loss masks them); every real row of O, LSE, dQ and every real key's dK, dV
    must then match the oracle run on that sequence alone."""
    lengths, S = [300, 129, 57], 300
    w = W.Workload("pad", len(lengths), S, 8, 2, 64, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=11)
    g = torch.Generator().manual_seed(12)
    for b, L in enumerate(lengths):
        for n in ("q", "k", "v"):
            junk = torch.randn(x[n][b, L:].shape, generator=g) * 3.0
            x[n][b, L:] = junk.to(x[n].dtype)
        x["dO"][b, L:] = 0
    out = run_gpu(w, x)
    for b, L in enumerate(lengths):
        wb = w.with_(B=1, S=L)
        xb = {n: x[n][b:b + 1, :L].contiguous() for n in x}
        ref = oracle_full(wb, xb)
        got = {n: out[n][b:b + 1, :L] for n in out}
        compare(got, ref, "bf16", f"sequence {b} (length {L})")


# ---- small problems: the deterministic backward with dQ resident in TMEM (one CTA per
# (batch, kv head) over all its key tiles; taken when group * ceil(S / 128) * hd <= 64) ----
RESIDENT = [
    # (B, S, nh, nkv, hd): S = 1; one tile at hd 64; two query tiles at hd 32; a query
    # group of 2 in one tile; partial second tile; more heads than SMs (a CTA takes two)
    (1, 1, 2, 2, 64),
    (2, 77, 6, 6, 64),
    (3, 200, 4, 4, 32),
    (2, 100, 4, 2, 32),
    (1, 130, 2, 2, 32),
    (160, 100, 2, 1, 32),
]


@pytest.mark.parametrize("shape", RESIDENT, ids=lambda s: "B%d_S%d_nh%d_nkv%d_hd%d" % s)
def test_resident_dq_shapes(shape):
    from bwd_xattn_fwd_gb300 import xattn
    B, S, nh, nkv, hd = shape
    assert xattn.xattn_bwd_dq_mode(S, nh, nkv, hd, True) == xattn.BWD_RESIDENT_DQ
    w = W.Workload("res", B, S, nh, nkv, hd, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=21)
    compare(run_gpu(w, x, deterministic=True), oracle_full(w, x), "bf16", "resident " + str(shape))


@pytest.mark.parametrize("scale", [0.0, -0.3], ids=lambda s: "scale=%g" % s)
def test_resident_dq_scales(scale):
    w = W.Workload("res", 2, 256, 4, 4, 32, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=22)
    compare(run_gpu(w, x, scale=scale, deterministic=True), oracle_full(w, x, scale=scale), "bf16",
            "resident scale=%g" % scale)


def test_resident_dq_workload_and_reproducible():
    """The dim384 workload (16 x 256 x 12 heads, hd 32) through the deterministic backward,
    which keeps dQ resident in TMEM there: every (batch, head) unit against the oracle,
    every output bit-identical run to run, and dK, dV bit-identical to the default
    backward's (the same key-stationary products in the same order)."""
    w = W.WORKLOADS["dim384"]
    x = W.make_inputs(w)
    a, b = run_gpu(w, x, deterministic=True), run_gpu(w, x, deterministic=True)
    ref = oracle_full(w, x)
    compare(a, ref, "bf16", "dim384 resident")
    compare_every_unit(w, a, ref, "dim384 resident")
    for name in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[name], b[name]), name
    c = run_gpu(w, x)
    for name in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[name], c[name]), name
    assert np.abs(a["dq"] - c["dq"]).max() <= TOL_BF16 * np.abs(c["dq"]).max()
