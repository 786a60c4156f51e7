"""Helpers shared by the GPU tests: run the libxattn path on seeded inputs and compare
its outputs with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bwd_xattn_fwd_gb300 import workloads as W

# Parity bar: per output tensor, max|gpu - ref| / max|ref| (LSE: absolute, natural log).
TOL_BF16 = 2e-2
TOL_F32 = 1e-4
TOL_LSE = 1e-3


def tol_for(dtype: str) -> float:
    return TOL_BF16 if dtype == "bf16" else TOL_F32


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    # The floor only matters where the exact result is (near) zero everywhere, e.g. dQ
    # and dK at S = 1; there the bar becomes an absolute 1e-4 * tol.
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-4))


def run_gpu(w: W.Workload, x: dict, device="cuda", scale=None, deterministic=False):
    """Forward then backward through the C ABI (with the workload's scale unless one is
    given; the deterministic backward on request). Returns float64 numpy outputs."""
    from bwd_xattn_fwd_gb300 import xattn
    scale = w.scale if scale is None else scale
    q, k, v, dO = (x[n].to(device) for n in ("q", "k", "v", "dO"))
    o, lse = xattn.attention_fwd(q, k, v, scale)
    dq, dk, dv = xattn.attention_bwd(q, k, v, o, dO, lse, scale, deterministic=deterministic)
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0
    return {n: W.as_f64(t) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def oracle_full(w: W.Workload, x: dict, scale=None):
    scale = w.scale if scale is None else scale
    q, k, v, dO = (W.as_f64(x[n]) for n in ("q", "k", "v", "dO"))
    orc = oracle.default()
    o, lse = orc.fwd(q, k, v, scale)
    dq, dk, dv = orc.bwd(q, k, v, dO, scale)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def gpu_unit(w: W.Workload, out: dict, b: int, kvh: int):
    g = w.group
    hs = slice(kvh * g, (kvh + 1) * g)
    return {"o": out["o"][b:b + 1, :, hs], "lse": out["lse"][b:b + 1, :, hs],
            "dq": out["dq"][b:b + 1, :, hs], "dk": out["dk"][b:b + 1, :, kvh:kvh + 1],
            "dv": out["dv"][b:b + 1, :, kvh:kvh + 1]}


def compare(got: dict, ref: dict, dtype: str, where: str = ""):
    tol = tol_for(dtype)
    report = {}
    for name in ("o", "dq", "dk", "dv"):
        assert np.all(np.isfinite(got[name])), f"{where} {name}: non-finite values"
        e = rel_err(got[name], ref[name])
        report[name] = e
        assert e <= tol, f"{where} {name}: max|err|/max|ref| = {e:.3e} > {tol}"
    e = float(np.abs(got["lse"] - ref["lse"]).max())
    report["lse"] = e
    assert e <= TOL_LSE, f"{where} lse: max|err| = {e:.3e} > {TOL_LSE}"
    return report


def compare_every_unit(w: W.Workload, got: dict, ref: dict, where: str = ""):
    """Element-by-element parity on every (batch, kv head) unit of a whole-batch run.

    Each unit is a complete attention problem of its own (B=1, nkv=1, nh=group), so its
    outputs are held to the bar with its own max|ref|, which is at least as strict as
    normalising by the whole tensor's. `ref` is one oracle run over the whole batch (the
    oracle computes every row from the definition; no unit depends on another).
    Returns the worst error per output over all units."""
    worst = {}
    for b in range(w.B):
        for kvh in range(w.nkv):
            rep = compare(gpu_unit(w, got, b, kvh), gpu_unit(w, ref, b, kvh), w.dtype,
                          f"{where} unit (b={b}, kvh={kvh})")
            for k_, e in rep.items():
                worst[k_] = max(worst.get(k_, 0.0), e)
    return worst
