"""The forward and the backward's stage calls captured in a CUDA graph and replayed: the
replay gives the eager results (o, lse, dK, dV bit for bit; dQ within the bf16 bar, its
fp32 reduce-adds having no fixed order), and a replay after new inputs are written into
the captured buffers gives the eager results for those inputs. The same for xattn_bwd at
hd = 128 (its own stream-ordered scratch allocation inside the graph)."""
import numpy as np
import pytest
import torch

from bwd_xattn_fwd_gb300 import workloads as W
from gpu_path import TOL_BF16, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _step_stages(xattn, t, w, ws, stream):
    B, S, nh, nkv, hd, scale = w.B, w.S, w.nh, w.nkv, w.hd, w.scale
    xattn.xattn_fwd(t["q"], t["k"], t["v"], B, S, nh, nkv, hd, scale, t["o"], t["lse"], stream)
    xattn.xattn_bwd_preprocess(t["o"], t["dO"], t["lse"], B, S, nh, hd, scale, ws, ws.numel(), stream)
    xattn.xattn_bwd_main(t["q"], t["k"], t["v"], t["dO"], B, S, nh, nkv, hd, scale, t["dk"], t["dv"],
                         ws, ws.numel(), stream)
    xattn.xattn_bwd_dq_convert(B, S, nh, hd, scale, t["dq"], ws, ws.numel(), stream)


def _step_api(xattn, t, w, ws, stream):
    B, S, nh, nkv, hd, scale = w.B, w.S, w.nh, w.nkv, w.hd, w.scale
    xattn.xattn_fwd(t["q"], t["k"], t["v"], B, S, nh, nkv, hd, scale, t["o"], t["lse"], stream)
    xattn.xattn_bwd(t["q"], t["k"], t["v"], t["o"], t["dO"], t["lse"], B, S, nh, nkv, hd, scale,
                    t["dq"], t["dk"], t["dv"], stream)


def _buffers(w, x):
    t = {n: x[n].cuda() for n in ("q", "k", "v", "dO")}
    t["o"] = torch.empty_like(t["q"])
    t["lse"] = torch.empty((w.B, w.S, w.nh), dtype=torch.float32, device="cuda")
    t["dq"], t["dk"], t["dv"] = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    return t


OUTS = ("o", "lse", "dq", "dk", "dv")


def _snapshot(t):
    return {n: t[n].float().cpu().numpy() for n in OUTS}


def _same(a, b, exact_dq):
    for n in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[n], b[n]), n
    if exact_dq:
        assert np.array_equal(a["dq"], b["dq"])
    else:
        assert rel_err(a["dq"], b["dq"]) <= TOL_BF16


@pytest.mark.parametrize("hd,step", [(64, "stages"), (32, "stages"), (128, "api")])
def test_graph_replay_matches_eager(hd, step):
    from bwd_xattn_fwd_gb300 import xattn
    w = W.Workload("graph", 2, 700, 8, 2, hd, "bf16", qkv_scale=0.5)
    x1, x2 = W.make_inputs(w, seed=41), W.make_inputs(w, seed=42)
    t = _buffers(w, x1)
    ws = None                               # xattn_bwd takes its own scratch
    if step == "stages":
        ws = torch.empty(xattn.xattn_bwd_workspace_bytes(w.B, w.S, w.nh, hd), dtype=torch.uint8, device="cuda")
    run = _step_stages if step == "stages" else _step_api
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):                  # eager warm-up: one-time set-up outside the capture
            run(xattn, t, w, ws, s)
    s.synchronize()
    eager1 = _snapshot(t)
    for n in ("q", "k", "v", "dO"):
        t[n].copy_(x2[n].cuda())
    with torch.cuda.stream(s):
        run(xattn, t, w, ws, s)
    s.synchronize()
    eager2 = _snapshot(t)

    for n in ("q", "k", "v", "dO"):
        t[n].copy_(x1[n].cuda())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(xattn, t, w, ws, s)
    for n in OUTS:
        t[n].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0
    _same(_snapshot(t), eager1, exact_dq=(hd == 128))
    for n in ("q", "k", "v", "dO"):
        t[n].copy_(x2[n].cuda())
    g.replay()
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0
    _same(_snapshot(t), eager2, exact_dq=(hd == 128))
