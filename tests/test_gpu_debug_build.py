"""The debug build of libxattn (XATTN_DEBUG: on-device bounds checks in the tensor-core
kernels -- TMA tile coordinates, shared-memory and tensor-memory offsets, global row
offsets of direct stores -- that record XATTN_ERR_DEVICE_BOUNDS instead of trapping) on
the GPU, in a child process that loads it in place of the release library:
  * its self-test's failing check is reported, once, and cleared by the read;
  * the attention path on edge shapes -- the fused-dQ backward with query groups and with
    one head per kv head, the deterministic backward (query-stationary and resident dQ),
    hd 32, 64 and 128, ragged last tiles, several units per CTA -- and the decode kernels
    (ragged last chunks, padded groups, hd 32, 64 and 128) pass every check (the status
    word stays clear) and match the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, "tests")
sys.path.insert(0, ".")
from bwd_xattn_fwd_gb300 import workloads as W, xattn
from gpu_path import compare, oracle_full, run_gpu

assert xattn.xattn_build_flags() & xattn.BUILD_DEVICE_CHECKS
assert xattn.xattn_check_device_status() == 0
xattn.xattn_selftest_bounds_check()
assert xattn.xattn_check_device_status() == xattn.ERR_DEVICE_BOUNDS
assert xattn.xattn_check_device_status() == 0
CASES = [
    ((2, 77, 4, 2, 64), False),     # one partial tile, query groups
    ((48, 300, 8, 2, 64), False),   # several units per CTA, ragged, query groups
    ((48, 200, 6, 3, 32), False),   # the same at hd 32
    ((40, 300, 4, 4, 64), False),   # one query head per kv head
    ((2, 300, 4, 2, 64), True),     # deterministic: query-stationary dQ
    ((3, 200, 4, 4, 32), True),     # deterministic: dQ resident in tensor memory
    ((1, 300, 4, 2, 128), False),   # hd 128 (deterministic backward)
]
for shape, det in CASES:
    B, S, nh, nkv, hd = shape
    w = W.Workload("debug", B, S, nh, nkv, hd, "bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=5)
    out = run_gpu(w, x, deterministic=det)   # asserts that the status word is clear
    compare(out, oracle_full(w, x), "bf16", str(shape))
# decode: ragged last chunks with tiles wholly past T, padded groups, hd 32 / 64 / 128
import numpy as np
import oracle
import torch
from gpu_path import TOL_BF16, TOL_LSE, rel_err
for B, T, nh, nkv, hd in [(3, 777, 8, 2, 64), (2, 2049, 8, 1, 32), (2, 300, 16, 4, 128)]:
    w = W.DecodeWorkload("debug", B=B, T=T, nh=nh, nkv=nkv, hd=hd)
    x = W.make_decode_inputs(w, seed=7)
    o, lse = xattn.attention_decode(*(x[n].cuda() for n in ("q", "k", "v")), w.scale)
    torch.cuda.synchronize()
    assert xattn.xattn_check_device_status() == 0, (B, T, nh, nkv, hd)
    ro, rl = oracle.default().decode(*(W.as_f64(x[n]) for n in ("q", "k", "v")), w.scale)
    assert rel_err(W.as_f64(o), ro) <= TOL_BF16 and float(np.abs(W.as_f64(lse) - rl).max()) <= TOL_LSE
print("debug build ok")
"""


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def test_debug_build_checks_pass_and_report():
    from bwd_xattn_fwd_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, XATTN_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout
