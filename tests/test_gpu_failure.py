"""Failure detection on the GPU without a fault: a bounded wait that nothing completes
runs out, the library reports XATTN_ERR_DEVICE_TIMEOUT through
xattn_check_device_status, clears it, and the context keeps computing correct results."""
import numpy as np
import pytest
import torch

from bwd_xattn_fwd_gb300 import workloads as W
from gpu_path import compare, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def test_expired_wait_is_reported_and_the_context_survives():
    from bwd_xattn_fwd_gb300 import xattn
    assert xattn.xattn_check_device_status() == 0
    xattn.xattn_selftest_wait_timeout(10_000_000)        # 10 ms
    assert xattn.xattn_check_device_status() == int(xattn.Status.ERR_DEVICE_TIMEOUT)
    assert xattn.xattn_check_device_status() == 0          # the word was cleared
    w = W.Workload("after", B=1, S=200, nh=4, nkv=2, hd=64, dtype="bf16", qkv_scale=0.5)
    x = W.make_inputs(w, seed=7)
    compare(run_gpu(w, x), oracle_full(w, x), "bf16", "after the expired wait")
