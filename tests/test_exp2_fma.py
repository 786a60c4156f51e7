"""The forward's FMA-pipe exponential (exp2_fma2 in attn_fwd_sm103.cu): x = rint(x) + f,
2^f from a cubic on [-1/2, 1/2], rint(x) added into the exponent field. Its coefficients
are read from the kernel source and the same steps are replayed in float32 here; the
relative error against 2^x must stay below 1e-4 over the exponents the softmax produces
(scores minus a running maximum that may be stale by up to 2^8)."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "bwd_xattn_fwd_gb300", "csrc", "attn_fwd_sm103.cu")


def _coefficients():
    text = open(SRC).read()
    body = text[text.index("void exp2_fma2("):]
    body = body[:body.index("\n}\n")]
    c = {k: np.float32(v) for k, v in re.findall(r"\b(c[0-3]) = ([0-9.eE+-]+)f", body)}
    assert sorted(c) == ["c0", "c1", "c2", "c3"]
    return c


def _exp2_fma(x):
    c = _coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    k = np.float32(12582912.0)
    j = (x + k).astype(np.float32)
    t = (j - k).astype(np.float32)
    f = (x - t).astype(np.float32)
    p = (f.astype(np.float64) * c["c3"] + c["c2"]).astype(np.float32)
    p = (p.astype(np.float64) * f + c["c1"]).astype(np.float32)
    p = (p.astype(np.float64) * f + c["c0"]).astype(np.float32)
    bits = p.view(np.int32) + (j.view(np.int32) << 23)
    return bits.view(np.float32)


def test_relative_error_over_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001), np.arange(-125, 9, dtype=np.float64)])
    got = _exp2_fma(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float32).astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 1e-4


def test_far_below_the_maximum_is_negligible():
    got = _exp2_fma(np.array([-126.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(got >= 0) and np.all(got < 2.0 ** -125)
