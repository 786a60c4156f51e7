"""Pins of the oracle to facts outside itself.

Each ``pin_*`` takes an oracle handle (``oracle.OracleLib``) and raises
AssertionError when the oracle disagrees with a fact fixed by the mathematics or by
a hand-worked example. They are collected as tests in ``test_oracle_pins.py`` and
reused by ``test_oracle_mutations.py``, which shows that each planted mistake in the
oracle fails at least one pin.

The function being pinned is causal softmax attention with grouped KV heads and its
gradient (xtrain "演进总览" / docs/evolution.md, phase table rows T14 and T15), and the
decode form of the same attention: one new query per sequence against its cached keys
and values (same page, post-training milestones M2a-M2c).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.composed as composed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _problem(B=2, S=7, nh=4, nkv=2, hd=3, seed=1):
    rng = np.random.default_rng(seed)
    q = _rand((B, S, nh, hd), rng)
    k = _rand((B, S, nkv, hd), rng)
    v = _rand((B, S, nkv, hd), rng)
    dO = _rand((B, S, nh, hd), rng)
    return q, k, v, dO


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def pin_golden_two_positions(orc):
    """Hand-worked S=2 example (tests/golden/two_position_example.json)."""
    with open(os.path.join(GOLDEN, "two_position_example.json")) as f:
        g = json.load(f)
    shp = (1, 2, 1, 1)
    q, k, v, dO = (np.array(g[n], dtype=np.float64).reshape(shp) for n in ("q", "k", "v", "dO"))
    o, lse = orc.fwd(q, k, v, g["scale"])
    dq, dk, dv = orc.bwd(q, k, v, dO, g["scale"])
    for name, got in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        want = np.array(g[name]).reshape(got.shape)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (name, got.ravel(), want.ravel())


def pin_zero_queries(orc):
    """Q = 0: every visible score is 0, so O_i is the prefix mean of V and LSE_i = ln(i+1)."""
    q, k, v, _ = _problem(B=2, S=9, nh=4, nkv=2, hd=3, seed=2)
    q[:] = 0.0
    o, lse = orc.fwd(q, k, v, 0.7)
    S = q.shape[1]
    counts = np.arange(1, S + 1, dtype=np.float64)
    prefix_mean = np.cumsum(v, axis=1) / counts[None, :, None, None]      # [B,S,nkv,hd]
    want = np.repeat(prefix_mean, 2, axis=2)                               # group 2, contiguous
    assert _rel(o, want) < 1e-13, _rel(o, want)
    want_lse = np.broadcast_to(np.log(counts)[None, :, None], lse.shape)
    assert np.abs(lse - want_lse).max() < 1e-13


def pin_single_position(orc):
    """S = 1: O = V of the head's kv head, LSE = scale q.k, dV = sum of the group's dO, dQ = dK = 0."""
    q, k, v, dO = _problem(B=3, S=1, nh=6, nkv=2, hd=4, seed=3)
    scale = 0.37
    o, lse = orc.fwd(q, k, v, scale)
    dq, dk, dv = orc.bwd(q, k, v, dO, scale)
    g = 3
    for h in range(6):
        kvh = h // g
        assert np.allclose(o[:, 0, h], v[:, 0, kvh], rtol=0, atol=1e-14)
        want = scale * (q[:, 0, h] * k[:, 0, kvh]).sum(-1)
        assert np.allclose(lse[:, 0, h], want, rtol=0, atol=1e-14)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    want_dv = dO.reshape(3, 1, 2, g, 4).sum(axis=3)
    assert np.allclose(dv, want_dv, rtol=0, atol=1e-14)


def pin_constant_values(orc):
    """V = 1 everywhere: the softmax rows sum to 1, so O = 1 everywhere."""
    q, k, v, _ = _problem(B=2, S=11, nh=4, nkv=1, hd=3, seed=4)
    v[:] = 1.0
    o, _ = orc.fwd(q, k, v, 1.3)
    assert np.abs(o - 1.0).max() < 1e-13


def pin_finite_differences(orc):
    """Central differences of L = sum(dO * O) against the analytic backward."""
    for (nh, nkv) in ((4, 2), (3, 3)):
        q, k, v, dO = _problem(B=1, S=5, nh=nh, nkv=nkv, hd=3, seed=5)
        scale = 0.8
        dq, dk, dv = orc.bwd(q, k, v, dO, scale)
        eps = 1e-6
        for x, grad in ((q, dq), (k, dk), (v, dv)):
            fd = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                keep = x[idx]
                x[idx] = keep + eps
                lp = (dO * orc.fwd(q, k, v, scale)[0]).sum()
                x[idx] = keep - eps
                lm = (dO * orc.fwd(q, k, v, scale)[0]).sum()
                x[idx] = keep
                fd[idx] = (lp - lm) / (2 * eps)
            err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-12)
            assert err < 1e-7, err


def pin_composed(orc):
    """Agreement with the composed path (full Jacobian, literal repeat of K/V)."""
    q, k, v, dO = _problem(B=2, S=13, nh=6, nkv=2, hd=5, seed=6)
    scale = 1 / math.sqrt(5)
    o, lse = orc.fwd(q, k, v, scale)
    o2, lse2 = composed.forward(q, k, v, scale)
    assert _rel(o, o2) < 1e-12 and np.abs(lse - lse2).max() < 1e-12
    for a, b in zip(orc.bwd(q, k, v, dO, scale), composed.backward(q, k, v, dO, scale)):
        assert _rel(a, b) < 1e-12, _rel(a, b)


def pin_torch_sdpa(orc):
    """Agreement with torch's causal SDPA in float64 on the CPU, with autograd (GQA enabled)."""
    import torch
    import torch.nn.functional as F
    q, k, v, dO = _problem(B=2, S=10, nh=4, nkv=2, hd=4, seed=7)
    scale = 0.45
    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3).copy(), requires_grad=True)
                  for x in (q, k, v))
    out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale, enable_gqa=True)
    out.backward(torch.tensor(dO.transpose(0, 2, 1, 3).copy()))
    o, _ = orc.fwd(q, k, v, scale)
    dq, dk, dv = orc.bwd(q, k, v, dO, scale)

    def back(t):
        return t.detach().numpy().transpose(0, 2, 1, 3)

    assert _rel(o, back(out)) < 1e-12
    for a, t in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert _rel(a, back(t)) < 1e-12, _rel(a, back(t))


def pin_torch_sdpa_head_dims(orc):
    """The same agreement at the head dims the kernels take (32, 64, 128), with groups of
    2 and 4 and a length that is not a multiple of anything in particular."""
    import torch
    import torch.nn.functional as F
    for hd, nh, nkv in ((32, 4, 2), (64, 4, 1), (128, 8, 2)):
        q, k, v, dO = _problem(B=1, S=19, nh=nh, nkv=nkv, hd=hd, seed=30 + hd)
        scale = 1 / math.sqrt(hd)
        tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3).copy(), requires_grad=True)
                      for x in (q, k, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale, enable_gqa=True)
        out.backward(torch.tensor(dO.transpose(0, 2, 1, 3).copy()))
        o, _ = orc.fwd(q, k, v, scale)
        dq, dk, dv = orc.bwd(q, k, v, dO, scale)
        back = lambda t: t.detach().numpy().transpose(0, 2, 1, 3)  # noqa: E731
        assert _rel(o, back(out)) < 1e-12, hd
        for a, t in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert _rel(a, back(t)) < 1e-12, (hd, _rel(a, back(t)))


def pin_gqa_equals_repeated_mha(orc):
    """GQA on (K, V) equals MHA on K/V repeated per group, with dK/dV summed over each group."""
    q, k, v, dO = _problem(B=2, S=8, nh=6, nkv=3, hd=4, seed=8)
    scale = 0.5
    g = 2
    kr, vr = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    o, lse = orc.fwd(q, k, v, scale)
    o2, lse2 = orc.fwd(q, kr, vr, scale)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    dq, dk, dv = orc.bwd(q, k, v, dO, scale)
    dq2, dkr, dvr = orc.bwd(q, kr, vr, dO, scale)
    assert _rel(dq, dq2) < 1e-14
    assert _rel(dk, dkr.reshape(2, 8, 3, g, 4).sum(3)) < 1e-13
    assert _rel(dv, dvr.reshape(2, 8, 3, g, 4).sum(3)) < 1e-13


def pin_invariants(orc):
    """Identities of the gradient, per (batch, kv head), summed over its query group.

    sum_j dV_j = sum_{i, heads of group} dO_i        (softmax rows sum to 1)
    sum_j dK_j = 0                                    (K -> K + c shifts each row's scores by a constant)
    sum_{i,h} q.dq = sum_j k.dk                       (Q -> aQ, K -> K/a leaves scores unchanged)
    max_j s_ij <= LSE_i <= max_j s_ij + ln(i+1)
    """
    q, k, v, dO = _problem(B=2, S=12, nh=8, nkv=2, hd=5, seed=9)
    scale = 0.6
    g = 4
    dq, dk, dv = orc.bwd(q, k, v, dO, scale)
    B, S = 2, 12
    sum_do = dO.reshape(B, S, 2, g, 5).sum(axis=(1, 3))
    assert np.allclose(dv.sum(axis=1), sum_do, atol=1e-12)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12
    lhs = (q * dq).reshape(B, S, 2, g, 5).sum(axis=(1, 3, 4))
    rhs = (k * dk).sum(axis=(1, 3))
    assert np.allclose(lhs, rhs, atol=1e-12)
    _, lse = orc.fwd(q, k, v, scale)
    s = scale * np.einsum("bihd,bjhd->bhij", q, np.repeat(k, g, axis=2))
    s = np.where(np.triu(np.ones((S, S), bool), 1), -np.inf, s)
    mx = s.max(-1).transpose(0, 2, 1)
    n = np.arange(1, S + 1)[None, :, None]
    assert np.all(lse >= mx - 1e-12) and np.all(lse <= mx + np.log(n) + 1e-12)


def pin_key_shift(orc):
    """K -> K + c for one vector c: O is unchanged and LSE_i moves by scale q_i.c."""
    q, k, v, _ = _problem(B=1, S=9, nh=2, nkv=1, hd=4, seed=10)
    c = np.array([0.3, -1.1, 0.7, 2.0])
    scale = 0.9
    o, lse = orc.fwd(q, k, v, scale)
    o2, lse2 = orc.fwd(q, k + c, v, scale)
    assert _rel(o2, o) < 1e-12
    assert np.abs(lse2 - lse - scale * (q * c).sum(-1)).max() < 1e-12


def _decode_problem(B=2, T=13, nh=4, nkv=2, hd=5, seed=11):
    rng = np.random.default_rng(seed)
    return _rand((B, nh, hd), rng), _rand((B, T, nkv, hd), rng), _rand((B, T, nkv, hd), rng)


def pin_decode_last_row(orc):
    """Decode equals the last row of full causal attention (milestone M2a's own gate):
    with the query placed at position T-1 of a full sequence, the causal forward's last
    row and LSE are the decode's output."""
    q, k, v = _decode_problem()
    B, T, nh, hd = 2, 13, 4, 5
    rng = np.random.default_rng(12)
    q_full = _rand((B, T, nh, hd), rng)
    q_full[:, T - 1] = q
    scale = 0.8
    o_full, lse_full = orc.fwd(q_full, k, v, scale)
    o, lse = orc.decode(q, k, v, scale)
    assert _rel(o, o_full[:, T - 1]) < 1e-12
    assert np.abs(lse - lse_full[:, T - 1]).max() < 1e-12


def pin_decode_closed_forms(orc):
    """T = 1: O = v_0 and LSE = scale q.k_0. q = 0: O is the mean of the cached V rows of
    the query's kv head (contiguous groups) and LSE = ln T."""
    q, k, v = _decode_problem(T=1, seed=13)
    scale = 0.45
    o, lse = orc.decode(q, k, v, scale)
    kv_of = np.arange(4) // 2
    assert _rel(o, v[:, 0, kv_of]) < 1e-14
    assert np.abs(lse - scale * np.einsum("bhd,bhd->bh", q, k[:, 0, kv_of])).max() < 1e-13
    q, k, v = _decode_problem(T=10, seed=14)
    o, lse = orc.decode(np.zeros_like(q), k, v, scale)
    assert _rel(o, v.mean(axis=1)[:, kv_of]) < 1e-13
    assert np.abs(lse - math.log(10)).max() < 1e-13


def pin_decode_composed(orc):
    """Decode against the composed formulation (repeated K/V, materialised scores)."""
    q, k, v = _decode_problem(B=3, T=21, nh=8, nkv=2, hd=6, seed=15)
    o, lse = orc.decode(q, k, v, 1.3)
    o2, lse2 = composed.decode(q, k, v, 1.3)
    assert _rel(o, o2) < 1e-12 and np.abs(lse - lse2).max() < 1e-12


PINS = [pin_golden_two_positions, pin_zero_queries, pin_single_position, pin_constant_values,
        pin_finite_differences, pin_composed, pin_torch_sdpa, pin_torch_sdpa_head_dims,
        pin_gqa_equals_repeated_mha,
        pin_invariants, pin_key_shift, pin_decode_last_row, pin_decode_closed_forms,
        pin_decode_composed]
