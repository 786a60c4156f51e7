"""Composed attention in numpy fp64 (test infrastructure; small inputs only).

The second, independent formulation of the oracle. It follows the pages' composed
path: materialise the causal S x S scores, take the row softmax, multiply by V
(xtrain "Known Issues & Perf Backlog", KI-1 fix: strided-batched GEMM, causal
softmax, strided-batched GEMM). Its backward uses the full softmax Jacobian-vector
product dS = P * (dP - rowsum(P * dP)), not the D = rowsum(dO * O) shortcut of the
fused method (xtrain "演进总览", phase table row T14), so agreement between the two
pins that shortcut. Grouped KV heads are handled by literally repeating K and V
``group`` times and summing their gradients back over each group (row T15).
"""
from __future__ import annotations

import numpy as np


def _repeat_kv(x: np.ndarray, group: int) -> np.ndarray:
    # kv head kvh feeds query heads kvh*group + r, r < group
    return np.repeat(x, group, axis=2)


def _sum_groups(dx: np.ndarray, nkv: int) -> np.ndarray:
    B, S, nh, hd = dx.shape
    return dx.reshape(B, S, nkv, nh // nkv, hd).sum(axis=3)


def _probs(q, k, scale):
    # q, k: [B, H, S, hd] -> P [B, H, S, S] and natural-log LSE [B, H, S]
    s = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    S = s.shape[-1]
    future = np.triu(np.ones((S, S), dtype=bool), k=1)
    s = np.where(future, -np.inf, s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def forward(q, k, v, scale):
    """Returns (o [B,S,nh,hd], lse [B,S,nh])."""
    nh, nkv = q.shape[2], k.shape[2]
    g = nh // nkv
    qh = np.swapaxes(q, 1, 2)
    kh = np.swapaxes(_repeat_kv(k, g), 1, 2)
    vh = np.swapaxes(_repeat_kv(v, g), 1, 2)
    p, lse = _probs(qh, kh, scale)
    o = np.matmul(p, vh)
    return np.swapaxes(o, 1, 2).copy(), np.swapaxes(lse, 1, 2).copy()


def backward(q, k, v, dO, scale):
    """Returns (dq, dk, dv) for the loss sum(dO * O)."""
    nh, nkv = q.shape[2], k.shape[2]
    g = nh // nkv
    qh = np.swapaxes(q, 1, 2)
    kh = np.swapaxes(_repeat_kv(k, g), 1, 2)
    vh = np.swapaxes(_repeat_kv(v, g), 1, 2)
    doh = np.swapaxes(dO, 1, 2)
    p, _ = _probs(qh, kh, scale)
    dp = np.matmul(doh, np.swapaxes(vh, -1, -2))
    # softmax Jacobian-vector product, row by row
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = scale * np.matmul(ds, kh)
    dk_rep = scale * np.matmul(np.swapaxes(ds, -1, -2), qh)
    dv_rep = np.matmul(np.swapaxes(p, -1, -2), doh)
    dq = np.swapaxes(dq, 1, 2).copy()
    dk = _sum_groups(np.swapaxes(dk_rep, 1, 2), nkv)
    dv = _sum_groups(np.swapaxes(dv_rep, 1, 2), nkv)
    return dq, dk, dv


def decode(q, k, v, scale):
    """One new query per sequence against its cached K/V (xtrain "演进总览", milestone
    M2a: single query x cached K/V through a strided GEMM and a plain softmax).

    q [B, nh, hd], k, v [B, T, nkv, hd] -> (o [B, nh, hd], lse [B, nh]). No mask: the
    query is the newest position, so every cached key is visible.
    """
    nh, nkv = q.shape[1], k.shape[2]
    g = nh // nkv
    kh = np.swapaxes(_repeat_kv(k, g), 1, 2)          # [B, nh, T, hd]
    vh = np.swapaxes(_repeat_kv(v, g), 1, 2)
    s = scale * np.einsum("bhd,bhtd->bht", q, kh)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=-1, keepdims=True)
    o = np.einsum("bht,bhtd->bhd", e / z, vh)
    return o, (m + np.log(z))[..., 0]
