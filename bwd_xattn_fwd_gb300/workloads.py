"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CUDA path's tests and benchmark and by the oracle's
tests. It draws random numbers and shapes them; it holds none of the attention
arithmetic. The shapes are the decoder attention shapes of the xtrain trainer
(xtrain "演进总览" / docs/evolution.md, scaling-runs table and phase rows T9, T14,
T15): per-head QK-norm makes Q/K rows unit-norm before scaling (row T9), GQA uses a
query group of 4 (rows T15, v9).

Recipe (every workload):
  * generator ``torch.Generator('cpu').manual_seed(seed)`` (seed 0 by default);
  * draw order q, k, v, dO, each ``torch.randn`` in float32 in its row-major shape
    q/dO [B,S,nh,hd], k/v [B,S,nkv,hd];
  * apply the workload's scaling in float32, then cast to the workload dtype
    (bf16 with round-to-nearest-even, or kept in float32).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    nh: int
    nkv: int
    hd: int
    dtype: str              # "bf16" or "f32"
    qkv_scale: float = 1.0  # multiplies q, k, v (unless qk_norm applies to q, k)
    do_scale: float = 1.0   # multiplies dO
    qk_norm: bool = False   # L2-normalise each q/k row over hd, then times sqrt(hd)
    description: str = ""

    @property
    def group(self) -> int:
        return self.nh // self.nkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)

    @property
    def pairs(self) -> int:
        """Causal (i, j) pairs per (batch, query head): S(S+1)/2."""
        return self.S * (self.S + 1) // 2

    @property
    def fwd_flops(self) -> int:
        """Q K^T and P V over the causal pairs: 4 hd flops per pair."""
        return 4 * self.hd * self.pairs * self.B * self.nh

    @property
    def bwd_flops(self) -> int:
        """Recomputed Q K^T, dP = dO V^T, dV, dK, dQ: 10 hd flops per pair."""
        return 10 * self.hd * self.pairs * self.B * self.nh

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=2, S=64, nh=4, nkv=4, hd=8, dtype="f32",
                     description="tiny oracle check, fp32, iid N(0,1)"),
    "dim384": Workload("dim384", B=16, S=256, nh=12, nkv=12, hd=32, dtype="bf16",
                       qkv_scale=0.5, do_scale=0.5,
                       description="dim384 decoder attention, MHA, iid N(0,1)*0.5"),
    "dim768": Workload("dim768", B=32, S=1024, nh=12, nkv=12, hd=64, dtype="bf16",
                       qk_norm=True,
                       description="dim768 decoder attention, MHA, QK-norm-like rows"),
    "gqa": Workload("gqa", B=8, S=2048, nh=8, nkv=2, hd=64, dtype="bf16",
                    qkv_scale=0.5, do_scale=1.0,
                    description="GQA attention, group 4, q/k/v N(0,1)*0.5, dO N(0,1)"),
    "long": Workload("long", B=4, S=4096, nh=16, nkv=4, hd=64, dtype="bf16",
                     qkv_scale=0.5, do_scale=1.0,
                     description="long-seq dim1024 GQA, group 4"),
    "long_hd128": Workload("long_hd128", B=4, S=4096, nh=16, nkv=4, hd=128, dtype="bf16",
                           qkv_scale=0.5, do_scale=1.0,
                           description="long-seq GQA at head dim 128 (dim2048), group 4"),
}

ORDER = ["tiny", "dim384", "dim768", "gqa", "long", "long_hd128"]


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def make_inputs(w: Workload, seed: int = 0):
    """Returns dict(q, k, v, dO) of CPU tensors in the workload dtype."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((w.B, w.S, w.nh, w.hd), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.S, w.nkv, w.hd), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.S, w.nkv, w.hd), generator=g, dtype=torch.float32)
    dO = torch.randn((w.B, w.S, w.nh, w.hd), generator=g, dtype=torch.float32)
    if w.qk_norm:
        root = math.sqrt(w.hd)
        q = q / q.norm(dim=-1, keepdim=True) * root
        k = k / k.norm(dim=-1, keepdim=True) * root
        v = v * w.qkv_scale
    else:
        q, k, v = q * w.qkv_scale, k * w.qkv_scale, v * w.qkv_scale
    dO = dO * w.do_scale
    dt = torch_dtype(w)
    return {name: t.to(dt).contiguous() for name, t in
            (("q", q), ("k", k), ("v", v), ("dO", dO))}


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decode step: B sequences, each one new query (all nh heads) against its T
    cached key/value positions (xtrain "演进总览", milestones M2a-M2c)."""
    name: str
    B: int
    T: int
    nh: int
    nkv: int
    hd: int
    qkv_scale: float = 0.5
    description: str = ""

    @property
    def group(self) -> int:
        return self.nh // self.nkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)

    @property
    def cache_bytes(self) -> int:
        """bf16 K and V caches, read once per step."""
        return 2 * self.B * self.T * self.nkv * self.hd * 2

    @property
    def io_bytes(self) -> int:
        """Algorithmic bytes per step: the caches, q and o (bf16), lse (fp32)."""
        return self.cache_bytes + 2 * self.B * self.nh * self.hd * 2 + self.B * self.nh * 4

    def with_(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


DECODE_WORKLOADS = {
    # The long workload's heads (nh=16, nkv=4, hd=64) over 64 sequences with 4096 cached
    # positions each: 268 MB of cache per step, more than the L2 holds.
    "decode": DecodeWorkload("decode", B=64, T=4096, nh=16, nkv=4, hd=64,
                             description="decode step, 64 sequences x 4096 cached positions, GQA group 4"),
}


def make_decode_inputs(w: DecodeWorkload, seed: int = 0):
    """Returns dict(q [B,nh,hd], k [B,T,nkv,hd], v [B,T,nkv,hd]) of bf16 CPU tensors:
    generator seeded as for make_inputs, draw order q, k, v, each torch.randn in
    float32 times qkv_scale, then cast to bf16."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((w.B, w.nh, w.hd), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.T, w.nkv, w.hd), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.T, w.nkv, w.hd), generator=g, dtype=torch.float32)
    return {name: (t * w.qkv_scale).to(torch.bfloat16).contiguous() for name, t in
            (("q", q), ("k", k), ("v", v))}


def as_f64(t: torch.Tensor):
    """Exact float64 numpy copy of a CPU tensor (bf16 and fp32 embed exactly)."""
    return t.detach().to("cpu", torch.float64).numpy()
