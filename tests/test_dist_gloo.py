"""The benchmark's multi-rank plumbing on CPU with the gloo backend, world size 2: each
rank draws its own batch of (batch, kv head) units (no data-path collective), ranks meet
at a barrier, and the timed figure is the maximum over ranks."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        from bwd_xattn_fwd_gb300 import workloads as W
        w = W.WORKLOADS["tiny"]
        x = W.make_inputs(w, seed=rank)                    # this rank's own units
        b.barrier(dist)
        t = b.max_over_ranks(dist, 1.0 + rank, torch.device("cpu"))
        out[rank] = (t, float(x["q"].double().sum()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_own_inputs():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0                   # max over ranks, seen by every rank
    assert res[0][1] != res[1][1]                          # different seeds: different units
