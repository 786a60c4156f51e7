"""Benchmark of fused causal GQA attention, forward + backward, on GB300.

One step = the whole hot path over one batch of seeded synthetic input already resident
in HBM: forward (xattn_fwd), then the backward's three kernels (D/LSE preprocess, main
recompute loop, dQ convert). The L2 cache (larger than the step's working set) is
flushed by a 256 MiB device write before every step, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gqa] [--impl ours|reference]

With --workload decode it times one decode step instead (xattn_decode: one new query
per sequence against 4096 cached positions, 64 sequences) and reports GB/s of cache
reads against the measured HBM copy bandwidth. Decode steps run back to back (no flush:
the 268 MB of caches exceed the L2, and alternate steps read two copies of them).

Prints ONE JSON line (rank 0). `value` is fwd+bwd TFLOP/s of algorithmic work
(4 hd flops per causal pair forward, 10 hd backward) summed over all ranks and divided
by the slowest rank's time. `--impl reference` times the CPU oracle on the host cores
instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bwd_xattn_fwd_gb300 import workloads as W  # noqa: E402

METRIC = "causal GQA attention fwd+bwd TFLOP/s & tok/s (bf16), % of GB300 tensor peak"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd_sm103.cu", "sm103_ptx.cuh"],
    "attn_bwd_main_kernel": ["attn_bwd_sm103.cu", "sm103_ptx.cuh"],
    "bwd_preprocess_kernel": ["attn_bwd_sm103.cu"],
    "dq_convert_kernel": ["attn_bwd_sm103.cu"],
    "decode_partial_kernel + decode_combine_kernel": ["attn_decode.cu", "sm103_ptx.cuh"],
    "bwd_deterministic": ["attn_bwd_sm103.cu", "attn_bwd_dq_sm103.cu", "sm103_ptx.cuh"],
    "bwd_resident_dq": ["attn_bwd_sm103.cu", "sm103_ptx.cuh"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gqa",
                    choices=[n for n in W.ORDER if n != "tiny"] + list(W.DECODE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as replays of one CUDA graph of it instead of stream launches")
    ap.add_argument("--deterministic", action="store_true",
                    help="time xattn_bwd_deterministic (bit-reproducible dQ) as the backward")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"tflops": p["bf16_tflops"], "tflops_sustained": p.get("bf16_tflops_sustained"),
                "gbs": p["hbm_gbs"], "source": "measured"}
    return {"tflops": 1900.0, "tflops_sustained": 1700.0, "gbs": 6800.0, "source": "fallback"}


def source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "bwd_xattn_fwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def packed_views(specs, device=None, pin=False):
    """One flat byte buffer holding tensors of the given (name, shape, dtype), each at a
    256-byte-aligned offset, so that a step moves its inputs (or outputs) with one copy.
    Returns (flat buffer, {name: typed view})."""
    import torch
    offs, total = {}, 0
    for n, shape, dt in specs:
        nbytes = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        offs[n] = (total, nbytes, shape, dt)
        total = (total + nbytes + 255) // 256 * 256
    flat = torch.empty(total, dtype=torch.uint8, device=device, pin_memory=pin)
    return flat, {n: flat[o:o + nb].view(dt).view(shape) for n, (o, nb, shape, dt) in offs.items()}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None if there is none
    for this kernel and workload or the kernel's source changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f).get(kernel, {}).get(workload)
    if not rec or rec.get("source_sha") != source_sha(kernel):
        return None
    return rec["dram_bytes_per_launch"]


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------
class NvmlClockSampler:
    """Reads the SM clock, power and clock-event reasons through NVML (the driver's
    libnvidia-ml, read-only queries) every 2 ms from a host thread while the timed loops
    run, so even a timed region of a few milliseconds gets samples under load. Falls back
    to ClockSampler (nvidia-smi, 100 ms) where NVML cannot be loaded."""
    PERIOD_S = 0.002
    # nvmlClocksEventReasons bits
    REASONS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"),
               (0x20, "sw_thermal_slowdown"), (0x4, "sw_power_cap"))

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        bus = torch_pci_bus_id(device_index)
        if bus is not None:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle))
        else:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.handle))
        if rc != 0:
            raise OSError(f"nvmlDeviceGetHandle failed ({rc})")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.rows = []
        self.stop = threading.Event()
        self.thread = None

    def _sample(self):
        ct = self.ct
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            ok = (self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(sm)) == 0 and
                  self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(mx)) == 0)
            pw = self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw)) == 0
            rr = self.reasons_fn(self.handle, ct.byref(rs)) == 0
            if ok:
                self.rows.append({"sm": float(sm.value), "max": float(mx.value),
                                  "power": mw.value / 1000.0 if pw else None,
                                  "reasons": rs.value if rr else 0})
            time.sleep(self.PERIOD_S)

    def __enter__(self):
        self.thread = threading.Thread(target=self._sample, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()

    def summary(self):
        if not self.rows:
            return None
        reasons = [name for bit, name in self.REASONS if any(r["reasons"] & bit for r in self.rows)]
        powers = [r["power"] for r in self.rows if r["power"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in self.rows),
                "sm_mhz_min": min(r["sm"] for r in self.rows),
                "sm_max_mhz": max(r["max"] for r in self.rows), "reasons": reasons,
                "samples": len(self.rows), "power_w_max": max(powers) if powers else None,
                "source": "NVML, every 2 ms during the timed loops"}


def torch_pci_bus_id(device_index: int):
    """PCI bus id of a CUDA device as NVML spells it, or None if torch does not expose it."""
    try:
        import torch
        p = torch.cuda.get_device_properties(device_index)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return None


def clock_sampler(device_index: int):
    try:
        return NvmlClockSampler(device_index)
    except (OSError, AttributeError):
        return ClockSampler(device_index)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hw_th": parts[6], "sw_th": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] is None or r["power"] > 200.0] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                          ("sw_th", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in loaded):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(loaded)}


# ---------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ---------------------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    pg = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
        pg = dist
    return rank, local, world, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float, device) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# CPU oracle timing (reported baseline)
# ---------------------------------------------------------------------------------------
def oracle_sample(w: W.Workload, x_cpu: dict, budget_s: float, max_units: int | None = None):
    """Times the oracle (fwd + bwd, all host cores) on whole (batch, kv head) units of the
    workload, in order, until `budget_s` seconds have passed or max_units are done."""
    cores = os.cpu_count() or 1
    os.environ["OMP_NUM_THREADS"] = str(cores)
    import oracle
    orc = oracle.default()
    units = [(b, kvh) for b in range(w.B) for kvh in range(w.nkv)]
    if max_units is not None:
        units = units[:max_units]
    done, elapsed = 0, 0.0
    for b, kvh in units:
        q, k, v, dO = (W.as_f64(x_cpu[n][b:b + 1]) for n in ("q", "k", "v", "dO"))
        uq, uk, uv, udo = oracle.unit_slices(q, k, v, dO, 0, kvh)
        t0 = time.perf_counter()
        orc.fwd(uq, uk, uv, w.scale)
        orc.bwd(uq, uk, uv, udo, w.scale)
        elapsed += time.perf_counter() - t0
        done += 1
        if elapsed >= budget_s:
            break
    frac = done / len([(b, k) for b in range(w.B) for k in range(w.nkv)])
    flops = (w.fwd_flops + w.bwd_flops) * frac
    return {"flops": flops, "tokens": w.tokens * frac, "seconds": elapsed, "units": done,
            "cores": cores,
            "sample": f"{done} of {w.B * w.nkv} (batch, kv-head) units of '{w.name}' at full S={w.S} "
                      f"({w.group} query heads each), fwd+bwd, fp64, OpenMP over rows"}


def run_reference(args, w: W.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = W.make_inputs(w, seed=0)
    for _ in range(args.warmup):
        oracle_sample(w, x, budget_s=0.0, max_units=1)
    per = [oracle_sample(w, x, budget_s=0.0, max_units=1) for _ in range(args.steps)]
    flops = sum(p["flops"] for p in per)
    secs = sum(p["seconds"] for p in per)
    toks = sum(p["tokens"] for p in per)
    value = flops / secs / 1e12
    cores = per[0]["cores"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "tok_per_s": toks / secs,
        "config": {"workload": w.name, "B": w.B, "S": w.S, "nh": w.nh, "nkv": w.nkv, "hd": w.hd,
                   "step": "one (batch, kv-head) unit, fwd+bwd"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": per[0]["sample"] + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def run_ours(args, w: W.Workload):
    import torch
    rank, local, world, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bwd_xattn_fwd_gb300 import xattn

    x_cpu = W.make_inputs(w, seed=rank)
    x = {n: t.to(dev) for n, t in x_cpu.items()}
    B, S, nh, nkv, hd, scale = w.B, w.S, w.nh, w.nkv, w.hd, w.scale
    o = torch.empty_like(x["q"])
    lse = torch.empty((B, S, nh), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    ws_bytes = xattn.xattn_bwd_workspace_bytes(B, S, nh, hd)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    names = ["attn_fwd_kernel", "bwd_preprocess_kernel", "attn_bwd_main_kernel", "dq_convert_kernel"]
    # The backward xattn_bwd (or, with --deterministic, xattn_bwd_deterministic) runs for
    # these sizes: the fused-dQ one is timed through its three stage calls (one segment
    # each); the deterministic one (xattn_bwd's at hd = 128) as one segment: its
    # preprocess, then dQ resident in tensor memory on small problems or the dK/dV and
    # query-stationary dQ kernels.
    mode = xattn.xattn_bwd_dq_mode(S, nh, nkv, hd, args.deterministic)
    det = mode != xattn.BWD_FUSED_DQ
    if det:
        names = ["attn_fwd_kernel",
                 "bwd_resident_dq" if mode == xattn.BWD_RESIDENT_DQ else "bwd_deterministic"]

    def step(evs=None, st=stream):
        if evs:
            evs[0].record(st)
        xattn.xattn_fwd(x["q"], x["k"], x["v"], B, S, nh, nkv, hd, scale, o, lse, st)
        if evs:
            evs[1].record(st)
        if det:
            xattn.xattn_bwd_deterministic(x["q"], x["k"], x["v"], o, x["dO"], lse, B, S, nh, nkv, hd,
                                          scale, dq, dk, dv, st)
            if evs:
                evs[2].record(st)
            return
        xattn.xattn_bwd_preprocess(o, x["dO"], lse, B, S, nh, hd, scale, ws, ws_bytes, st)
        if evs:
            evs[2].record(st)
        xattn.xattn_bwd_main(x["q"], x["k"], x["v"], x["dO"], B, S, nh, nkv, hd, scale, dk, dv,
                             ws, ws_bytes, st)
        if evs:
            evs[3].record(st)
        xattn.xattn_bwd_dq_convert(B, S, nh, hd, scale, dq, ws, ws_bytes, st)
        if evs:
            evs[4].record(st)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    status = xattn.xattn_check_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} during warm-up")

    # --graph: the headline replays one CUDA graph of the step (the forward and the
    # backward's calls, captured once after the eager warm-up), as a training loop may:
    # the same kernels and programmatic-launch edges without the host launch path. It
    # measured the same as the eager launches on every workload (the programmatic launches
    # already overlap each kernel's set-up with its predecessor), so eager is the default.
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            step(st=cap)
        torch.cuda.synchronize(dev)
        for _ in range(args.warmup):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize(dev)

    def timed_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    # Two timed loops over the same steps. The headline takes one pair of events per
    # step, so consecutive kernels of a step follow each other directly in the stream (an
    # event between them would stop the next one's programmatic early launch). The
    # per-kernel breakdown (roofline) comes from a second loop with an event between
    # every two kernels.
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
              for _ in range(args.steps)]
    barrier(pg)
    torch.cuda.synchronize(dev)
    with clock_sampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            step_events[i][0].record(stream)
            timed_step()
            step_events[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg)
        for i in range(args.steps):
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize(dev)
    barrier(pg)
    status = xattn.xattn_check_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")

    per_kernel = {n: [ev[j].elapsed_time(ev[j + 1]) for ev in events] for j, n in enumerate(names)}
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in step_events]
    total_ms = max_over_ranks(pg, sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    flops_step = w.fwd_flops + w.bwd_flops
    value = flops_step * world * args.steps / (total_ms * 1e-3) / 1e12
    tok_s = w.tokens * world * args.steps / (total_ms * 1e-3)

    pk = peaks()
    kavg = {n: statistics.mean(v) for n, v in per_kernel.items()}
    S_pad = (S + 127) // 128 * 128
    elems = B * S * nh * hd
    # Algorithmic work per launch: the forward's 2 products and the backward's 5 (2 hd
    # flops per causal pair and head each); the preprocess reads O, dO and lse and
    # writes the auxiliary rows, D and the zeroed dQ accumulator; the convert reads the
    # accumulator and writes dq.
    kernel_work = {
        "attn_fwd_kernel": ("tensor", w.fwd_flops),
        "attn_bwd_main_kernel": ("tensor", w.bwd_flops),
        "bwd_preprocess_kernel": ("hbm", 2 * elems * 2 + B * S * nh * 4 + B * nh * S_pad * 32
                                  + B * S * nh * 4 + elems * 4),
        "dq_convert_kernel": ("hbm", elems * 4 + elems * 2),
        "bwd_deterministic": ("tensor", w.bwd_flops),
        "bwd_resident_dq": ("tensor", w.bwd_flops),
    }
    kernels = {}
    for n in names:
        bound, work = kernel_work[n]
        ms = kavg[n]
        if bound == "tensor":
            ach = work / (ms * 1e-3) / 1e12
            kernels[n] = {"ms": ms, "bound": "tensor", "achieved": ach, "unit": "TFLOP/s",
                          "frac": ach / pk["tflops"], "share": ms / sum(kavg.values())}
        else:
            ach = work / (ms * 1e-3) / 1e9
            kernels[n] = {"ms": ms, "bound": "hbm", "achieved": ach, "unit": "GB/s",
                          "frac": ach / pk["gbs"], "share": ms / sum(kavg.values())}
    dominant = max(names, key=lambda n: kavg[n])
    d = kernels[dominant]
    bound, work = kernel_work[dominant]
    roofline = {"kernel": dominant, "bound": d["bound"], "achieved": d["achieved"],
                "peak": pk["tflops"] if bound == "tensor" else pk["gbs"], "unit": d["unit"],
                "frac": d["frac"], "traffic": ncu_traffic(dominant, w.name),
                "algorithmic_per_launch": work, "peak_source": pk["source"] + " (burst)"}

    # End to end through the public API with host buffers: every step copies its inputs
    # in from pinned host memory (H2D), runs xattn_fwd + xattn_bwd (which takes its own
    # scratch) and copies every output back (D2H). The steps are pipelined over three
    # streams with two sets of device buffers, as a training loop would overlap them: the
    # H2D copies of step i+1 and the D2H copies of step i-1 run while step i computes.
    e2e = None
    if not args.no_e2e:
        # Each step's inputs sit in one pinned buffer and its outputs in one device buffer
        # (256-byte-aligned views), so a step is one H2D and one D2H copy.
        in_specs = [(n, tuple(t.shape), t.dtype) for n, t in x_cpu.items()]
        out_specs = [(n, tuple(t.shape), t.dtype) for n, t in
                     (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))]
        h_in_flat, h_in = packed_views(in_specs, pin=True)
        for n, t in x_cpu.items():
            h_in[n].copy_(t)
        d_in = [packed_views(in_specs, device=dev) for _ in range(2)]
        d_out = [packed_views(out_specs, device=dev) for _ in range(2)]
        h_out = [packed_views(out_specs, pin=True) for _ in range(2)]
        h2d = h_in_flat.numel()
        d2h = h_out[0][0].numel()
        s_h2d, s_cmp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]
        bwd = xattn.xattn_bwd_deterministic if det else xattn.xattn_bwd

        def e2e_step(i):
            j = i % 2
            (di_flat, di), (do_flat, do_), (ho_flat, _) = d_in[j], d_out[j], h_out[j]
            if i >= 2:
                s_h2d.wait_event(cmp_done[j])          # step i-2 has consumed d_in[j]
            with torch.cuda.stream(s_h2d):
                di_flat.copy_(h_in_flat, non_blocking=True)
            h2d_done[j].record(s_h2d)
            s_cmp.wait_event(h2d_done[j])
            if i >= 2:
                s_cmp.wait_event(d2h_done[j])          # step i-2's outputs have left d_out[j]
            xattn.xattn_fwd(di["q"], di["k"], di["v"], B, S, nh, nkv, hd, scale, do_["o"], do_["lse"],
                            s_cmp)
            bwd(di["q"], di["k"], di["v"], do_["o"], di["dO"], do_["lse"], B, S, nh, nkv, hd, scale,
                do_["dq"], do_["dk"], do_["dv"], s_cmp)
            cmp_done[j].record(s_cmp)
            s_d2h.wait_event(cmp_done[j])
            with torch.cuda.stream(s_d2h):
                ho_flat.copy_(do_flat, non_blocking=True)
            d2h_done[j].record(s_d2h)

        for i in range(max(3, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(pg)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_h2d)
        for i in range(args.steps):
            e2e_step(i)
        s_d2h.wait_stream(s_cmp)
        e1.record(s_d2h)
        torch.cuda.synchronize(dev)
        t_e2e = max_over_ranks(pg, e0.elapsed_time(e1), dev)
        if xattn.xattn_check_device_status(s_cmp) != 0:
            raise RuntimeError("device status in the e2e run")
        # The last step's results are the same as the device-resident run's.
        last = (args.steps - 1) % 2
        ho_last = h_out[last][1]
        if not (torch.equal(ho_last["o"], o.cpu()) and torch.equal(ho_last["dk"], dk.cpu())):
            raise RuntimeError("e2e outputs differ from the device-resident run")
        e2e = {"value": flops_step * world * args.steps / (t_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "tok_per_s": w.tokens * world * args.steps / (t_e2e * 1e-3),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "steps pipelined over three streams (H2D of the next step and D2H of the "
                       "previous one overlap this step's kernels), two sets of device buffers; a "
                       "step's inputs and outputs each move as one packed copy"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = oracle_sample(w, x_cpu, budget_s=12.0)
        cpu = {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"],
               "tok_per_s": r["tokens"] / r["seconds"], "seconds": r["seconds"]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "S": w.S, "nh": w.nh, "nkv": w.nkv,
                       "hd": w.hd, "scale": scale,
                       "backward": ("deterministic, dQ resident in tensor memory" if mode == xattn.BWD_RESIDENT_DQ
                                    else "deterministic dQ" if det else "default"),
                       "launch": "eager stream launches" if graph is None else
                                 "CUDA graph of the step, replayed (per-kernel times: eager launches)",
                       "parallelism": f"{world} rank(s), each its own batch of (batch, kv-head) units; no collective",
                       "l2": "flushed before every step (256 MiB device write, outside the timed events)"},
            "tok_per_s": tok_s,
            "frac_of_peak": value / world / pk["tflops"],
            "frac_of_sustained_peak": value / world / pk["tflops_sustained"] if pk["tflops_sustained"] else None,
            "roofline": roofline, "kernels": kernels,
            "ms_per_step_with_kernel_events": statistics.mean(ev[0].elapsed_time(ev[len(names)]) for ev in events),
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (3 if mode == xattn.BWD_RESIDENT_DQ else 4) * args.steps, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ---------------------------------------------------------------------------------------
# decode mode: one decode step (one new query per sequence against its cached K/V)
# ---------------------------------------------------------------------------------------
DECODE_METRIC = "decode attention GB/s of KV-cache reads (bf16), % of GB300 HBM copy bandwidth"


def decode_oracle_sample(w, x_cpu, budget_s: float, max_seqs=None):
    """Times the oracle's decode (fp64, all host cores) on whole sequences, in order."""
    cores = os.cpu_count() or 1
    os.environ["OMP_NUM_THREADS"] = str(cores)
    import oracle
    orc = oracle.default()
    n = w.B if max_seqs is None else min(max_seqs, w.B)
    done, elapsed = 0, 0.0
    for b in range(n):
        q, k, v = (W.as_f64(x_cpu[name][b:b + 1]) for name in ("q", "k", "v"))
        t0 = time.perf_counter()
        orc.decode(q, k, v, w.scale)
        elapsed += time.perf_counter() - t0
        done += 1
        if elapsed >= budget_s:
            break
    frac = done / w.B
    return {"bytes": w.io_bytes * frac, "seqs": done, "seconds": elapsed, "cores": cores,
            "sample": f"{done} of {w.B} sequences of '{w.name}' (T={w.T}, {w.nh} query heads), fp64, "
                      f"OpenMP over heads"}


def run_decode_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    x = W.make_decode_inputs(w, seed=0)
    for _ in range(args.warmup):
        decode_oracle_sample(w, x, 0.0, max_seqs=1)
    per = [decode_oracle_sample(w, x, 0.0, max_seqs=1) for _ in range(args.steps)]
    secs = sum(p["seconds"] for p in per)
    value = sum(p["bytes"] for p in per) / secs / 1e9
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "nh": w.nh, "nkv": w.nkv, "hd": w.hd,
                       "step": "one sequence's decode"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": per[0]["cores"], "kind": "oracle",
                             "sample": per[0]["sample"] + " per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decode(args, w):
    import torch
    rank, local, world, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bwd_xattn_fwd_gb300 import xattn
    x_cpu = W.make_decode_inputs(w, seed=rank)
    x = {n: t.to(dev) for n, t in x_cpu.items()}
    B, T, nh, nkv, hd, scale = w.B, w.T, w.nh, w.nkv, w.hd, w.scale
    o = torch.empty_like(x["q"])
    lse = torch.empty((B, nh), dtype=torch.float32, device=dev)
    # Two copies of the caches, read by alternate steps: each copy exceeds the L2, and no
    # step finds in the L2 what the step before it left there.
    caches = [(x["k"], x["v"]), (x["k"].clone(), x["v"].clone())]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        k, v = caches[i % 2]
        xattn.xattn_decode(x["q"], k, v, B, T, nh, nkv, hd, scale, o, lse, stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    if xattn.xattn_check_device_status(stream) != 0:
        raise RuntimeError("device status during warm-up")
    # The steps run back to back between two events (a decode loop's cadence): a flush
    # inside the loop would leave the device waiting for the host between steps.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize(dev)
    with clock_sampler(local) as clk:
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(pg)
    if xattn.xattn_check_device_status(stream) != 0:
        raise RuntimeError("device status in the timed region")
    total_ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    ms = total_ms / args.steps
    value = w.io_bytes * world * args.steps / (total_ms * 1e-3) / 1e9
    # one kernel when each (sequence, kv head) is one run, else the partial kernel and the combine
    runs = xattn.xattn_decode_runs(B, T, nh, nkv, hd, torch.cuda.get_device_properties(dev).multi_processor_count)
    launches_per_step = 1 if runs == 1 else 2
    pk = peaks()
    roofline = {"kernel": "decode_partial_kernel + decode_combine_kernel", "bound": "hbm",
                "achieved": value / world, "peak": pk["gbs"], "unit": "GB/s",
                "frac": value / world / pk["gbs"],
                "traffic": ncu_traffic("decode_partial_kernel + decode_combine_kernel", w.name),
                "algorithmic_per_launch": w.io_bytes, "peak_source": pk["source"] + " (copy)"}

    e2e = None
    if not args.no_e2e:
        h_q = x_cpu["q"].pin_memory()
        h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        h_l = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        d_q = torch.empty_like(x["q"])

        def e2e_step(i):
            k, v = caches[i % 2]
            d_q.copy_(h_q, non_blocking=True)
            xattn.xattn_decode(d_q, k, v, B, T, nh, nkv, hd, scale, o, lse, stream)
            h_o.copy_(o, non_blocking=True)
            h_l.copy_(lse, non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t = max_over_ranks(pg, e0.elapsed_time(e1), dev)
        # Decode is bit-reproducible: the host copy of the last step equals the device run's.
        if not (torch.equal(h_o, o.cpu()) and torch.equal(h_l, lse.cpu())):
            raise RuntimeError("decode e2e outputs differ from the device-resident run")
        e2e = {"value": w.io_bytes * world * args.steps / (t * 1e-3) / 1e9, "unit": "GB/s",
               "tok_per_s": B * world * args.steps / (t * 1e-3),
               "h2d_bytes_per_step": h_q.numel() * h_q.element_size(),
               "d2h_bytes_per_step": h_o.numel() * h_o.element_size() + h_l.numel() * h_l.element_size(),
               "note": "the K/V caches stay resident on the device (as in a decode loop); the new "
                       "token's query comes in and the output goes out each step"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = decode_oracle_sample(w, x_cpu, budget_s=10.0)
        cpu = {"value": r["bytes"] / r["seconds"] / 1e9, "unit": "GB/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"], "seconds": r["seconds"]}
    if rank == 0:
        line = {"metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name, "B": B, "T": T, "nh": nh, "nkv": nkv, "hd": hd,
                           "parallelism": f"{world} rank(s), each its own sequences; no collective",
                           "l2": "no flush: each step reads caches of %.0f MB (> L2), alternating "
                                 "between two copies" % (w.cache_bytes / 1e6)},
                "tok_per_s": B * world / (ms * 1e-3), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.workload in W.DECODE_WORKLOADS:
        w = W.DECODE_WORKLOADS[args.workload]
        if args.impl == "reference":
            run_decode_reference(args, w)
        else:
            run_decode(args, w)
        return
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
