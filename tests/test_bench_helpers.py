"""Host-side helpers of bench.py on CPU: the packed transfer buffers of the end-to-end
run (one copy per direction per step) and the committed ncu traffic lookup."""
import importlib.util
import json
import os

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_helpers_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_packed_views_layout():
    b = _bench()
    specs = [("q", (2, 3, 4, 8), torch.bfloat16), ("lse", (2, 3, 4), torch.float32),
             ("k", (2, 3, 2, 8), torch.bfloat16), ("one", (1,), torch.float32)]
    flat, v = b.packed_views(specs)
    base = flat.data_ptr()
    end = 0
    for n, shape, dt in specs:
        t = v[n]
        assert t.shape == torch.Size(shape) and t.dtype == dt and t.is_contiguous()
        off = t.data_ptr() - base
        assert off % 256 == 0 and off >= end                 # aligned, in order, no overlap
        end = off + t.numel() * t.element_size()
    assert end <= flat.numel() and flat.numel() % 256 == 0
    # Writing through one view leaves the others untouched.
    for n in v:
        v[n].zero_()
    v["lse"].fill_(3.0)
    assert float(v["q"].float().abs().sum()) == 0.0 and float(v["k"].float().abs().sum()) == 0.0
    assert float(v["lse"].sum()) == 3.0 * 24


def test_traffic_entries_match_current_sources():
    """Every committed traffic figure whose kernel sources are unchanged is reported, and a
    figure recorded against other sources is not."""
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    for kernel, per_workload in rec.items():
        if kernel.startswith("_"):
            continue
        assert kernel in b.KERNEL_SOURCES, kernel
        for workload, e in per_workload.items():
            got = b.ncu_traffic(kernel, workload)
            if e["source_sha"] == b.source_sha(kernel):
                assert got == e["dram_bytes_per_launch"] == e["read"] + e["write"]
            else:
                assert got is None


def test_nvml_clock_summary_reports_reasons_and_median():
    """The 2 ms NVML sampler's summary: median and minimum SM clock over the samples, and
    every throttle reason seen in any sample (bits of nvmlClocksEventReasons)."""
    bench = _bench()
    s = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    s.rows = [{"sm": 2070.0, "max": 2070.0, "power": 900.0, "reasons": 0},
              {"sm": 2040.0, "max": 2070.0, "power": 1300.0, "reasons": 0x4},
              {"sm": 2070.0, "max": 2070.0, "power": None, "reasons": 0x1}]
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_mhz_min"] == 2040.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3 and out["power_w_max"] == 1300.0
    s.rows = [{"sm": 1500.0, "max": 2070.0, "power": 500.0, "reasons": 0x8 | 0x40}]
    assert s.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
