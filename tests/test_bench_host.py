"""Host logic of bench.py that needs no GPU: the algorithmic bytes of the
prefill roofline and the clock summary (NVML samples with the idle ones
left out, or nvidia-smi lines), fed with made-up samples."""
from __future__ import annotations

import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_algorithmic_bytes_counts_valid_prefixes_and_ids():
    # row i of 4096 has cols - 4096 + i + 1 valid columns
    for cols in (8192, 51200, 102400):
        ends = cols - 4096 + np.arange(4096) + 1
        assert bench.algorithmic_bytes(cols) == int(ends.sum()) * 4 + 4096 * 512 * 4
    assert bench.algorithmic_bytes(102400) == 1652563968
    # more rows than columns: leading rows are empty, never negative
    assert bench.algorithmic_bytes(10, rows=16, k=1) == sum(range(1, 11)) * 4 + 16 * 4


def _nvml_sampler(samples, max_mhz=2070.0):
    c = bench.ClockSampler(0)
    c.thread = object()  # as if the NVML poller had run
    c.samples = samples
    c.max_mhz = max_mhz
    return c


def test_clock_summary_leaves_out_idle_samples():
    idle = bench.NVML_REASON_BITS["gpu_idle"]
    cap = bench.NVML_REASON_BITS["sw_power_cap"]
    c = _nvml_sampler([(345.0, idle), (2070.0, 0), (2055.0, cap), (2070.0, 0), (600.0, idle)])
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["source"] == "nvml"


def test_clock_summary_names_every_slowdown():
    bits = bench.NVML_REASON_BITS
    c = _nvml_sampler([(1500.0, bits["hw_slowdown"]), (1400.0, bits["hw_thermal_slowdown"]),
                       (1300.0, bits["sw_thermal_slowdown"] | bits["sw_power_cap"])])
    assert c.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown",
                                      "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_all_idle_is_unsampled():
    c = _nvml_sampler([(345.0, bench.NVML_REASON_BITS["gpu_idle"])])
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["unsampled"]


def test_clock_summary_from_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["2070, 2070, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "[N/A], 2070, x, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["source"] == "nvidia-smi" and s["samples"] == 2
    assert s["sm_mhz"] == pytest.approx(2025.0) and s["reasons"] == ["sw_power_cap"]


def test_device_uuid_without_a_gpu_is_none():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert bench.device_uuid(0) is None


def test_vs_baseline_reference_figure():
    # 12288 rows over the pages' 80.9 + 321.4 + 688.3 us
    assert bench.pages_rows_per_s() == pytest.approx(12288 / 1090.6e-6)
    assert bench.pages_rows_per_s(widths=(8192,)) is None
    assert bench.pages_rows_per_s(rows=1024) is None
