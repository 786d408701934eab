"""bench.py's host-side pieces, without a GPU: the ncu export parser behind
profiles/traffic.json, the nvidia-smi clock summary, and the throughput
arithmetic of the JSON line."""

import importlib.util
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


NCU_RAW = "\n".join([
    '"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum","gpu__time_duration.sum"',
    '"","","Mbyte","Kbyte","us"',
    '"0","void fa2::fa2_fwd_kernel<128, true, true>(CUtensorMap_st, FwdArgs)","201.5","51765.5","411.7"',
    '"1","void fa2::fa2_bwd_pre_kernel<128, true>(const unsigned short *, int)","0.135","4.4","27.3"',
    '"2","void fa2::fa2_fwd_kernel<128, true, true>(CUtensorMap_st, FwdArgs)","999","999","1"',
    '"3","fa2_bwd_main_kernel","1.5","2","520"',
])


def test_ncu_export_parsing(bench):
    got = bench.parse_ncu_dram(NCU_RAW)
    assert set(got) == {"fa2_fwd_kernel", "fa2_bwd_pre_kernel", "fa2_bwd_main_kernel"}
    assert got["fa2_fwd_kernel"] == pytest.approx((201.5e6, 51765.5e3))  # first launch only
    assert got["fa2_bwd_pre_kernel"] == pytest.approx((0.135e6, 4.4e3))
    assert got["fa2_bwd_main_kernel"] == pytest.approx((1.5e6, 2e3))


def test_clock_summary(bench):
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1399.2, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = ["0, 1500, 2070, 800, 0x8, Active, Not Active, Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.lines = []
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_throughput_arithmetic(bench):
    # 2 ranks x 10 steps x 1 TFLOP in 5 ms on the slowest rank = 4000 TFLOP/s
    assert bench.job_tflops(1e12, 2, 10, 5.0) == pytest.approx(4000.0)
    assert bench.slowest_rank_ms(3.25) == 3.25
