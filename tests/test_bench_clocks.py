"""bench.py's clock summary: only samples taken inside the timed region count.

nvidia-smi prints one row per 50 ms; the summary keeps the rows whose
timestamp falls inside the host-time window around the timed region, reports
their median SM clock, the highest maximum clock and every active throttle
reason, and falls back to all rows (saying so) when none can be placed.
"""
import datetime
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

T0 = datetime.datetime(2026, 12, 2, 12, 0, 0)


def _row(sec, sm, reasons=()):
    ts = (T0 + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if nm in reasons else "Not Active" for nm in bench.CLOCK_REASONS]
    return ", ".join([ts, "0", str(sm), "2070", "900.5", "0x0000000000000000"] + flags)


def _t(sec):
    return (T0 + datetime.timedelta(seconds=sec)).timestamp()


def test_only_samples_inside_the_window_count():
    lines = [_row(0.00, 1200), _row(0.05, 1300), _row(0.30, 2070), _row(0.35, 2040, ["sw_power_cap"]),
             _row(0.40, 2060), _row(0.70, 900, ["hw_slowdown"])]
    s = bench.summarise_clocks(lines, _t(0.28), _t(0.45))
    assert s == {"sm_mhz": 2060.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3, "in_window": True}


def test_falls_back_to_every_sample_when_none_is_inside():
    lines = [_row(0.0, 2000), _row(1.0, 2070, ["hw_thermal_slowdown"])]
    s = bench.summarise_clocks(lines, _t(0.4), _t(0.5))
    assert s["samples"] == 2 and not s["in_window"] and s["reasons"] == ["hw_thermal_slowdown"]
    assert s["sm_mhz"] == 2035.0


def test_unreadable_timestamps_and_short_rows():
    lines = ["not a time, 0, 1800, 2070, 800, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage", ""]
    s = bench.summarise_clocks(lines, _t(0.0), _t(1.0))
    assert s["samples"] == 1 and not s["in_window"] and s["sm_mhz"] == 1800.0
    assert bench.summarise_clocks(["garbage"]) is None


def test_launch_count_names_and_fallback():
    names = ["void (anonymous namespace)::index_scores_kernel<64, 128, 64>(IdxArgs, CUtensorMap_st)",
             "void (anonymous namespace)::topk_kernel<true>(int, float const*)", "Memset (Device)",
             "void (anonymous namespace)::attend_kernel<9, true, false>(AttnArgs)",
             "void smla::kvpack_store_kernel<16>(KernelLayout)", "void at::native::vectorized_elementwise_kernel"]
    assert bench.count_lib_kernels(names) == 4
    # no CUDA here: the profiler count gives 0 and the bench falls back to its formula
    assert bench.count_step_launches(lambda: None) == 0


def test_launch_count_must_fit_the_schedule():
    assert bench.plausible_launches(4, 1) == (4, "profiled one step")
    assert bench.plausible_launches(6, 1)[0] == 6                 # split top-k and split attention
    assert bench.plausible_launches(0, 1)[0] == 4                 # no profiler: the formula
    n, how = bench.plausible_launches(8, 1)                       # e.g. counted twice: not taken
    assert n == 4 and "outside" in how
    assert bench.plausible_launches(10, 3)[0] == 10
