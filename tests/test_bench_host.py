"""CPU: the bench's clock record and its work accounting, on synthetic input.

The clock record is what decides whether a timed region ran at full clocks: samples are kept by
their timestamps inside the timed region (or, when none landed there, within one sampling period
of it), the throttle reasons seen there are reported, and the SM clock is the median of the kept
samples.  The flop count is the window-effective one (visible pairs only, 4 D per pair forward,
10 D backward); the fused dK/dV/dQ split of the backward must add up to it.
"""
import datetime

import pytest

import bench
import swa_inputs as si


def _line(t: datetime.datetime, sm: float, reasons=()):
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    stamp = t.strftime("%Y/%m/%d %H:%M:%S.") + f"{t.microsecond // 1000:03d}"
    return ", ".join([stamp, "0", f"{sm:.0f}", "2070", "950.00", "0x0"] + flags)


def _sampler(lines, window=None):
    s = bench.ClockSampler(0)
    s.lines = lines
    if window is not None:
        s.mark(*window)
    return s


def test_smi_time_parses_and_rejects():
    t = datetime.datetime(2026, 12, 2, 10, 0, 0, 250000)
    assert bench._smi_time(t.strftime("%Y/%m/%d %H:%M:%S.250")) == pytest.approx(t.timestamp())
    assert bench._smi_time("not a time") is None


def test_clock_summary_keeps_samples_inside_the_window():
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0)
    step = datetime.timedelta(milliseconds=10)
    # before the region: a throttled, slow sample; inside: three at full clocks (one power-capped)
    lines = [_line(t0, 1200, {"hw_slowdown"})]
    lines += [_line(t0 + (i + 10) * step, sm, r)
              for i, (sm, r) in enumerate([(2070, ()), (2055, {"sw_power_cap"}), (2070, ())])]
    window = ((t0 + 9 * step).timestamp(), (t0 + 13 * step).timestamp())
    s = _sampler(lines, window).summary()
    assert s["selection"] == "inside the timed region"
    assert s["samples"] == 3 and s["samples_total"] == 4
    assert s["sm_mhz"] == 2070 and s["sm_mhz_min"] == 2055 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside the region


def test_clock_summary_falls_back_to_samples_next_to_a_short_window():
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(t0, 2070), _line(t0 + 40 * ms, 1900, {"hw_thermal_slowdown"})]
    # a 3 ms region 5 ms after the first sample: nothing inside, the first sample is near it
    window = ((t0 + 5 * ms).timestamp(), (t0 + 8 * ms).timestamp())
    s = _sampler(lines, window).summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2070 and s["reasons"] == []
    assert s["selection"].startswith("within")


def test_clock_summary_without_samples_says_so():
    s = _sampler([]).summary()
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"] and s["sm_mhz"] is None
    # malformed lines are skipped, not misread
    assert _sampler(["garbage", "a, b, c"]).summary()["samples"] == 0


def test_step_flops_split_adds_up():
    case = si.long_swa_case(32768)
    fl = bench.step_flops(case)
    assert fl["pairs"] == bench.visible_pairs(case.N, case.W) * case.B * case.Hq
    assert fl["fwd"] == 4 * case.D * fl["pairs"]
    assert fl["bwd"] == 10 * case.D * fl["pairs"]
    assert fl["dkdv"] + fl["dq"] == fl["bwd"]
    cfg = bench.headline_config(case, 1)
    assert cfg["flops_per_step"] == {"fwd": fl["fwd"], "bwd": fl["bwd"]}
    assert cfg["seq_len"] == case.N and cfg["global_batch"] == case.B
