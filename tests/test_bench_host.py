"""Host-side logic of the benchmark (no GPU): the clock summary keeps the
samples taken in and just before the timed region and decodes the
clock-event reasons; whole-job throughput divides all ranks' units by the
slowest rank's time."""
import bench


def _sampler(samples):
    c = bench.ClockSampler(0)
    c.samples = list(samples)
    return c


def test_clock_summary_window_and_reasons():
    # (host time s, sm MHz, max MHz, reason mask): idle before the lead-in, under load after
    c = _sampler([(0.0, 345.0, 2070.0, 0x1), (9.6, 2055.0, 2070.0, 0x0), (9.8, 2070.0, 2070.0, 0x4),
                  (10.05, 1980.0, 2070.0, 0x4), (10.3, 2070.0, 2070.0, 0x0), (12.0, 600.0, 2070.0, 0x8)])
    # timed region [10.0, 10.1] after a 0.5 s lead-in; the window is [9.5, 10.25]
    s = c.summary(10.0, 10.1, 0.5)
    assert s["samples"] == 3 and s["samples_in_timed_region"] == 1
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]  # gpu_idle and the later hw_slowdown are outside


def test_clock_summary_throttle_and_unsampled():
    c = _sampler([(1.0, 1500.0, 2070.0, 0x8 | 0x40)])
    assert set(c.summary(1.0, 1.05, 0.5)["reasons"]) == {"hw_slowdown", "sw_thermal_slowdown"}
    assert _sampler([]).summary(0.0, 1.0, 0.5)["reasons"] == ["unsampled"]


def test_job_throughput_single_rank():
    v, ms = bench.job_throughput(2.0e12, 4.0, 1)
    assert ms == 4.0 and abs(v - 5.0e14) < 1.0
