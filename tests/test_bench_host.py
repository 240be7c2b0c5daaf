"""Host-side pieces of bench.py that need no GPU: the clock sampler's
parsing of nvidia-smi's CSV (reasons, the timed-region window, the nearest
poll when the region is shorter than the poll interval)."""
import datetime as dt

import bench


def _sampler(tmp_path, lines):
    s = object.__new__(bench.ClockSampler)
    s.path = str(tmp_path / "clocks.csv")
    s.proc = object()  # stands in for the nvidia-smi process
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def _row(t, mhz, hw="Not Active", cap="Not Active"):
    ts = dt.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, {mhz}, 2032, 0x0000000000000000, {hw}, Not Active, Not Active, {cap}"


def test_samples_inside_the_timed_region_and_reasons(tmp_path):
    t0 = 1_800_000_000.0
    s = _sampler(tmp_path, [_row(t0 - 1.0, 900), _row(t0 + 0.1, 2032), _row(t0 + 0.3, 1990, cap="Active"),
                            _row(t0 + 0.5, 2032), _row(t0 + 2.0, 800, hw="Active")])
    r = s.summary(t0, t0 + 0.6)
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2032.0 and r["sm_max_mhz"] == 2032.0
    assert r["reasons"] == ["sw_power_cap"]  # the hw_slowdown poll lies outside the region


def test_region_shorter_than_a_poll_uses_the_nearest_poll(tmp_path):
    t0 = 1_800_000_000.0
    s = _sampler(tmp_path, [_row(t0 - 0.5, 1500), _row(t0 + 0.45, 2032)])
    r = s.summary(t0 + 0.2, t0 + 0.3)
    assert r["samples"] == 0 and r["sm_mhz"] == 2032.0


def test_malformed_lines_are_skipped(tmp_path):
    t0 = 1_800_000_000.0
    s = _sampler(tmp_path, ["garbage", "a, b, c", _row(t0, 2032)])
    assert s.summary(t0 - 0.1, t0 + 0.1)["samples"] == 1
