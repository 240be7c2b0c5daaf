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


def test_workload_flags_and_update_bytes():
    """The K4 roofline numerator: every operand read once, every result
    written once (4 B fp32, 2 B for bf16 predictions, no x0_new in txt2img)."""
    import argparse
    base = dict(workload="c2_sdturbo_image", streams=None, cfg_type=None, update_kind=None,
                noise_rate_on=False, eps_c_bf16=False, txt2img=False)
    w = bench.workload(argparse.Namespace(**base))
    n, N = w["n"], w["N_s"]
    # x, x0 (virtual negative), eps_c, x_next per slot; z for n-1; out; x0_new, eps_new
    assert bench.step_bytes(w, False, False) == 4.0 * N * (4 * n + (n - 1) + 1 + 2)
    wb = bench.workload(argparse.Namespace(**dict(base, eps_c_bf16=True)))
    assert bench.step_bytes(wb, False, False) == bench.step_bytes(w, False, False) - 2.0 * N * n
    wt = bench.workload(argparse.Namespace(**dict(base, txt2img=True)))
    assert wt["txt2img"] == 1 and wt["cfg_type"] == 0  # no x0, so no self-negative guidance
    # without guidance there is no negative operand: 4 arrays per slot
    assert bench.step_bytes(wt, False, False) == 4.0 * N * (3 * n + (n - 1) + 1 + 1)
    assert bench.step_bytes(w, True, False) - bench.step_bytes(w, False, False) == 12.0 * w["ssf_E"]
