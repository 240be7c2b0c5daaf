"""The SLO-aware stream-batch controller (host code, no device).

The oracle's fit is pinned to closed forms (exact recovery of an affine
latency law, the equal-weight least-squares line), and the library's
controller is checked against the oracle on noisy observations, through
exploration, the SLO boundary and the knee cap."""
import numpy as np
import pytest

from oracle import slo_oracle as SO
from streaming_diffusion_stream_b300 import binding as B


def test_oracle_fit_recovers_an_exact_affine_law():
    T, a, b = 3, 2.0e-3, 1.7e-4
    obs = [(B_, a + b * B_ * T) for B_ in (1, 2, 5, 8, 3)]
    fa, fb = SO.fit(obs, T, 0.9)
    assert abs(fa - a) < 1e-15 and abs(fb - b) < 1e-16


def test_oracle_fit_equal_weights_is_the_textbook_line():
    rng = np.random.default_rng(0)
    T = 2
    obs = [(int(B_), float(0.01 + 0.002 * B_ * T + rng.normal(0, 1e-4))) for B_ in rng.integers(1, 9, 20)]
    x = np.array([B_ * T for B_, _ in obs], float)
    y = np.array([L for _, L in obs])
    b_ref = np.sum((x - x.mean()) * (y - y.mean())) / np.sum((x - x.mean()) ** 2)
    a_ref = y.mean() - b_ref * x.mean()
    fa, fb = SO.fit(obs, T, 1.0)
    assert abs(fa - a_ref) < 1e-12 and abs(fb - b_ref) < 1e-12


def test_oracle_choice_meets_slo_and_stops_at_the_knee():
    T = 3
    # memory-bound law: fixed part dominates, so throughput keeps growing
    obs = [(1, 0.010 + 0.0002 * 3), (4, 0.010 + 0.0002 * 12)]
    r = SO.choose(obs, target_fps=200.0, T=T, b_min=1, b_max=8, knee_gain=0.0)
    lat = lambda B_: 0.010 + 0.0002 * B_ * T
    assert r["b_slo"] == max(B_ for B_ in range(1, 9) if T / lat(B_) >= 200.0)
    assert r["batch"] == r["b_slo"] and r["meets_slo"] == 1
    # compute-bound law (latency proportional to B): flat throughput, knee at b_min
    obs = [(1, 0.0005 * 3), (4, 0.0005 * 12)]
    r = SO.choose(obs, target_fps=30.0, T=T, b_min=1, b_max=8, knee_gain=0.05)
    assert r["b_knee"] == 1 and r["batch"] == 1
    # an unreachable target: the smallest batch, flagged
    r = SO.choose(obs, target_fps=1e6, T=T, b_min=2, b_max=8)
    assert r["b_slo"] == 0 and r["batch"] == 2 and r["meets_slo"] == 0


@pytest.mark.parametrize("forget,knee,fps", [(1.0, 0.05, 150.0), (0.8, 0.02, 60.0), (0.95, 0.0, 400.0)])
def test_library_controller_matches_the_oracle(forget, knee, fps):
    rng = np.random.default_rng(int(fps))
    T, b_min, b_max = 3, 1, 8
    ctl = B.SloController(fps, T, b_min, b_max, forget=forget, knee_gain=knee)
    obs = []
    try:
        for it in range(40):
            got = ctl.choose()
            ref = SO.choose(obs, fps, T, b_min, b_max, forget, knee)
            assert got["batch"] == ref["batch"] and got["exploring"] == ref["exploring"], (it, got, ref)
            if not ref["exploring"]:
                assert got["b_slo"] == ref["b_slo"] and got["b_knee"] == ref["b_knee"]
                assert got["meets_slo"] == ref["meets_slo"]
                assert abs(got["a"] - ref["a"]) <= 1e-9 * max(1.0, abs(ref["a"]))
                assert abs(got["b"] - ref["b"]) <= 1e-9 * max(1e-6, abs(ref["b"]))
                assert abs(got["total_fps"] - ref["total_fps"]) <= 1e-9 * ref["total_fps"]
            Bb = got["batch"]
            lat = 0.004 + 0.0011 * Bb * T + rng.normal(0, 2e-5)
            ctl.observe(Bb, lat)
            obs.append((Bb, lat))
            if it % 7 == 3:  # the serving loop also sees other batch sizes
                Bo = int(rng.integers(b_min, b_max + 1))
                lo = 0.004 + 0.0011 * Bo * T + rng.normal(0, 2e-5)
                ctl.observe(Bo, lo)
                obs.append((Bo, lo))
    finally:
        ctl.close()


def test_invalid_controller_configs_are_rejected():
    for bad in (dict(target_fps=0.0), dict(forget=0.0), dict(knee_gain=1.0), dict(b_min=0),
                dict(b_min=5, b_max=4)):
        kw = dict(target_fps=30.0, frames_T=3, b_min=1, b_max=8, forget=1.0, knee_gain=0.05)
        kw.update(bad)
        with pytest.raises(B.SdsError):
            B.SloController(kw["target_fps"], kw["frames_T"], kw["b_min"], kw["b_max"],
                            forget=kw["forget"], knee_gain=kw["knee_gain"])
