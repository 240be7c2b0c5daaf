"""GPU parity of the degenerate cases the method has, through K4 (the fused
update pass and the filter-only call) against the oracle.

StreamDiffusion notes, "Stochastic Similarity Filter": identical frames have
cosine 1, so the skip probability max(0, (1 - eta)/(1 - eta)) is exactly 1
and every draw u < 1 skips -- until the overview page's max_skip_frame cap
forces a frame through.  StreamDiffusionV2 summary, "Motion-aware noise
scheduler": frames that do not move have zero motion, so the noise rate is
pulled to (and held at) its lower bound s_min.

Both results are exact on the GPU, not merely close: K4 forms dot, |I|^2 and
|R|^2 with one operation sequence, so identical frames give three bitwise
equal sums, cosine 1.0 and P 1.0; zero frame differences sum to exactly 0,
and the EMA s + (1 - lambda)(s_min - s) leaves s_min unchanged.
"""
import numpy as np
import pytest

from oracle import oracle as O
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import GpuPipe, OraclePipe, tensor_rel_err

pytestmark = pytest.mark.gpu

UPD_TOL = 1e-5


def _u_series(steps: int) -> np.ndarray:
    """Draws in [0, 1) including both ends' extremes."""
    top = np.float32(np.nextafter(np.float32(1.0), np.float32(0.0)))
    base = np.array([0.0, 0.5, top, 0.25, 0.999, 0.0, top, 0.75], dtype=np.float32)
    return np.resize(base, steps)


@pytest.mark.parametrize("fused", [False, True])
def test_identical_frames_skip_with_probability_one_until_the_cap(fused):
    """A stream of one repeated frame: the first is processed (no reference
    yet), then cos == 1.0 and P == 1.0 exactly, and skips run in groups of
    max_skip_frame followed by one forced frame: 0, 1,1,1, 0, 1,1,1, 0, ..."""
    max_skip = 3
    w = W.get_config("c1_tiny", streams=2, max_skip=max_skip)
    g, o = GpuPipe(w), OraclePipe(w)
    frame = W.FrameWalk(w).next()  # [S][E], one frame per stream, repeated
    us = _u_series(14)
    expect = [0] + [1, 1, 1, 0] * 4
    try:
        for step in range(14):
            u = np.full(w["streams"], us[step], dtype=np.float32)
            if fused:
                lat = W.gen_latents(w, step)
                xn, out = g.step(lat, frame, u, None)
                (xr, outr), _ = o.step(lat)
                assert tensor_rel_err(out[0], outr) <= UPD_TOL
            else:
                g.ssf(frame, u)
            st = g.state()
            ref = o.ssf(frame, u)
            for s in range(w["streams"]):
                assert st[s]["ssf_skip"] == ref[s]["skip"] == expect[step], (step, s)
                assert st[s]["ssf_skip_count"] == ref[s]["skip_count"]
                if step > 0:
                    assert st[s]["ssf_cos"] == 1.0 and ref[s]["cos"] == 1.0, (step, s, st[s]["ssf_cos"])
                    assert st[s]["ssf_p"] == 1.0 and ref[s]["p"] == 1.0, (step, s, st[s]["ssf_p"])
                assert st[s]["error_word"] == 0
        assert g.state()[0]["ssf_evals"] == 14
    finally:
        g.close()


def test_zero_skip_cap_processes_every_frame():
    """max_skip_frame = 0: P is still 1, but no frame may be skipped."""
    w = W.get_config("c1_tiny", max_skip=0)
    g, o = GpuPipe(w), OraclePipe(w)
    frame = W.FrameWalk(w).next()
    try:
        for step in range(4):
            u = np.zeros(1, dtype=np.float32)
            g.ssf(frame, u)
            st, ref = g.state()[0], o.ssf(frame, u)[0]
            assert st["ssf_skip"] == ref["skip"] == 0
            if step > 0:
                assert st["ssf_p"] == ref["p"] == 1.0
    finally:
        g.close()


@pytest.mark.parametrize("T,rate_on", [(1, 0), (3, 1)])
def test_identical_motion_frames_hold_the_noise_rate_at_s_min(T, rate_on):
    """Chunks whose frames never change: every pair's motion is exactly 0,
    dhat is 0, and the noise rate stays exactly s_min (with the rate applied,
    the incoming frame enters at the timestep of rate s_min every step)."""
    w = W.get_config("c1_tiny", T=T, R=max(4, T), mot_k=T, noise_rate_on=rate_on, streams=2)
    g, o = GpuPipe(w), OraclePipe(w)
    still = W.LatentWalk(w).next()[:, :1, :]              # [S][1][N_f]
    chunk = np.ascontiguousarray(np.repeat(still, T, axis=1))
    t1 = O.slot_timestep(w, 1)  # the entry runs from slot 1's timestep (rate 0) to N - 1 (rate 1)
    t_entry = t1 + int(np.floor(w["s_min"] * (w["n_train"] - 1 - t1) + 0.5))
    try:
        for step in range(5):
            lat = W.gen_latents(w, step)
            xn, out = g.step(lat, None, None, chunk)
            ores = o.step(lat)
            om = o.motion(chunk)
            st = g.state()
            for s in range(w["streams"]):
                xr, outr = ores[s]
                assert tensor_rel_err(out[s], outr) <= UPD_TOL
                for i in range(w["n"]):
                    assert tensor_rel_err(xn[i, s], xr[i]) <= UPD_TOL
                d = np.array(st[s]["motion_d"][:T])
                first = 1 if step == 0 else 0  # no previous frame before the first chunk
                assert np.all(np.isnan(d[:first])) and np.all(d[first:] == 0.0), (step, s, d)
                assert np.array_equal(np.nan_to_num(d, nan=-1.0), np.nan_to_num(om[s]["d"], nan=-1.0))
                if step > 0 or T > 1:
                    assert st[s]["motion_dhat"] == 0.0 and om[s]["dhat"] == 0.0
                assert st[s]["noise_rate"] == w["s_min"] and om[s]["s"] == w["s_min"], (step, s)
                if rate_on:
                    assert st[s]["slot0_timestep"] == t_entry == o.s[s].slot0_timestep()
                assert st[s]["error_word"] == 0
    finally:
        g.close()


def test_motion_after_a_burst_decays_back_toward_s_min_when_frames_stop():
    """A moving chunk raises s; then still frames pull it back by the EMA,
    s_k = s_min + lambda^k (s_0 - s_min), on both sides."""
    w = W.get_config("c1_tiny", lat_step=0.5)
    g, o = GpuPipe(w), OraclePipe(w)
    walk = W.LatentWalk(w)
    try:
        moving = walk.next()
        moving2 = walk.next()
        for step, chunk in enumerate([moving, moving2] + [moving2[:, -1:, :].copy()] * 4):
            chunk = np.ascontiguousarray(chunk)
            lat = W.gen_latents(w, step)
            g.step(lat, None, None, chunk)
            o.step(lat)
            om = o.motion(chunk)[0]
            st = g.state()[0]
            assert abs(st["noise_rate"] - om["s"]) <= 1e-5, (step, st["noise_rate"], om["s"])
            if step == 1:
                s_peak = om["s"]
                assert s_peak > w["s_min"] + 0.01
            if step >= 2:
                k = step - 1
                closed = w["s_min"] + w["lam"] ** k * (s_peak - w["s_min"])
                assert abs(om["s"] - closed) <= 1e-12
                assert np.all(np.array(st["motion_d"][:1]) == 0.0)
    finally:
        g.close()
