"""GPU parity of the whole per-step path (K2 push, K3 sink refresh, K1
attend, K4 fused update + SSF + motion) against the oracle, over seeded
multi-chunk sequences.

Bars: ring indices, RoPE positions, sink choices and skip decisions
bit-exact (a decision the oracle flags as a near tie may go either way);
ring V bit-exact, ring K within max(1 bf16 ulp, 2^-20 * pair norm) (fp32 vs
double rotation: near-zero results carry the fp32 error of the pair);
attention within 2e-2 of the block max; the fp32 latent update within 1e-5
of the tensor max; cosines within 1e-6; motion and noise rate within 1e-5.
"""
import numpy as np
import pytest

from oracle import oracle as O
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import (GpuPipe, OraclePipe, attn_rel_err, rope_k_excess, tensor_rel_err)

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-2
UPD_TOL = 1e-5


def sample_rows(nrows: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    edge = [0, 1, 127, 128, nrows // 2, nrows - 129, nrows - 128, nrows - 2, nrows - 1]
    pick = rng.choice(nrows, size=min(k, nrows), replace=False)
    rows = np.unique(np.clip(np.concatenate([edge, pick]), 0, nrows - 1))
    return rows.astype(np.int64)


def run_sequence(w: dict, steps: int, rows_per_step=None, attend_every=1, check_kv_every=1,
                 ssf=None, motion=None):
    """Run `steps` chunks through both paths and compare everything each step."""
    ssf = w["ssf"] if ssf is None else ssf
    motion = w["motion"] if motion is None else motion
    S = w["streams"]
    g, o = GpuPipe(w), OraclePipe(w)
    emb, lat_walk, frames = W.EmbeddingWalk(w), W.LatentWalk(w), W.FrameWalk(w)
    ssf_live = [True] * S
    rate_live = [True] * S  # False once a flagged near tie of the entry timestep went the other way
    stats = dict(sink_fires=0, resets=0, skips=0, near=0, dropped=0)
    try:
        for step in range(steps):
            k, v = W.gen_kv(w, step)
            g.push(k, v)
            o.push(k, v)
            m, om = g.meta(), o.s[0].meta()
            assert (m["frames_pushed"], m["rope_offset"], m["chunk_p0"], m["ring_valid"]) == \
                (om["F"], om["o"], om["p0"], om["valid"]), step
            h = emb.next()
            g.refresh(h)
            ores = o.refresh(h)
            st = g.state()
            assert g.meta()["sinks_filled"] == o.s[0].meta()["sinks_filled"]
            for s in range(S):
                r = ores[s]
                if r["near"]:
                    stats["near"] += 1
                    continue
                if r["fire"] == 0 and r["j"] < 0:
                    continue
                assert st[s]["sink_fire"] == r["fire"], (step, s, st[s], r)
                assert st[s]["sink_j"] == r["j"], (step, s)
                if r["fire"] == 1:
                    stats["sink_fires"] += 1
                if r["fire"] != 2:
                    assert abs(st[s]["sink_alpha_min"] - r["alpha_min"]) < 1e-12
            if step % check_kv_every == 0 or step == steps - 1:
                gk, gv = g.kv()
                for s in range(S):
                    ok, ov = o.s[s].kv()
                    assert np.array_equal(gv[s], ov), (step, s)
                    assert rope_k_excess(gk[s], ok) <= 1.0, (step, s)
                if w["M"] > 0:
                    ge = g.sink_emb()
                    for s in range(S):
                        filled = o.s[s].meta()["sinks_filled"]
                        assert np.array_equal(ge[s][:filled].astype(np.float64), o.s[s].emb()[:filled])
            if step % attend_every == 0 or step == steps - 1:
                q = W.gen_q(w, step)
                got = g.attend(q)
                rows = None if rows_per_step is None else sample_rows(w["q_rows"], rows_per_step, step)
                refs = o.attend(q, rows)
                for s in range(S):
                    gs = got[s] if rows is None else got[s][rows]
                    err = attn_rel_err(gs, refs[s])
                    assert err <= ATTN_TOL, (step, s, err)
            lat = W.gen_latents(w, step)
            frame = frames.next() if ssf else None
            u = W.gen_u(w, step) if ssf else None
            chunk = lat_walk.next() if motion else None
            # the entry timestep t1 + round(s (N - 1 - t1)) is decided from an
            # s that the two sides agree on to ~1e-8: flag near half-integers
            rate_near = [False] * S
            if w.get("noise_rate_on"):
                t1 = O.slot_timestep(w, 1) if w["n"] > 1 else 0
                for s in range(S):
                    xe = o.s[s].noise_rate() * (w["n_train"] - 1 - t1) + 0.5
                    rate_near[s] = abs(xe - round(xe)) < 1e-4
            xn, out = g.step(lat, frame, u, chunk)
            ores = o.step(lat)
            st = g.state()
            if w.get("noise_rate_on"):
                for s in range(S):
                    if rate_live[s] and st[s]["slot0_timestep"] != o.s[s].slot0_timestep():
                        assert rate_near[s], (step, s)
                        rate_live[s] = False  # slot 0 now differs; stop comparing this stream
                        stats["near"] += 1
                        stats["dropped"] += 1
            for s in range(S):
                if not rate_live[s]:
                    continue
                xr, outr = ores[s]
                assert tensor_rel_err(out[s], outr) <= UPD_TOL, (step, s)
                for i in range(w["n"]):
                    assert tensor_rel_err(xn[i, s], xr[i]) <= UPD_TOL, (step, s, i)
            if ssf:
                oss = o.ssf(frame, u)
                for s in range(S):
                    if not ssf_live[s]:
                        continue
                    assert abs(st[s]["ssf_cos"] - oss[s]["cos"]) <= 1e-6, (step, s)
                    assert abs(st[s]["ssf_p"] - oss[s]["p"]) <= 5e-5, (step, s)
                    if oss[s]["near"] and st[s]["ssf_skip"] != oss[s]["skip"]:
                        ssf_live[s] = False  # a flagged near tie went the other way
                        stats["near"] += 1
                        stats["dropped"] += 1
                        continue
                    assert st[s]["ssf_skip"] == oss[s]["skip"], (step, s, st[s], oss[s])
                    assert st[s]["ssf_skip_count"] == oss[s]["skip_count"]
                    stats["skips"] += oss[s]["skip"]
            if motion:
                om_ = o.motion(chunk)
                for s in range(S):
                    dref = om_[s]["d"]
                    dg = np.array(st[s]["motion_d"][:w["T"]])
                    assert np.array_equal(np.isnan(dg), np.isnan(dref)), (step, s)
                    ok_ = ~np.isnan(dref)
                    assert np.all(np.abs(dg[ok_] - dref[ok_]) <= 1e-5 * np.maximum(1.0, dref[ok_]))
                    assert abs(st[s]["noise_rate"] - om_[s]["s"]) <= 1e-5, (step, s)
            for s in range(S):
                assert st[s]["error_word"] == 0
        stats["resets"] = o.s[0].meta()["resets"]
        assert g.meta()["rope_resets"] == stats["resets"]
        # a flagged near tie that went the other way stops one stream's
        # comparisons; more than one in a short sequence would hide a bug
        assert stats["dropped"] <= 1, stats
        return stats
    finally:
        g.close()


def test_c1_tiny_sequence_all_rows():
    w = W.get_config("c1_tiny")
    stats = run_sequence(w, w["steps"])
    assert stats["sink_fires"] >= 1  # the embedding walk of c1 crosses s_th within 8 chunks
    assert stats["skips"] >= 1       # the filter skipped, and agreed on it, at least once


def test_c1_two_streams():
    w = W.get_config("c1_tiny", streams=2, steps=6)
    run_sequence(w, 6)


def test_c1_split_key_schedule_with_sink_fill():
    """Video mode on the persistent split schedule (keys of each query tile
    split between CTAs), through sink fill, refresh and ring wrap."""
    w = W.get_config("c1_tiny", M=2, T=3, R=6, mot_k=3, emb_step=0.5, attn_ctas=5)
    run_sequence(w, 6)


def test_c1_d128_split_key_schedule_with_sink_fill():
    """The same at head_dim 128 (64-key compute tiles, one MMA issuer per
    query tile) on the persistent split schedule."""
    w = W.get_config("c1_tiny", d=128, M=2, T=3, R=6, mot_k=3, emb_step=0.5, attn_ctas=5)
    run_sequence(w, 6)


@pytest.mark.parametrize("cfg_type,update_kind,n", [(2, 0, 2), (2, 1, 4), (1, 1, 3), (0, 1, 2)])
def test_guidance_and_update_variants(cfg_type, update_kind, n):
    """Onetime-negative R-CFG (supplied negative prediction), the strided DDPM
    posterior update and their combinations against the oracle."""
    t_index = [0, 16, 32, 45][:n] if n > 2 else [32, 45]
    w = W.get_config("c1_tiny", cfg_type=cfg_type, update_kind=update_kind, n=n,
                     t_index=t_index, steps=4)
    run_sequence(w, 4)


@pytest.mark.parametrize("update_kind,streams", [(0, 1), (1, 2)])
def test_noise_rate_sets_the_incoming_frames_timestep(update_kind, streams):
    """The motion-aware noise rate chooses the timestep at which each
    stream's incoming frame enters slot 0 (bursts move the rate around)."""
    w = W.get_config("c1_tiny", noise_rate_on=1, update_kind=update_kind, streams=streams,
                     burst_prob=0.4, lat_step=0.3, steps=8)
    run_sequence(w, 8)


@pytest.mark.parametrize("cfg_type,update_kind", [(1, 0), (2, 1)])
def test_bf16_noise_predictions(cfg_type, update_kind):
    """eps_c handed over as bf16 (the network's usual output dtype): the
    update widens it exactly, so it matches the oracle fed the same values."""
    t_index = [0, 16, 32, 45] if update_kind == 1 else [32, 45]
    w = W.get_config("c1_tiny", eps_c_bf16=1, cfg_type=cfg_type, update_kind=update_kind,
                     n=len(t_index), t_index=t_index, steps=4)
    run_sequence(w, 4)


@pytest.mark.parametrize("cfg_type,bf16", [(0, 0), (2, 1)])
def test_txt2img_incoming_frame_is_the_noise_draw(cfg_type, bf16):
    """txt2img: no input image, so the incoming latent is eps_new itself
    (x0_new is passed as NULL); everything else as in img2img."""
    w = W.get_config("c1_tiny", txt2img=1, cfg_type=cfg_type, eps_c_bf16=bf16, steps=4)
    g = GpuPipe(w)
    try:
        lat = W.gen_latents(w, 0)
        xn, _ = g.step(lat, None, None, W.LatentWalk(w).next())
        assert np.array_equal(xn[0], lat["eps_new"])  # bit-exact copy of the draw
    finally:
        g.close()
    run_sequence(w, 4)


def test_c3_full_size_with_noise_rate_application():
    w = W.get_config("c3_dit1p3b_video", noise_rate_on=1, burst_prob=0.5)
    run_sequence(w, 4, rows_per_step=8, attend_every=3)


def test_c4_full_size_ddpm_update_with_supplied_negative():
    w = W.get_config("c4_dit14b_video", cfg_type=2, update_kind=1)
    run_sequence(w, 2, rows_per_step=8, attend_every=2, check_kv_every=2)


def test_rope_reset_fires_with_small_tau():
    w = W.get_config("c1_tiny", rope_tau=3, steps=11)
    stats = run_sequence(w, 11)
    assert stats["resets"] == 2  # p0: 0 1 2 3 | 0 1 2 3 | 0 1 2


def test_multi_sink_fill_and_refresh_with_chunks_of_three():
    w = W.get_config("c1_tiny", M=2, T=3, R=6, mot_k=3, emb_step=0.5, latent_h=4, latent_w=4)
    run_sequence(w, 7)


def test_c3_full_size_sampled_rows():
    w = W.get_config("c3_dit1p3b_video")
    run_sequence(w, 4, rows_per_step=40, attend_every=3)


def test_c4_full_size_sampled_rows():
    w = W.get_config("c4_dit14b_video")
    run_sequence(w, 5, rows_per_step=16, attend_every=4, check_kv_every=4)


def test_c2_image_stream_update_and_ssf():
    """Image batch mode at full size: fused update + SSF over 12 frames.
    The update is compared on every frame; a skip decision the oracle flags
    as a near tie (|u - P| < 1e-4) is not asserted, and if it went the other
    way the reference frames differ from then on, so the filter's later
    decisions are no longer compared (at most one such frame is allowed)."""
    w = W.get_config("c2_sdturbo_image")
    g, o = GpuPipe(w), OraclePipe(w)
    frames = W.FrameWalk(w)
    ssf_live, diverged, skips = True, 0, 0
    try:
        for step in range(12):
            lat = W.gen_latents(w, step)
            frame, u = frames.next(), W.gen_u(w, step)
            xn, out = g.step(lat, frame, u)
            (xr, outr), = o.step(lat)
            assert tensor_rel_err(out[0], outr) <= UPD_TOL, step
            for i in range(w["n"]):
                assert tensor_rel_err(xn[i, 0], xr[i]) <= UPD_TOL, (step, i)
            st = g.state()[0]
            ref = o.ssf(frame, u)[0]
            if not ssf_live:
                continue
            assert abs(st["ssf_cos"] - ref["cos"]) <= 1e-6, step
            assert abs(st["ssf_p"] - ref["p"]) <= 5e-5, step
            if ref["near"] and st["ssf_skip"] != ref["skip"]:
                ssf_live = False
                diverged += 1
                continue
            assert st["ssf_skip"] == ref["skip"] and st["ssf_skip_count"] == ref["skip_count"], step
            skips += ref["skip"]
        assert diverged <= 1
        assert skips >= 1  # the oracle skips 6 of these 12 frames
    finally:
        g.close()


def test_c5_stress_three_streams_with_bursts():
    """Long-run shape with 3 concurrent streams: refreshes and bursts; K/V
    compared every 10 chunks, attention sampled at the end."""
    w = W.get_config("c5_stress", streams=3, burst_prob=0.2, emb_step=0.4)
    stats = run_sequence(w, 30, rows_per_step=12, attend_every=29, check_kv_every=10)
    assert stats["sink_fires"] >= 1
