"""Write the oracle-regression fixtures of tests/golden/ (oracle/ only).

    python tests/golden/make_golden.py

Every value here comes from oracle/ on fixed small inputs; the fixtures pin
the oracle against unnoticed changes of its arithmetic (tests/test_golden.py
recomputes them).  A change to a fixture must come with the passage, or the
reading of it, that justifies the oracle change.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import oracle as O  # noqa: E402
from streaming_diffusion_stream_b300 import workloads as W  # noqa: E402


def compute() -> dict:
    w = W.get_config("c1_tiny")
    out = {}
    ab = O.alpha_bar(w)
    out["alpha_bar_at"] = {str(t): float(ab[t]) for t in (0, 99, 359, 679, 999)}
    out["rope_angle"] = {f"{wd}:{pr}:{pos}": O.rope_angle(10000.0, wd, pr, pos)
                         for wd, pr, pos in ((44, 0, 7), (44, 21, 1000), (42, 20, 51), (20, 9, 3))}
    # tiny attention: 3 queries x 4 keys x 1 head x d 64, values in bf16
    rng = np.random.default_rng(11)
    bits = lambda sh: W.to_bf16_bits(rng.standard_normal(sh).astype(np.float32))
    q, k, v = bits((3, 1, 64)), bits((4, 1, 64)), bits((4, 1, 64))
    out["attention_inputs"] = {"q": q.tolist(), "k": k.tolist(), "v": v.tolist()}
    out["attention"] = O.attention(q, k, v).reshape(3, 64)[:, :8].tolist()
    # one R-CFG + update step of c1 (first 6 elements of each output)
    st = O.Stream(w)
    lat = W.gen_latents(w, 0)
    xn, o = st.step_update(lat["x"][:, 0], lat["x0"][:, 0], lat["eps_c"][:, 0], lat["z"][:, 0],
                           lat["x0_new"][0], lat["eps_new"][0])
    out["step_update_x_next"] = xn[:, :6].tolist()
    out["step_update_out"] = o[:6].tolist()
    # SSF decisions and the noise rate over a short walk
    fw, lw = W.FrameWalk(w), W.LatentWalk(w)
    ssf, mot = [], []
    for t in range(6):
        r = st.ssf(fw.next()[0], float(W.gen_u(w, t)[0]))
        ssf.append([r["skip"], r["skip_count"], r["cos"], r["p"]])
        m = st.motion(lw.next()[0])
        mot.append([m["dhat"], m["s"]])
    out["ssf"] = ssf
    out["motion"] = mot
    st.close()
    # guidance / update / entry variants of one step (first 6 elements)
    variants = {}
    for name, kw in (("supplied_negative_ddpm", dict(cfg_type=2, update_kind=1, n=4,
                                                     t_index=[0, 16, 32, 45])),
                     ("txt2img_no_guidance", dict(cfg_type=0, txt2img=1))):
        wv = W.get_config("c1_tiny", **kw)
        sv = O.Stream(wv)
        lv = W.gen_latents(wv, 1)
        en = lv["eps_neg"][:, 0] if "eps_neg" in lv else None
        x0n = None if wv["txt2img"] else lv["x0_new"][0]
        xn, o = sv.step_update(lv["x"][:, 0], lv["x0"][:, 0], lv["eps_c"][:, 0], lv["z"][:, 0], x0n,
                               lv["eps_new"][0], eps_neg=en)
        variants[name] = {"x_next": xn[:, :6].tolist(), "out": o[:6].tolist()}
        sv.close()
    out["step_update_variants"] = variants
    # the noise rate choosing the incoming frame's entry timestep over a walk
    wr = W.get_config("c1_tiny", noise_rate_on=1, burst_prob=0.5, lat_step=0.3)
    sr, lwr = O.Stream(wr), W.LatentWalk(wr)
    entry = []
    for t in range(6):
        lr = W.gen_latents(wr, t)
        sr.step_update(lr["x"][:, 0], lr["x0"][:, 0], lr["eps_c"][:, 0], lr["z"][:, 0],
                       lr["x0_new"][0], lr["eps_new"][0])
        m = sr.motion(lwr.next()[0])
        entry.append([sr.slot0_timestep(), m["s"]])
    out["noise_rate_entry"] = entry
    sr.close()
    return out


if __name__ == "__main__":
    path = os.path.join(HERE, "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(compute(), f, indent=1)
    print("wrote", path)
