"""Workload definitions and seeded synthetic input generators.

This module is the one place that both the CUDA path's tests/bench and the
CPU oracle draw their inputs from.  It holds shapes, parameters and random
number generation only -- none of the method's arithmetic (no attention, no
RoPE, no schedule, no guidance, no similarity test).

Every random draw is counter based: a (seed, purpose, index) triple selects
an independent numpy PCG64 stream, so an input depends only on its indices
and never on the order in which other inputs were drawn.

The five workloads follow the shapes the StreamDiffusion / StreamDiffusionV2
pages describe (StreamDiffusion notes: "Stream Batch", "R-CFG", "SSF";
StreamDiffusionV2 summary: "Adaptive sink and RoPE refresh", "Motion-aware
noise scheduler").  No trained weights or datasets are used; Q/K/V are
N(0,1) and latents/frames/embeddings are seeded random walks.
"""
from __future__ import annotations

import copy
import numpy as np

# purpose ids for the counter-based streams
_P_Q, _P_K, _P_V, _P_X, _P_X0, _P_EPSC, _P_Z, _P_X0NEW, _P_EPSNEW = range(9)
_P_U, _P_SSF, _P_EMB, _P_LAT, _P_JUMP, _P_BURST, _P_MISC = range(9, 16)
_P_EPSNEG = 16

_BASE = dict(
    streams=1,
    rope_base=10000.0,
    rope_tau=1024,
    n_inf=50,
    n_train=1000,
    beta_start=0.00085,
    beta_end=0.012,
    cfg_type=1,          # 1 = self-negative R-CFG, 2 = supplied negative prediction
    update_kind=0,       # 0 = predict x0 then re-noise, 1 = strided DDPM posterior
    noise_rate_on=0,     # 1 = the incoming frame enters slot 0 at the motion noise rate
    eps_c_bf16=0,        # 1 = the noise predictions eps_c arrive as bf16
    txt2img=0,           # 1 = no input image: the incoming frame is the noise draw itself
    gamma=1.4,
    delta=1.0,
    s_th=0.9,
    eta=0.98,
    max_skip=10,
    sigma=1.0,
    lam=0.9,
    s_min=0.3,
    s_max=0.9,
    emb_step=0.1,        # embedding random-walk step (scaled by 1/sqrt(D))
    lat_step=0.05,       # motion latent random-walk step
    burst_prob=0.0,
    burst_scale=20.0,
    ssf_step=0.1,
    ssf_jump_prob=1.0 / 32.0,
)

CONFIGS = {
    # tiny CPU-seconds case (seed 0)
    "c1_tiny": dict(
        _BASE, name="c1_tiny", seed=0, mode="video",
        n=2, T=1, L=64, grid_h=8, grid_w=8, H=2, d=64, M=1, R=4,
        rope=True, D=128, emb_step=0.3, t_index=[32, 45],
        latent_c=16, latent_h=8, latent_w=8,
        ssf=True, ssf_c=3, ssf_h=64, ssf_w=64,
        motion=True, mot_k=1, steps=8),
    # SD-turbo shaped image stream batch (external cross-frame K/V)
    "c2_sdturbo_image": dict(
        _BASE, name="c2_sdturbo_image", seed=1, mode="image",
        n=4, T=1, L=4096, grid_h=64, grid_w=64, H=5, d=64, M=0, R=0,
        rope=False, D=0, t_index=[0, 16, 32, 45],
        latent_c=4, latent_h=64, latent_w=64,
        ssf=True, ssf_c=3, ssf_h=512, ssf_w=512,
        motion=False, mot_k=1, steps=256),
    # 1.3B-DiT shaped video stream
    "c3_dit1p3b_video": dict(
        _BASE, name="c3_dit1p3b_video", seed=2, mode="video",
        n=2, T=3, L=1560, grid_h=30, grid_w=52, H=12, d=128, M=1, R=6,
        rope=True, D=1536, t_index=[32, 45],
        latent_c=16, latent_h=60, latent_w=104,
        ssf=False, ssf_c=3, ssf_h=512, ssf_w=512,
        motion=True, mot_k=3, steps=64),
    # 14B-DiT shaped video stream
    "c4_dit14b_video": dict(
        _BASE, name="c4_dit14b_video", seed=3, mode="video",
        n=4, T=3, L=1560, grid_h=30, grid_w=52, H=40, d=128, M=1, R=12,
        rope=True, D=5120, t_index=[0, 16, 32, 45],
        latent_c=16, latent_h=60, latent_w=104,
        ssf=False, ssf_c=3, ssf_h=512, ssf_w=512,
        motion=True, mot_k=3, steps=16),
    # long-run stress at the 1.3B shape, B = 1..8 concurrent streams
    "c5_stress": dict(
        _BASE, name="c5_stress", seed=4, mode="video",
        n=2, T=3, L=1560, grid_h=30, grid_w=52, H=12, d=128, M=1, R=6,
        rope=True, D=1536, t_index=[32, 45],
        latent_c=16, latent_h=60, latent_w=104,
        ssf=False, ssf_c=3, ssf_h=512, ssf_w=512,
        motion=True, mot_k=3, steps=10000, burst_prob=0.05),
}


def get_config(name: str, **overrides) -> dict:
    """Return a copy of a named workload with derived sizes filled in."""
    cfg = copy.deepcopy(CONFIGS[name])
    cfg.update(overrides)
    return derive(cfg)


def derive(cfg: dict) -> dict:
    """Fill in the sizes that follow from a workload's shape fields."""
    cfg["N_f"] = cfg["latent_c"] * cfg["latent_h"] * cfg["latent_w"]
    cfg["N_s"] = cfg["T"] * cfg["N_f"]
    cfg["ssf_E"] = cfg["ssf_c"] * cfg["ssf_h"] * cfg["ssf_w"]
    cfg["HD"] = cfg["H"] * cfg["d"]
    if cfg["mode"] == "video":
        cfg["q_rows"] = cfg["n"] * cfg["T"] * cfg["L"]
        cfg["kv_rows"] = cfg["T"] * cfg["L"]          # one pushed chunk
        cfg["key_cap"] = (cfg["M"] + cfg["R"]) * cfg["L"]
    else:
        cfg["q_rows"] = cfg["n"] * cfg["L"]
        cfg["kv_rows"] = cfg["n"] * cfg["L"]          # external batch K/V
        cfg["key_cap"] = cfg["n"] * cfg["L"]
    if cfg["D"] == 0:
        cfg["D"] = cfg["HD"]
    return cfg


# ---------------------------------------------------------------------------
# counter-based random streams


def _rng(seed: int, purpose: int, *idx: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, purpose] + [int(i) for i in idx])
    return np.random.Generator(np.random.PCG64(ss))


def normal_f32(seed: int, purpose: int, shape, *idx: int) -> np.ndarray:
    return _rng(seed, purpose, *idx).standard_normal(shape, dtype=np.float32)


def uniform_f32(seed: int, purpose: int, shape, *idx: int) -> np.ndarray:
    """Uniform draws in [0, 1) as float32 (never rounds up to 1.0)."""
    u = _rng(seed, purpose, *idx).random(shape, dtype=np.float64)
    u = u.astype(np.float32)
    return np.minimum(u, np.float32(np.nextafter(np.float32(1.0), np.float32(0.0))))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as bfloat16 bit patterns (round to nearest even).

    This is an input encoding step (the tensors handed to both sides are
    bf16); inputs are finite so no NaN handling is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# per-step tensors


def gen_q(cfg: dict, step: int) -> np.ndarray:
    """Queries of all n slots, bf16 bits, [S][q_rows][H][d]."""
    sh = (cfg["streams"], cfg["q_rows"], cfg["H"], cfg["d"])
    return to_bf16_bits(normal_f32(cfg["seed"], _P_Q, sh, step))


def gen_kv(cfg: dict, step: int):
    """K and V of one step, bf16 bits, [S][kv_rows][H][d] each.

    Video mode: the chunk pushed into the ring.  Image mode: the external
    cross-frame batch K/V of all n slots.
    """
    sh = (cfg["streams"], cfg["kv_rows"], cfg["H"], cfg["d"])
    k = to_bf16_bits(normal_f32(cfg["seed"], _P_K, sh, step))
    v = to_bf16_bits(normal_f32(cfg["seed"], _P_V, sh, step))
    return k, v


def gen_latents(cfg: dict, step: int) -> dict:
    """fp32 stream-batch latents of one step, slot-major [n][S][N_s]."""
    n, S, N = cfg["n"], cfg["streams"], cfg["N_s"]
    sd = cfg["seed"]
    out = dict(
        x=normal_f32(sd, _P_X, (n, S, N), step),
        x0=normal_f32(sd, _P_X0, (n, S, N), step),
        eps_c=normal_f32(sd, _P_EPSC, (n, S, N), step),
        z=normal_f32(sd, _P_Z, (max(n - 1, 1), S, N), step)[: max(n - 1, 0)],
        x0_new=normal_f32(sd, _P_X0NEW, (S, N), step),
        eps_new=normal_f32(sd, _P_EPSNEW, (S, N), step),
    )
    if cfg.get("cfg_type", 1) == 2:  # a supplied negative / unconditional prediction per slot
        out["eps_neg"] = normal_f32(sd, _P_EPSNEG, (n, S, N), step)
    return out


def gen_u(cfg: dict, step: int) -> np.ndarray:
    """SSF uniform draws, one per stream, [S] float32 in [0,1)."""
    return uniform_f32(cfg["seed"], _P_U, (cfg["streams"],), step)


class EmbeddingWalk:
    """Unit-norm random walk of chunk embeddings, e_k = normalize(e_{k-1} + a*xi/sqrt(D))."""

    def __init__(self, cfg: dict):
        self.cfg = cfg
        self.k = 0
        self.e = None

    def next(self) -> np.ndarray:
        c = self.cfg
        S, D = c["streams"], c["D"]
        xi = normal_f32(c["seed"], _P_EMB, (S, D), self.k).astype(np.float64)
        if self.e is None:
            e = xi
        else:
            e = self.e + c["emb_step"] * xi / np.sqrt(D)
        e = e / np.linalg.norm(e, axis=1, keepdims=True)
        self.e = e
        self.k += 1
        return e.astype(np.float32)


class LatentWalk:
    """Random-walk latent frames v_f = v_{f-1} + a*xi, with rare bursts.

    A chunk whose burst draw fires uses a step burst_scale times larger for
    all its frames (the high-motion bursts of the long-run stress case).
    Returns [S][T][N_f] float32 per chunk.
    """

    def __init__(self, cfg: dict):
        self.cfg = cfg
        self.k = 0
        self.prev = None

    def next(self) -> np.ndarray:
        c = self.cfg
        S, T, N = c["streams"], c["T"], c["N_f"]
        xi = normal_f32(c["seed"], _P_LAT, (S, T, N), self.k).astype(np.float64)
        burst = uniform_f32(c["seed"], _P_BURST, (S,), self.k) < c["burst_prob"]
        step = np.where(burst, c["lat_step"] * c["burst_scale"], c["lat_step"])[:, None]
        if self.prev is None:
            self.prev = normal_f32(c["seed"], _P_LAT, (S, N), 1 << 30).astype(np.float64)
        out = np.empty((S, T, N), dtype=np.float64)
        cur = self.prev
        for j in range(T):
            cur = cur + step * xi[:, j, :]
            out[:, j, :] = cur
        self.prev = cur
        self.k += 1
        return out.astype(np.float32)


class FrameWalk:
    """Unit-RMS random walk of SSF input frames with sparse jumps.

    I_t = rms_normalize(I_{t-1} + a*xi); with probability ssf_jump_prob a
    frame is a fresh N(0,1) draw instead (an uncorrelated scene cut).
    Returns [S][E] float32.
    """

    def __init__(self, cfg: dict):
        self.cfg = cfg
        self.k = 0
        self.cur = None

    def next(self) -> np.ndarray:
        c = self.cfg
        S, E = c["streams"], c["ssf_E"]
        xi = normal_f32(c["seed"], _P_SSF, (S, E), self.k).astype(np.float64)
        jump = uniform_f32(c["seed"], _P_JUMP, (S,), self.k) < c["ssf_jump_prob"]
        if self.cur is None:
            nxt = xi
        else:
            nxt = np.where(jump[:, None], xi, self.cur + c["ssf_step"] * xi)
        nxt = nxt / np.sqrt(np.mean(nxt * nxt, axis=1, keepdims=True))
        self.cur = nxt
        self.k += 1
        return nxt.astype(np.float32)
