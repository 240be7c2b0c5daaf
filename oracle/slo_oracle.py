"""Plain restatement of the SLO-aware stream-batch controller.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/).

StreamDiffusionV2 summary, "SLO-aware batching scheduler": an iteration over
B streams of T frames has latency L(T, B); in the memory-bound regime L is
affine in the activation volume, linear in B*T; a stream meets the target
frame rate f when T / L >= f; the aggregate rate B*T / L grows with B until
the roofline knee.  Readings: L = a + b*B*T fitted by least squares with
older observations weighted by forget^age; the choice is the largest B
meeting the target, capped at the knee = the smallest B whose predicted
aggregate rate is within knee_gain of the rate at b_max; with fewer than two
distinct B observed, the next unobserved B from b_min up.
"""
from __future__ import annotations

import numpy as np


def fit(obs, T: int, forget: float):
    """obs: [(B, latency)] oldest first.  Returns (a, b) or None."""
    if len({B for B, _ in obs}) < 2:
        return None
    n = len(obs)
    x = np.array([B * T for B, _ in obs], dtype=np.float64)
    y = np.array([L for _, L in obs], dtype=np.float64)
    w = np.array([forget ** (n - 1 - i) for i in range(n)], dtype=np.float64)
    # weighted least squares via the normal equations of [1, x]
    A = np.stack([np.ones(n), x], axis=1)
    coef = np.linalg.solve(A.T @ (w[:, None] * A), A.T @ (w * y))
    return float(coef[0]), float(coef[1])


def choose(obs, target_fps: float, T: int, b_min: int, b_max: int, forget: float = 1.0,
           knee_gain: float = 0.05) -> dict:
    ab = fit(obs, T, forget)
    if ab is None:
        seen = {B for B, _ in obs}
        nxt = next((B for B in range(b_min, b_max) if B not in seen), b_max)
        return dict(batch=nxt, exploring=1)
    a, b = ab
    lat = {B: a + b * B * T for B in range(b_min, b_max + 1)}
    tot = {B: B * T / lat[B] for B in lat if lat[B] > 0}
    meets = [B for B in lat if lat[B] > 0 and T / lat[B] >= target_fps]
    b_slo = max(meets) if meets else 0
    f_max = tot.get(b_max, 0.0)
    b_knee = next((B for B in range(b_min, b_max + 1) if B in tot and tot[B] >= (1 - knee_gain) * f_max),
                  b_max)
    batch = min(b_slo, b_knee) if b_slo else b_min
    return dict(batch=batch, exploring=0, b_slo=b_slo, b_knee=b_knee, a=a, b=b,
                per_stream_fps=T / lat[batch], total_fps=batch * T / lat[batch],
                meets_slo=int(T / lat[batch] >= target_fps))
