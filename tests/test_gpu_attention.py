"""GPU parity of K1 (cross-frame attention) against the oracle.

Tolerance: per (row block, head), max |o - o_ref| <= 2e-2 * max(max|o_ref|,
rms(o_ref)) -- the bf16 attention bound; the oracle accumulates in double.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import GpuPipe, attn_rel_err, bf16_dev, bf16_host

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _bf(rng, shape, scale=1.0):
    return W.to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("S,Lq,Lk,H,d", [
    (1, 128, 128, 1, 64),      # one tile each way
    (1, 1, 1, 1, 64),          # degenerate: one query, one key
    (1, 200, 300, 2, 64),      # ragged queries and keys
    (2, 257, 1000, 3, 128),    # several tiles, ragged tails, two problems
    (1, 37, 5, 1, 128),        # fewer keys than one tile
    (1, 384, 4096, 2, 64),     # many key tiles (online-softmax rescaling)
    (1, 1, 1, 1, 128),         # d = 128 degenerate
    (1, 300, 130, 2, 128),     # last key tile: 2 keys, its second 64-key half empty
    (1, 256, 192, 1, 128),     # last key tile: exactly 64 keys
    (1, 384, 4096, 2, 128),    # d = 128, many key tiles
])
def test_raw_attention_matches_oracle(S, Lq, Lk, H, d):
    rng = np.random.default_rng(1000 + Lq + Lk)
    q = _bf(rng, (S, Lq, H, d))
    k = _bf(rng, (S, Lk, H, d))
    v = _bf(rng, (S, Lk, H, d))
    o = torch.empty((S, Lq, H, d), dtype=torch.bfloat16, device="cuda")
    B.sds_attention(bf16_dev(q), bf16_dev(k), bf16_dev(v), o, S, Lq, Lk, H, d)
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(bf16_host(o)).astype(np.float64)
    for s in range(S):
        ref = O.attention(q[s], k[s], v[s])
        err = attn_rel_err(got[s], ref)
        assert err <= TOL, (s, err)


def _rising_case(rng, S, Lq, Lk, H, d, ramp):
    """Queries and keys that share one direction u, with the keys' weight on
    u growing along the key index: every row's scores climb (ramp > 0) or
    fall (ramp < 0) across the keys, so the running maximum keeps moving up
    inside key tiles, not only at their first keys."""
    u = rng.standard_normal(d)
    w = np.linspace(0.0, 1.0, Lk) * ramp
    q = rng.standard_normal((S, Lq, H, d)) + 1.5 * u
    k = rng.standard_normal((S, Lk, H, d)) + w[None, :, None, None] * u
    v = rng.standard_normal((S, Lk, H, d))
    return [W.to_bf16_bits(a.astype(np.float32)) for a in (q, k, v)]


def _mid_tile_jumps(q, k, d):
    """Rows x 32-key parts (not the first part of a 128-key tile) at which
    the part's largest score, in log2 units, exceeds the largest of all
    earlier keys by more than 8."""
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    kf = W.bf16_bits_to_f32(k).astype(np.float64)
    s = np.einsum("qhd,khd->hqk", qf, kf) / np.sqrt(d) / np.log(2.0)
    Lk = s.shape[-1]
    n = 0
    for p0 in range(32, Lk, 32):
        if p0 % 128 == 0:
            continue
        before = s[..., :p0].max(axis=-1)
        part = s[..., p0:p0 + 32].max(axis=-1)
        n += int(np.sum(part > before + 8.0))
    return n


@pytest.mark.parametrize("S,Lq,Lk,H,d,ramp", [
    (1, 512, 1024, 2, 64, 6.0),
    (1, 256, 640, 1, 64, 20.0),
    (2, 384, 2048, 1, 64, 12.0),
    (1, 256, 1000, 1, 64, -6.0),
    (1, 256, 640, 1, 64, 80.0),    # jumps past the reference overflow exp2: recomputed
    (1, 300, 700, 1, 64, 200.0),   # ragged, every later tile overflows
    (1, 256, 1024, 1, 128, 12.0),
])
def test_raw_attention_scores_rising_along_the_keys(S, Lq, Lk, H, d, ramp):
    """The online softmax's reference maximum moves inside key tiles; the
    probabilities already made against the old reference must follow it."""
    rng = np.random.default_rng(int(500 + Lq + Lk + 10 * abs(ramp)))
    q, k, v = _rising_case(rng, S, Lq, Lk, H, d, ramp)
    if ramp > 0:
        assert _mid_tile_jumps(q[0], k[0], d) > 0  # the case exercises mid-tile moves
    o = torch.empty((S, Lq, H, d), dtype=torch.bfloat16, device="cuda")
    B.sds_attention(bf16_dev(q), bf16_dev(k), bf16_dev(v), o, S, Lq, Lk, H, d)
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(bf16_host(o)).astype(np.float64)
    for s in range(S):
        ref = O.attention(q[s], k[s], v[s])
        err = attn_rel_err(got[s], ref)
        assert err <= TOL, (s, err)


@pytest.mark.parametrize("ctas,ramp,d", [
    (37, 20.0, 64),    # 2-3 key tiles per CTA: later tiles move the reference (stored P rescaled)
    (37, 80.0, 64),    # ... or overflow and are recomputed
    (160, 80.0, 64),   # single-tile contributors: every partial starts from its own maximum
    # d = 128: O is rescaled at most tiles, inside segments (after the next
    # tile's scores) and at a segment's last tile (after its o_done)
    (37, 20.0, 128),
    (160, 20.0, 128),  # one key tile per segment: its last tile is also its first
])
def test_split_key_schedule_with_rising_scores(ctas, ramp, d):
    """Items split between CTAs whose contributors ended on different
    references (some moved inside their key range) merge to the oracle's
    result."""
    w = W.get_config("c2_sdturbo_image", L=320, H=2, d=d, grid_h=16, grid_w=20, latent_h=16, latent_w=20,
                     ssf_h=64, ssf_w=64, attn_ctas=ctas)
    rng = np.random.default_rng(int(900 + ctas + ramp + (d - 64)))
    q, k, v = _rising_case(rng, w["streams"], w["q_rows"], w["kv_rows"], w["H"], w["d"], ramp)
    g = GpuPipe(w)
    try:
        for rep in range(2):  # the second launch reuses the arrival counters
            got = g.attend(q, k, v)
            assert attn_rel_err(got[0], O.attention(q[0], k[0], v[0])) <= TOL, rep
    finally:
        g.close()


@pytest.mark.parametrize("d", [64, 128])
def test_raw_attention_large_scores_stay_finite(d):
    """Peaked softmax (scores ~ +-100): the running max must keep exp2 in range."""
    rng = np.random.default_rng(7)
    S, Lq, Lk, H = 1, 128, 640, 1
    q = _bf(rng, (S, Lq, H, d), 6.0 * (64 / d) ** 0.25)
    k = _bf(rng, (S, Lk, H, d), 6.0 * (64 / d) ** 0.25)
    v = _bf(rng, (S, Lk, H, d))
    o = torch.empty((S, Lq, H, d), dtype=torch.bfloat16, device="cuda")
    B.sds_attention(bf16_dev(q), bf16_dev(k), bf16_dev(v), o, S, Lq, Lk, H, d)
    torch.cuda.synchronize()
    got = W.bf16_bits_to_f32(bf16_host(o)).astype(np.float64)
    assert np.all(np.isfinite(got))
    assert attn_rel_err(got[0], O.attention(q[0], k[0], v[0])) <= TOL


def test_image_mode_attend_small_batch():
    w = W.get_config("c2_sdturbo_image", L=320, grid_h=16, grid_w=20, latent_h=16, latent_w=20,
                     ssf_h=64, ssf_w=64)
    g = GpuPipe(w)
    try:
        q = W.gen_q(w, 0)
        k, v = W.gen_kv(w, 0)
        got = g.attend(q, k, v)
        ref = O.attention(q[0], k[0], v[0])
        assert attn_rel_err(got[0], ref) <= TOL
    finally:
        g.close()


@pytest.mark.parametrize("ctas,L,H", [
    (7, 320, 5),     # items split across many CTAs, several contributors each
    (37, 320, 5),    # ragged split points
    (148, 320, 5),   # more CTAs than items
    (160, 96, 2),    # one query pair, keys split into single tiles
])
def test_image_mode_split_key_schedule(ctas, L, H):
    """The persistent schedule with keys of a query tile split between CTAs
    (partials merged by the last contributor) against the oracle."""
    w = W.get_config("c2_sdturbo_image", L=L, H=H, grid_h=16, grid_w=L // 16, latent_h=16,
                     latent_w=L // 16, ssf_h=64, ssf_w=64, attn_ctas=ctas)
    g = GpuPipe(w)
    try:
        for rep in range(2):  # the second launch reuses the arrival counters
            q = W.gen_q(w, rep)
            k, v = W.gen_kv(w, rep)
            got = g.attend(q, k, v)
            ref = O.attention(q[0], k[0], v[0])
            assert attn_rel_err(got[0], ref) <= TOL, (ctas, rep)
    finally:
        g.close()


def test_image_mode_full_size_sampled_rows():
    """c2 at full size (4 slots x 4096 queries against 16384 batch keys), sampled rows."""
    w = W.get_config("c2_sdturbo_image")
    g = GpuPipe(w)
    try:
        q = W.gen_q(w, 3)
        k, v = W.gen_kv(w, 3)
        got = g.attend(q, k, v)
        rows = np.unique(np.concatenate([np.arange(0, 16384, 61), [0, 127, 128, 4095, 4096, 16383]]))
        ref = O.attention(q[0], k[0], v[0], rows=rows)
        assert attn_rel_err(got[0][rows], ref) <= TOL
    finally:
        g.close()
