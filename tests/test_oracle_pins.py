"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against a closed form, an invariant,
a special case that reduces to a library routine, or brute force on tiny
inputs -- chosen so that a dropped term, a wrong sign or index or a swapped
operand in the oracle fails at least one of them.  CPU only.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from streaming_diffusion_stream_b300 import workloads as W


def tiny(**kw):
    return W.get_config("c1_tiny", **kw)


# --------------------------------------------------------------- bf16

def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000), rng.standard_normal(1000) * 1e-30,
                        rng.standard_normal(1000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([O.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_ties_to_even_and_value_roundtrip():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert O.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even): goes up
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above a tie rounds up (no intermediate float rounding)
    assert O.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    for b in (0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F):
        assert O.bf16_round(O.bf16_value(b)) == b


# --------------------------------------------------------------- schedule

def test_alpha_bar_scaled_linear_closed_form_bounds():
    w = tiny()
    ab = O.alpha_bar(w)
    N = w["n_train"]
    a, b = math.sqrt(w["beta_start"]), math.sqrt(w["beta_end"])
    h = (b - a) / (N - 1)
    # first step: beta_0 = beta_start exactly
    assert abs(ab[0] - (1.0 - w["beta_start"])) < 1e-15
    # ratio of consecutive entries recovers beta_t; the last equals beta_end
    assert abs((1.0 - ab[-1] / ab[-2]) - w["beta_end"]) < 1e-12
    # closed form sum of the quadratic betas bounds -log(alphabar_{N-1})
    s1 = N * a * a + 2 * a * h * N * (N - 1) / 2 + h * h * (N - 1) * N * (2 * N - 1) / 6
    s2 = sum((a + s * h) ** 4 for s in range(N))
    nl = -math.log(ab[-1])
    assert s1 <= nl <= s1 + 0.5 * s2 / (1 - w["beta_end"]) + 1e-12
    assert np.all(np.diff(ab) < 0)


def test_slot_timesteps_reading():
    w = tiny(t_index=[32, 45])
    assert [O.slot_timestep(w, i) for i in range(2)] == [359, 99]
    w = tiny(t_index=[0, 16, 32, 45], n=4)
    assert [O.slot_timestep(w, i) for i in range(4)] == [999, 679, 359, 99]


# --------------------------------------------------------------- RoPE

def test_rope_segments():
    assert O.rope_segments(128) == [44, 42, 42]
    assert O.rope_segments(64) == [24, 20, 20]


def test_rope_position_zero_is_identity_and_norms_preserved():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 128))
    out = O.rope_rotate(v, np.zeros((5, 3), dtype=np.int64))
    assert np.array_equal(out, v)
    pos = rng.integers(0, 2000, size=(5, 3))
    out = O.rope_rotate(v, pos)
    pn_in = v[:, 0::2] ** 2 + v[:, 1::2] ** 2
    pn_out = out[:, 0::2] ** 2 + out[:, 1::2] ** 2
    assert np.allclose(pn_in, pn_out, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("d", [64, 128])
def test_rope_unit_vectors_turn_by_closed_form_angle(d):
    seg = O.rope_segments(d)
    starts = [0, seg[0], seg[0] + seg[1]]
    pos = np.array([[7, 3, 11]])
    for a in range(3):
        for i in range(seg[a] // 2):
            e = np.zeros((1, d))
            e[0, starts[a] + 2 * i] = 1.0
            out = O.rope_rotate(e, pos)
            th = pos[0, a] * 10000.0 ** (-2.0 * i / seg[a])
            expect = np.zeros(d)
            expect[starts[a] + 2 * i] = math.cos(th)
            expect[starts[a] + 2 * i + 1] = math.sin(th)
            assert np.allclose(out[0], expect, atol=1e-12), (a, i)


def test_rope_relative_position_property():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for _ in range(5):
        p = rng.integers(0, 500, size=(1, 3))
        pk = rng.integers(0, 500, size=(1, 3))
        c = rng.integers(0, 500, size=(1, 3))
        a = float((O.rope_rotate(q, p) @ O.rope_rotate(k, pk).T)[0, 0])
        b = float((O.rope_rotate(q, p + c) @ O.rope_rotate(k, pk + c).T)[0, 0])
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_rope_axes_are_independent():
    rng = np.random.default_rng(3)
    seg = O.rope_segments(128)
    v = np.zeros((1, 128))
    v[0, seg[0]:seg[0] + seg[1]] = rng.standard_normal(seg[1])  # row-axis segment only
    a = O.rope_rotate(v, np.array([[5, 2, 9]]))
    b = O.rope_rotate(v, np.array([[900, 2, 1]]))
    assert np.array_equal(a, b)


# --------------------------------------------------------------- attention

def _bf(x):
    return W.to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f(b):
    return W.bf16_bits_to_f32(b).astype(np.float64)


def test_attention_single_key_returns_value():
    rng = np.random.default_rng(4)
    q = _bf(rng.standard_normal((3, 2, 64)))
    k = _bf(rng.standard_normal((1, 2, 64)))
    v = _bf(rng.standard_normal((1, 2, 64)))
    o = O.attention(q, k, v)
    assert np.array_equal(o, np.broadcast_to(_f(v)[0], o.shape))


def test_attention_equal_keys_and_zero_query_give_mean():
    rng = np.random.default_rng(5)
    v = _bf(rng.standard_normal((37, 2, 64)))
    k = np.broadcast_to(_bf(rng.standard_normal((1, 2, 64))), (37, 2, 64)).copy()
    q = _bf(rng.standard_normal((4, 2, 64)))
    o = O.attention(q, k, v)
    assert np.allclose(o, _f(v).mean(axis=0)[None], atol=1e-13)
    k2 = _bf(rng.standard_normal((37, 2, 64)))
    o2 = O.attention(np.zeros_like(q), k2, v)
    assert np.allclose(o2, _f(v).mean(axis=0)[None], atol=1e-13)


def test_attention_two_keys_logistic_closed_form():
    rng = np.random.default_rng(6)
    q = _bf(rng.standard_normal((5, 1, 64)))
    k = _bf(rng.standard_normal((2, 1, 64)))
    v = _bf(rng.standard_normal((2, 1, 64)))
    o = O.attention(q, k, v)
    qf, kf, vf = _f(q)[:, 0], _f(k)[:, 0], _f(v)[:, 0]
    s = qf @ kf.T / 8.0
    w0 = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    expect = w0[:, None] * vf[0] + (1 - w0)[:, None] * vf[1]
    assert np.allclose(o[:, 0], expect, atol=1e-12)


def test_attention_matches_torch_sdpa_float64_and_invariances():
    rng = np.random.default_rng(7)
    q = _bf(rng.standard_normal((9, 3, 64)))
    k = _bf(rng.standard_normal((50, 3, 64)))
    v = _bf(rng.standard_normal((50, 3, 64)))
    o = O.attention(q, k, v)
    tq = torch.from_numpy(_f(q)).permute(1, 0, 2)
    tk = torch.from_numpy(_f(k)).permute(1, 0, 2)
    tv = torch.from_numpy(_f(v)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(1, 0, 2).numpy()
    assert np.allclose(o, ref, atol=1e-12)
    perm = rng.permutation(50)
    assert np.allclose(O.attention(q, k[perm], v[perm]), o, atol=1e-13)
    v2 = _bf(_f(v) * 2.0)  # exact in bf16
    assert np.allclose(O.attention(q, k, v2), 2.0 * o, atol=1e-13)
    rows = np.array([8, 0, 4])
    assert np.array_equal(O.attention(q, k, v, rows=rows), o[rows])


# --------------------------------------------------------------- ring, RoPE reset, sinks

def _chunk(w, seed):
    rng = np.random.default_rng(seed)
    sh = (w["T"] * w["L"], w["H"], w["d"])
    return _bf(rng.standard_normal(sh)), _bf(rng.standard_normal(sh))


def test_ring_holds_exactly_the_last_R_frames():
    w = tiny(T=1, R=4, rope=False)
    s = O.Stream(w)
    frames = []
    L, HD = w["L"], w["H"] * w["d"]
    for c in range(11):
        k, v = _chunk(w, 100 + c)
        s.push(k, v)
        frames.append((k, v))
        m = s.meta()
        F = m["F"]
        assert F == c + 1 and m["valid"] == min(F, 4)
        kb, vb = s.kv()
        for f in range(max(0, F - 4), F):
            slot = f % 4
            rows = slice((w["M"] + slot) * L, (w["M"] + slot + 1) * L)
            assert np.array_equal(vb[rows], frames[f][1])
            assert np.array_equal(kb[rows], frames[f][0])  # RoPE off: plain copy


def test_rope_reset_sequence_tau3():
    for T, expect in ((1, [0, 1, 2, 3, 0, 1, 2, 3, 0]), (2, [0, 2, 0, 2, 0, 2])):
        w = tiny(T=T, R=4, rope_tau=3)
        s = O.Stream(w)
        seen = []
        for c in range(len(expect)):
            k, v = _chunk(w, c)
            seen.append(s.push(k, v))
        assert seen == expect, (T, seen)
        assert s.meta()["resets"] == expect.count(0) - 1


def test_pushed_keys_are_rotated_at_their_positions():
    w = tiny(T=2, R=4, rope_tau=3)
    s = O.Stream(w)
    L, H, d, gw = w["L"], w["H"], w["d"], w["grid_w"]
    for c in range(3):
        k, v = _chunk(w, 40 + c)
        p0 = s.push(k, v)
    kb, _ = s.kv()
    # last chunk (c=2): F before push = 4 > ... p0 == 0 after reset; frame j -> slot (4+j) % 4
    assert p0 == 0
    for j in range(2):
        slot = (4 + j) % 4
        for l in (0, 9, L - 1):
            pos = np.array([[p0 + j, l // gw, l % gw]])
            for h in range(H):
                src = _f(k[j * L + l, h])[None]
                rot = O.rope_rotate(src, pos)[0]
                expect = np.array([O.bf16_round(x) for x in rot], dtype=np.uint16)
                assert np.array_equal(kb[(w["M"] + slot) * L + l, h], expect)


@pytest.mark.parametrize("M", [0, 1])
def test_query_rows_take_the_positions_of_the_chunk_just_pushed(M):
    """Which position a query row of orc_attend gets (StreamDiffusionV2
    summary, "Adaptive sink and RoPE refresh": every slot's queries belong
    to the chunk just pushed).  Query row r of slot s is token
    tok = r mod (T*L) of that chunk, frame j = tok // L, grid cell l = tok % L.
    Feed as queries the chunk's own raw keys, tiled over the n slots: a
    query is then rotated by the same arithmetic and at the same position as
    its key, so its rotated bf16 value must equal, bit for bit, the key the
    push stored for frame j, cell l (whose position is pinned by
    test_pushed_keys_are_rotated_at_their_positions).  The expected output
    is the brute-force attention of those stored keys against the key list.
    A query at another frame, a swapped row/column, or a slot with its own
    positions changes the rotation and the output by far more than the
    tolerance.  Runs across a RoPE reset (tau = 3) so p0 takes 0, 2 and 0."""
    w = tiny(n=3, T=2, R=4, M=M, rope_tau=3)
    s = O.Stream(w)
    L, TL, n, gw = w["L"], w["T"] * w["L"], w["n"], w["grid_w"]
    cells = [0, 3, gw + 5, 2 * gw + 1, 5 * gw + 2, L - 1]  # y != x for most
    seen_p0 = []
    F = 0
    for c in range(3):
        k, v = _chunk(w, 70 + c)
        seen_p0.append(s.push(k, v))
        if M:
            s.sink_refresh(np.ones(w["D"], dtype=np.float32))
        first = F
        F += w["T"]
        kb, vb = s.kv()
        keys = s.key_rows()
        q = np.concatenate([k] * n)  # [n*T*L][H][d]: slot s holds the chunk's keys
        rows, stored = [], []
        for sl in range(n):
            for j in range(w["T"]):
                for l in cells:
                    rows.append(sl * TL + j * L + l)
                    stored.append((M + (first + j) % w["R"]) * L + l)
        got = s.attend(q, np.array(rows))
        expect = O.attention(kb[np.array(stored)], kb[keys], vb[keys])
        np.testing.assert_allclose(got, expect, rtol=0, atol=1e-12)
        # the slots share the positions: identical outputs for the same token
        per = len(cells) * w["T"]
        for sl in range(1, n):
            assert np.array_equal(got[sl * per:(sl + 1) * per], got[:per])
    assert seen_p0 == [0, 2, 0]
    # the check has teeth: a query rotated one frame later (or with its row and
    # column swapped) gives a clearly different output
    kb, vb = s.kv()
    keys = s.key_rows()
    l = 2 * gw + 1
    src = _f(k[l])  # frame 0, cell (2, 1) of the last chunk, p0 = 0
    for pos in ([1, 2, 1], [0, 1, 2]):
        rot = O.rope_rotate(src, np.array([pos] * w["H"]))
        wrong = np.array([[O.bf16_round(x) for x in r] for r in rot], dtype=np.uint16)[None]
        o_wrong = O.attention(wrong, kb[keys], vb[keys])
        o_right = s.attend(np.concatenate([k] * n), np.array([l]))
        assert np.max(np.abs(o_wrong - o_right)) > 1e-3


def test_sink_fill_then_least_similar_refresh():
    w = tiny(M=2, T=3, R=6, D=2, s_th=0.96, rope=False)
    s = O.Stream(w)
    L = w["L"]
    k, v = _chunk(w, 1)
    s.push(k, v)
    r = s.sink_refresh(np.array([3.0, 4.0], dtype=np.float32))
    assert r["fire"] == 2 and s.meta()["sinks_filled"] == 2
    kb, vb = s.kv()
    for j in range(2):  # sinks 0,1 hold frames 0,1 of the first chunk
        assert np.array_equal(vb[j * L:(j + 1) * L], v[j * L:(j + 1) * L])
    assert np.array_equal(s.emb(), np.array([[3.0, 4.0], [3.0, 4.0]]))
    # equal cosines -> lowest index; cos = 24/25 == s_th exactly -> strict '<' does not fire
    k2, v2 = _chunk(w, 2)
    s.push(k2, v2)
    r = s.sink_refresh(np.array([4.0, 3.0], dtype=np.float32))
    assert r["j"] == 0 and r["fire"] == 0 and r["alpha_min"] == 0.96 and r["near"] == 1
    # orthogonal -> fires, replaces sink 0 with frame 0 of this chunk
    r = s.sink_refresh(np.array([-4.0, 3.0], dtype=np.float32))
    assert r["j"] == 0 and r["fire"] == 1 and r["alpha_min"] == 0.0
    kb, vb = s.kv()
    assert np.array_equal(vb[0:L], v2[0:L]) and np.array_equal(vb[L:2 * L], v[L:2 * L])
    assert np.array_equal(s.emb()[0], [-4.0, 3.0])
    # now sink 1 (3,4) is least similar to (-4,3)-ish query (cos 0 vs 1)
    r = s.sink_refresh(np.array([-4.0, 3.0], dtype=np.float32))
    assert r["j"] == 1 and r["fire"] == 1


def test_key_rows_are_filled_sinks_then_valid_ring():
    w = tiny(M=1, T=1, R=4)
    s = O.Stream(w)
    L = w["L"]
    k, v = _chunk(w, 3)
    s.push(k, v)
    assert len(s.key_rows()) == L  # sink not yet filled: ring frame only
    s.sink_refresh(np.ones(w["D"], dtype=np.float32))
    rows = s.key_rows()
    assert np.array_equal(rows, np.concatenate([np.arange(L), np.arange(L, 2 * L)]))
    for c in range(5):
        s.push(*_chunk(w, 10 + c))
    assert len(s.key_rows()) == 5 * L


# --------------------------------------------------------------- R-CFG + update

def _slots(w, rng):
    n, N = w["n"], w["N_s"]
    return {k: rng.standard_normal((n, N)).astype(np.float32) for k in ("x0", "eps", "eps_c", "z")}


def test_constructed_xt_returns_true_noise_and_x0():
    w = tiny(n=4, t_index=[0, 16, 32, 45])
    ab = O.alpha_bar(w)
    t = [O.slot_timestep(w, i) for i in range(4)]
    rng = np.random.default_rng(8)
    N = w["N_s"]
    x0 = rng.standard_normal((4, N)).astype(np.float32)
    eps = rng.standard_normal((4, N)).astype(np.float32)
    x = np.stack([np.sqrt(ab[t[i]]) * x0[i].astype(np.float64) + np.sqrt(1 - ab[t[i]]) * eps[i]
                  for i in range(4)]).astype(np.float32)
    z = rng.standard_normal((3, N)).astype(np.float32)
    xn_new = rng.standard_normal((2, N)).astype(np.float32)
    s = O.Stream(w)
    # eps_c = the noise actually used (from the fp32 x) -> eps_cfg == eps_neg == that noise -> x0hat = x0
    xd = x.astype(np.float64)
    eps_true = np.stack([(xd[i] - np.sqrt(ab[t[i]]) * x0[i]) / np.sqrt(1 - ab[t[i]]) for i in range(4)])
    assert np.allclose(eps_true, eps, atol=1e-5)  # fp32 storage of x
    xnext, out = s.step_update(x, x0, eps_true.astype(np.float32), z, xn_new[0], xn_new[1])
    # with eps_c rounded to fp32 the identity holds to ~1e-6 relative
    assert np.allclose(out, x0[3], atol=2e-5)
    for i in range(3):
        expect = np.sqrt(ab[t[i + 1]]) * x0[i] + np.sqrt(1 - ab[t[i + 1]]) * z[i].astype(np.float64)
        assert np.allclose(xnext[i + 1], expect, atol=2e-5)
    assert np.allclose(xnext[0], np.sqrt(ab[t[0]]) * xn_new[0] + np.sqrt(1 - ab[t[0]]) * xn_new[1].astype(np.float64),
                       atol=1e-13)


def test_gamma_one_returns_eps_c_and_printed_combine_agrees():
    rng = np.random.default_rng(9)
    w = tiny(gamma=1.0)
    ab = O.alpha_bar(w)
    t = [O.slot_timestep(w, i) for i in range(2)]
    sl = _slots(w, rng)
    s = O.Stream(w)
    x = sl["eps"]
    xn, out = s.step_update(x, sl["x0"], sl["eps_c"], sl["z"][:1], sl["x0"][0], sl["eps"][0])
    # gamma=1: x0hat = (x - sqrt(1-ab) eps_c)/sqrt(ab), exactly the formula with eps_cfg = eps_c
    a = ab[t[1]]
    expect = (x[1].astype(np.float64) - np.sqrt(1 - a) * sl["eps_c"][1]) / np.sqrt(a)
    assert np.array_equal(out, expect)
    # general gamma/delta: compare with the printed form delta*eps_neg + gamma*(eps_c - delta*eps_neg)
    for g, dl in ((1.4, 1.0), (2.5, 0.7), (0.3, 0.0)):
        w2 = tiny(gamma=g, delta=dl)
        s2 = O.Stream(w2)
        xn2, out2 = s2.step_update(x, sl["x0"], sl["eps_c"], sl["z"][:1], sl["x0"][0], sl["eps"][0])
        xd = x[1].astype(np.float64)
        en = (xd - np.sqrt(a) * sl["x0"][1]) / np.sqrt(1 - a)
        ecfg = dl * en + g * (sl["eps_c"][1] - dl * en)
        ref = (xd - np.sqrt(1 - a) * ecfg) / np.sqrt(a)
        assert np.allclose(out2, ref, rtol=1e-12, atol=1e-12)
        if dl == 0.0:  # delta = 0: eps_cfg = gamma * eps_c
            ref0 = (xd - np.sqrt(1 - a) * g * sl["eps_c"][1]) / np.sqrt(a)
            assert np.allclose(out2, ref0, rtol=1e-13, atol=1e-13)


def test_cfg_none_uses_eps_c():
    rng = np.random.default_rng(10)
    w = tiny(cfg_type=0, gamma=3.0)
    ab = O.alpha_bar(w)
    t1 = O.slot_timestep(w, 1)
    sl = _slots(w, rng)
    s = O.Stream(w)
    _, out = s.step_update(sl["eps"], sl["x0"], sl["eps_c"], sl["z"][:1], sl["x0"][0], sl["eps"][0])
    expect = (sl["eps"][1].astype(np.float64) - np.sqrt(1 - ab[t1]) * sl["eps_c"][1]) / np.sqrt(ab[t1])
    assert np.array_equal(out, expect)


def test_frame_encoded_at_t_completes_at_t_plus_n():
    """Stream Batch: a frame noised into slot 0 by step t leaves as the output of step t+n."""
    n = 4
    w = tiny(n=n, t_index=[0, 16, 32, 45], gamma=1.7)
    N = w["N_s"]
    rng = np.random.default_rng(11)
    s = O.Stream(w)
    frames = [rng.standard_normal(N).astype(np.float32) for _ in range(n + 4)]
    # slot state: latent x, its clean x0 and the noise that produced it
    x = np.zeros((n, N), dtype=np.float32)
    x0 = np.zeros((n, N), dtype=np.float32)
    outs = []
    ab = O.alpha_bar(w)
    t = [O.slot_timestep(w, i) for i in range(n)]
    for step in range(n + 4):
        eps_new = rng.standard_normal(N).astype(np.float32)
        z = rng.standard_normal((n - 1, N)).astype(np.float32)
        # ideal predictor: eps_c is the true noise of each slot's latent
        eps_c = np.stack([(x[i].astype(np.float64) - np.sqrt(ab[t[i]]) * x0[i]) / np.sqrt(1 - ab[t[i]])
                          for i in range(n)]).astype(np.float32)
        xn, out = s.step_update(x, x0, eps_c, z, frames[step], eps_new)
        outs.append(out)
        x = xn.astype(np.float32)
        x0 = np.concatenate([frames[step][None], x0[:-1]])
    for step in range(n, n + 4):
        assert np.allclose(outs[step], frames[step - n], atol=1e-4), step


# --------------------------------------------------------------- SSF

def test_ssf_identical_frames_probability_one_and_skip_cap():
    w = tiny(max_skip=3)
    s = O.Stream(w)
    f = np.random.default_rng(12).standard_normal(w["ssf_E"]).astype(np.float32)
    r = s.ssf(f, 0.0)
    assert r["skip"] == 0 and r["p"] == 0.0  # first frame: processed
    pattern = []
    for _ in range(9):
        r = s.ssf(f, 0.999)
        assert r["cos"] == 1.0 and r["p"] == 1.0
        pattern.append(r["skip"])
    assert pattern == [1, 1, 1, 0, 1, 1, 1, 0, 1]


def test_ssf_closed_form_cosines():
    w = tiny(eta=0.5)
    E = w["ssf_E"]
    s = O.Stream(w)
    ref = np.zeros(E, dtype=np.float32)
    ref[0::2] = 1.0
    s.ssf(ref, 0.0)
    r = s.ssf(np.ones(E, dtype=np.float32), 0.99)  # cos = 1/sqrt(2)
    assert abs(r["cos"] - 1 / math.sqrt(2)) < 1e-15
    assert abs(r["p"] - (1 / math.sqrt(2) - 0.5) / 0.5) < 1e-14
    assert r["skip"] == 0
    s2 = O.Stream(tiny(eta=0.98))
    s2.ssf(ref, 0.0)
    assert s2.ssf(np.ones(E, dtype=np.float32), 0.0)["p"] == 0.0  # cos <= eta -> 0
    s3 = O.Stream(tiny())
    s3.ssf(ref, 0.0)
    r = s3.ssf(-ref, 0.0)
    assert r["cos"] == -1.0 and r["p"] == 0.0
    odd = np.zeros(E, dtype=np.float32)
    odd[1::2] = 1.0
    r = s3.ssf(odd, 0.0)  # ref is still `ref` (last processed was -ref? no: -ref was processed)
    assert r["cos"] == 0.0
    r = s3.ssf(np.zeros(E, dtype=np.float32), 0.0)
    assert r["cos"] == 0.0 and r["p"] == 0.0


def test_ssf_reference_is_last_processed_frame():
    w = tiny(max_skip=10)
    E = w["ssf_E"]
    s = O.Stream(w)
    a = np.random.default_rng(13).standard_normal(E).astype(np.float32)
    b = (a + 0.01 * np.random.default_rng(14).standard_normal(E)).astype(np.float32)
    s.ssf(a, 0.0)
    r1 = s.ssf(b, 0.0)       # u = 0 < P: skipped, ref stays a
    assert r1["skip"] == 1
    r2 = s.ssf(b, 0.0)
    assert r2["cos"] == r1["cos"]  # still compared against a
    r3 = s.ssf(b, 0.9999999)  # not skipped -> ref becomes b
    assert r3["skip"] == 0
    assert s.ssf(b, 0.5)["cos"] == 1.0


# --------------------------------------------------------------- motion

def test_motion_identical_frames_hold_s_min():
    w = tiny(T=3, mot_k=3)
    s = O.Stream(w)
    f = np.random.default_rng(15).standard_normal(w["N_f"]).astype(np.float32)
    chunk = np.stack([f] * 3)
    for _ in range(6):
        r = s.motion(chunk)
        assert r["s"] == w["s_min"] and r["dhat"] == 0.0
    assert np.all(r["d"] == 0.0)


def test_motion_constant_shift_and_ema_closed_form():
    w = tiny(T=2, mot_k=2, sigma=0.5, lam=0.8)
    s = O.Stream(w)
    N = w["N_f"]
    base = np.random.default_rng(16).standard_normal(N)
    c = 0.125  # exact in fp32; every difference is exactly c
    fr = 0
    s0 = w["s_min"]
    target = w["s_min"] + (w["s_max"] - w["s_min"]) * (c / 0.5)
    vals = []
    for kch in range(5):
        chunk = np.stack([(base * 0 + (fr + j) * c) for j in range(2)]).astype(np.float32)
        fr += 2
        r = s.motion(chunk)
        if kch == 0:
            assert np.isnan(r["d"][0]) and abs(r["d"][1] - c) < 1e-12
        else:
            assert np.allclose(r["d"], c, atol=1e-12)
        vals.append(r["s"])
    for kk, sv in enumerate(vals, start=1):
        assert abs(sv - (target + 0.8 ** kk * (s0 - target))) < 1e-12


def test_motion_clips_at_one_and_window_max():
    w = tiny(T=1, mot_k=2, sigma=1.0, lam=0.0)  # lam = 0: s jumps to target
    s = O.Stream(w)
    N = w["N_f"]
    r = s.motion(np.zeros((1, N), dtype=np.float32))
    assert r["s"] == w["s_min"] and np.isnan(r["d"][0])  # first chunk, T=1: no pair
    r = s.motion(np.full((1, N), 3.0, dtype=np.float32))  # d = 3 -> clip to 1
    assert r["dhat"] == 1.0 and abs(r["s"] - w["s_max"]) < 1e-15
    r = s.motion(np.full((1, N), 3.25, dtype=np.float32))  # d = .25, window max still 3
    assert r["dhat"] == 1.0
    r = s.motion(np.full((1, N), 3.5, dtype=np.float32))   # window {.25, .25}
    assert abs(r["dhat"] - 0.25) < 1e-12


def test_lazy_provenance_then_materialize_equals_eager_push():
    """The long-run checks record provenance and build the ring later; the
    result must be the ring an eager push sequence builds (through sink
    fills, refreshes, ring wrap and a RoPE reset)."""
    w = tiny(M=2, T=3, R=6, rope_tau=5, emb_step=0.8, steps=9)
    eager, lazy = O.Stream(w), O.Stream(w)
    lazy.set_lazy(True)
    walk = W.EmbeddingWalk(w)
    chunks = []
    for c in range(9):
        k, v = W.gen_kv(w, c)
        chunks.append((k[0], v[0]))
        eager.push(k[0], v[0])
        lazy.push(k[0], v[0])
        h = walk.next()[0]
        assert eager.sink_refresh(h) == lazy.sink_refresh(h)
    assert eager.meta() == lazy.meta() and eager.meta()["resets"] >= 1
    prov = lazy.provenance()
    TL = w["T"] * w["L"]
    kf = np.zeros((w["M"] + w["R"], w["L"], w["H"], w["d"]), dtype=np.uint16)
    vf = np.zeros_like(kf)
    for f, (c, j, p0) in enumerate(prov):
        if c >= 0:
            kf[f] = chunks[c][0].reshape(w["T"], w["L"], w["H"], w["d"])[j]
            vf[f] = chunks[c][1].reshape(w["T"], w["L"], w["H"], w["d"])[j]
    lazy.materialize(kf, vf)
    ke, ve = eager.kv()
    kl, vl = lazy.kv()
    assert np.array_equal(ke, kl) and np.array_equal(ve, vl)
    assert np.array_equal(eager.emb(), lazy.emb())


# --------------------------------------------------------------- guidance / update variants

def _slot_inputs(w, rng):
    n, N = w["n"], w["N_s"]
    return dict(x=rng.standard_normal((n, N)).astype(np.float32),
                x0=rng.standard_normal((n, N)).astype(np.float32),
                eps_c=rng.standard_normal((n, N)).astype(np.float32),
                z=rng.standard_normal((max(n - 1, 1), N)).astype(np.float32)[: max(n - 1, 0)],
                x0_new=rng.standard_normal(N).astype(np.float32),
                eps_new=rng.standard_normal(N).astype(np.float32),
                eps_neg=rng.standard_normal((n, N)).astype(np.float32))


def test_supplied_negative_with_delta_one_is_standard_cfg():
    """cfg_type 2, delta = 1, eps_neg = the unconditional prediction eps_u:
    eps_cfg must be eps_u + gamma (eps_c - eps_u), seen through x0hat of the
    completed slot."""
    w = tiny(cfg_type=2, delta=1.0, gamma=1.7, n=2)
    st = O.Stream(w)
    d = _slot_inputs(w, np.random.default_rng(3))
    xn, out = st.step_update(d["x"], d["x0"], d["eps_c"], d["z"], d["x0_new"], d["eps_new"],
                             eps_neg=d["eps_neg"])
    ab = O.alpha_bar(w)[O.slot_timestep(w, 1)]
    eu, ec, x = (d[k][1].astype(np.float64) for k in ("eps_neg", "eps_c", "x"))
    cfg = eu + 1.7 * (ec - eu)
    assert np.allclose(out, (x - math.sqrt(1 - ab) * cfg) / math.sqrt(ab), rtol=1e-12, atol=1e-12)


def test_supplied_virtual_residual_reproduces_self_negative():
    """Feeding the virtual residual as the supplied negative gives the
    self-negative result: the two guidance paths use eps_neg in one role."""
    d = _slot_inputs(tiny(n=2), np.random.default_rng(4))
    w_self, w_sup = tiny(n=2, cfg_type=1), tiny(n=2, cfg_type=2)
    ab = O.alpha_bar(w_self)
    res = np.stack([(d["x"][i].astype(np.float64) - math.sqrt(ab[O.slot_timestep(w_self, i)]) * d["x0"][i])
                    / math.sqrt(1 - ab[O.slot_timestep(w_self, i)]) for i in range(2)])
    a = O.Stream(w_self).step_update(d["x"], d["x0"], d["eps_c"], d["z"], d["x0_new"], d["eps_new"])
    # the residual rounds to float32 on its way in: compare within that rounding
    b = O.Stream(w_sup).step_update(d["x"], d["x0"], d["eps_c"], d["z"], d["x0_new"], d["eps_new"],
                                    eps_neg=res.astype(np.float32))
    assert np.allclose(a[0], b[0], rtol=1e-6, atol=1e-6) and np.allclose(a[1], b[1], rtol=1e-6, atol=1e-6)


def test_ddpm_update_mean_is_the_posterior_mean():
    """update_kind 1 with the true noise and z = 0 lands on the DDPM posterior
    mean of q(x_t' | x_t, x0) written in its x0 / x_t form."""
    w = tiny(n=2, cfg_type=0, update_kind=1)
    rng = np.random.default_rng(5)
    N = w["N_s"]
    ab = O.alpha_bar(w)
    t0, t1 = O.slot_timestep(w, 0), O.slot_timestep(w, 1)
    a_t, a_n = ab[t0], ab[t1]
    x0 = rng.standard_normal((2, N))
    eps = rng.standard_normal((2, N))
    xt = np.sqrt(np.array([a_t, ab[t1]]))[:, None] * x0 + np.sqrt(1 - np.array([a_t, ab[t1]]))[:, None] * eps
    f32 = lambda v: v.astype(np.float32)
    xt32, eps32, x032 = f32(xt), f32(eps), f32(x0)
    xn, _ = O.Stream(w).step_update(xt32, x032, eps32, np.zeros((1, N), np.float32),
                                    f32(x0[0]), f32(eps[0]))
    al = a_t / a_n
    mu = (math.sqrt(a_n) * (1 - al) / (1 - a_t)) * x032[0].astype(np.float64) + \
         (math.sqrt(al) * (1 - a_n) / (1 - a_t)) * xt32[0].astype(np.float64)
    # the true noise of the rounded x_t differs from eps by the rounding: loose on that
    assert np.allclose(xn[1], mu, rtol=0, atol=5e-6)


def test_ddpm_adjacent_step_noise_scale_is_beta_tilde():
    """With adjacent timesteps the noise scale of update_kind 1 is the DDPM
    posterior standard deviation sqrt((1 - abar_{t-1}) / (1 - abar_t) beta_t),
    beta_t taken straight from the scaled-linear definition."""
    w = tiny(n=2, cfg_type=0, update_kind=1, n_inf=1000, t_index=[5, 6])
    t0, t1 = O.slot_timestep(w, 0), O.slot_timestep(w, 1)
    assert t0 - t1 == 1
    N = w["N_s"]
    x = np.ones((2, N), np.float32)
    e = np.zeros((2, N), np.float32)
    z1 = np.ones((1, N), np.float32)
    st = O.Stream(w)
    a = st.step_update(x, x, e, z1, x[0], e[0])[0][1]
    b = st.step_update(x, x, e, np.zeros_like(z1), x[0], e[0])[0][1]
    sb, eb = math.sqrt(w["beta_start"]), math.sqrt(w["beta_end"])
    beta = (sb + t0 * (eb - sb) / (w["n_train"] - 1)) ** 2
    ab = O.alpha_bar(w)
    sigma = math.sqrt((1 - ab[t1]) / (1 - ab[t0]) * beta)
    assert np.allclose(a - b, sigma, rtol=1e-10)


# --------------------------------------------------------------- noise-rate application

def test_noise_rate_sets_the_entry_timestep_and_the_next_update_uses_it():
    """With the rate at s_min (no motion yet) and one slot (nothing below
    slot 0), the incoming frame enters at round(s_min (N - 1)); next step the
    frame in slot 0 is treated at that timestep: built from its x0 and true
    noise at that level, it predicts x0."""
    w = tiny(n=1, T=1, noise_rate_on=1, cfg_type=0, s_min=0.3, s_max=0.9)
    st = O.Stream(w)
    N = w["N_s"]
    rng = np.random.default_rng(9)
    x0 = rng.standard_normal(N).astype(np.float32)
    eps = rng.standard_normal(N).astype(np.float32)
    t_entry = int(math.floor(0.3 * (w["n_train"] - 1) + 0.5))
    assert t_entry == 300
    one = lambda a: a[None, :]
    xn, _ = st.step_update(one(x0), one(x0), one(eps), np.zeros((0, N), np.float32), x0, eps)
    assert st.slot0_timestep() == t_entry
    ab = O.alpha_bar(w)[t_entry]
    expect = math.sqrt(ab) * x0.astype(np.float64) + math.sqrt(1 - ab) * eps.astype(np.float64)
    assert np.allclose(xn[0], expect, rtol=1e-12, atol=1e-12)
    # the frame now in slot 0 (x at t_entry, its noise known) completes to its x0
    xt = xn[0].astype(np.float32)
    _, out = st.step_update(one(xt), one(x0), one(eps), np.zeros((0, N), np.float32), x0, eps)
    assert np.allclose(out, x0, atol=2e-6)


def test_noise_rate_follows_motion_into_the_entry_timestep():
    """A burst that clips the motion to 1 drives the rate toward s_max, and
    the next incoming frame enters the fraction `rate` of the way from slot
    1's timestep (99 for t_index [32, 45]) to N - 1."""
    w = tiny(n=2, T=1, noise_rate_on=1, mot_k=1, sigma=1.0, lam=0.5)
    st = O.Stream(w)
    N, Nf = w["N_s"], w["N_f"]
    z = lambda *sh: np.zeros(sh, np.float32)
    st.motion(z(1, Nf))
    st.motion(np.full((1, Nf), 5.0, np.float32))         # d = 5 -> dhat = 1
    s = st.noise_rate()
    assert abs(s - (0.3 + 0.5 * (0.9 - 0.3))) < 1e-12    # one EMA step of lambda = 0.5 toward s_max
    st.step_update(z(2, N), z(2, N), z(2, N), z(1, N), z(N), z(N))
    t1 = O.slot_timestep(w, 1)
    assert t1 == 99
    assert st.slot0_timestep() == t1 + int(math.floor(s * (w["n_train"] - 1 - t1) + 0.5))


def test_entry_timestep_keeps_the_stream_batch_in_descending_order():
    """StreamDiffusion notes, "Stream Batch": the n slots hold frames at
    descending timesteps, each frame one denoise step further than the one
    before it.  Whatever rate the motion sets, the incoming frame must not be
    less noisy than the frame in slot 1: for the four-slot schedule
    999 / 679 / 359 / 99 the entry timestep runs from 679 (rate 0) to 999
    (rate 1), never decreasing as the rate grows.  (lambda = 0 makes the
    rate equal its target, s_min = 0 and s_max = 1 make the target the
    clipped motion itself, and a constant shift c has motion |c|.)"""
    w = tiny(n=4, t_index=[0, 16, 32, 45], T=1, noise_rate_on=1, mot_k=1, sigma=1.0, lam=0.0,
             s_min=0.0, s_max=1.0, cfg_type=0)
    assert [O.slot_timestep(w, i) for i in range(4)] == [999, 679, 359, 99]
    N, Nf = w["N_s"], w["N_f"]
    zeros = lambda *sh: np.zeros(sh, np.float32)
    last = -1
    for c in (0.0, 0.05, 0.25, 0.5, 0.75, 0.95, 1.0, 3.0):
        st = O.Stream(w)
        st.motion(zeros(1, Nf))
        st.motion(np.full((1, Nf), c, np.float32))  # d = |c|
        assert abs(st.noise_rate() - min(float(np.float32(c)), 1.0)) < 1e-12
        st.step_update(zeros(4, N), zeros(4, N), zeros(4, N), zeros(3, N), zeros(N), zeros(N))
        t = st.slot0_timestep()
        assert 679 <= t <= 999 and t >= last, (c, t)
        last = t
        if c == 0.0:
            assert t == 679
        if c >= 1.0:
            assert t == 999
        st.close()


# --------------------------------------------------------------- txt2img

def test_txt2img_incoming_frame_is_the_noise_draw_and_matches_an_equivalent_img2img_frame():
    """With no input image the incoming latent is the N(0, I) draw itself.
    The same latent arises in img2img from the input x0 = eps (1 - sqrt(1 -
    abar_0)) / sqrt(abar_0), so the two paths agree on everything else."""
    w = tiny(n=2, cfg_type=0, txt2img=1)
    N = w["N_s"]
    rng = np.random.default_rng(11)
    x, x0, ec = (rng.standard_normal((2, N)).astype(np.float32) for _ in range(3))
    z = rng.standard_normal((1, N)).astype(np.float32)
    eps = rng.standard_normal(N).astype(np.float32)
    xn_t, out_t = O.Stream(w).step_update(x, x0, ec, z, None, eps)
    assert np.array_equal(xn_t[0], eps.astype(np.float64))
    ab0 = O.alpha_bar(w)[(w["n_train"] - 1) - w["t_index"][0] * (w["n_train"] // w["n_inf"])]
    x0_equiv = eps.astype(np.float64) * (1 - math.sqrt(1 - ab0)) / math.sqrt(ab0)
    xn_i, out_i = O.Stream(dict(w, txt2img=0)).step_update(x, x0, ec, z, x0_equiv.astype(np.float32), eps)
    assert np.allclose(xn_i[0], eps, rtol=0, atol=1e-6)   # up to the fp32 rounding of x0_equiv
    assert np.array_equal(xn_i[1], xn_t[1]) and np.array_equal(out_i, out_t)
