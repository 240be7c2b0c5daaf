"""The allocation-free similarity filter, sds_ssf_noalloc.

sds_ssf_noalloc serves callers that cannot allocate device memory (a fixed
budget owned by another allocator, or a loop where cudaMalloc/cudaFree must
not run), so they cannot create a context.  It keeps its scratch in a static
device array and runs K4's filter reduction unchanged.  Here it is called
through the C ABI: twice in a row on new frames it must give bit for bit
what the context path (sds_ssf) records for the same frame, reference, draw
and skip count, and agree with the oracle within the bars of the other
filter tests (cosine 1e-6, probability 5e-5, the skip decision unless the
oracle flags a near tie).  Further cases: identical frames (P exactly 1),
frame sizes that are not a multiple of the 8192-element work block, a NULL
skip count, a count at the cap, and a request at the scratch limit.  This
file is collected last so that a failure here leaves every other test
already run.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_PARTIALS = 32736
BLOCK = 8192


def _outs(S):
    return (torch.empty(S, dtype=torch.float64, device="cuda"),
            torch.empty(S, dtype=torch.float64, device="cuda"),
            torch.empty(S, dtype=torch.int64, device="cuda"))


def _call(frame, ref, u, count, S, E, eta, max_skip):
    c, p, k = _outs(S)
    B.sds_ssf_noalloc(frame, ref, u, count, S, E, eta, max_skip, c, p, k)
    torch.cuda.synchronize()
    return c.cpu().numpy(), p.cpu().numpy(), k.cpu().numpy()


def _oracle(w, ref_np, frame_np, u_np):
    """The oracle's filter on `frame` with `ref` as the reference (the first
    frame a stream sees is processed and becomes its reference)."""
    out = []
    for s in range(ref_np.shape[0]):
        st = O.Stream(w)
        st.ssf(ref_np[s], 0.0)
        out.append(st.ssf(frame_np[s], float(u_np[s])))
        st.close()
    return out


def test_noalloc_matches_context_path_bit_for_bit_and_the_oracle_on_two_calls():
    w = W.get_config("c2_sdturbo_image", streams=2)
    S, E = w["streams"], w["ssf_E"]
    ctx = B.sds_create(B.config_from_workload(w))
    try:
        walk = W.FrameWalk(w)
        first_np = walk.next()
        first = torch.from_numpy(first_np).cuda()
        B.sds_ssf(ctx, first, torch.zeros(S, dtype=torch.float32, device="cuda"))
        ref, ref_np = first.clone(), first_np
        for call in range(2):
            frame_np = walk.next()
            u_np = W.gen_u(w, 50 + call)
            frame, u = torch.from_numpy(frame_np).cuda(), torch.from_numpy(u_np).cuda()
            before = B.sds_read_state(ctx, S)
            count = torch.tensor([st["ssf_skip_count"] for st in before], dtype=torch.int64,
                                 device="cuda")
            got_cos, got_p, got_skip = _call(frame, ref, u, count, S, E, w["eta"], w["max_skip"])
            B.sds_ssf(ctx, frame, u)
            after = B.sds_read_state(ctx, S)
            orc = _oracle(w, ref_np, frame_np, u_np)
            for s in range(S):
                assert got_cos[s] == after[s]["ssf_cos"], (call, s)
                assert got_p[s] == after[s]["ssf_p"], (call, s)
                assert got_skip[s] == after[s]["ssf_skip"], (call, s)
                assert abs(got_cos[s] - orc[s]["cos"]) <= 1e-6, (call, s)
                assert abs(got_p[s] - orc[s]["p"]) <= 5e-5, (call, s)
                if not orc[s]["near"] and before[s]["ssf_skip_count"] == 0:
                    assert got_skip[s] == orc[s]["skip"], (call, s)
            # the context keeps a processed frame as its reference; mirror that
            keep = np.array([st["ssf_skip"] == 0 for st in after])
            ref = torch.where(torch.from_numpy(keep).cuda()[:, None], frame, ref)
            ref_np = np.where(keep[:, None], frame_np, ref_np)
    finally:
        B.sds_destroy(ctx)


def test_noalloc_identical_frames_null_count_and_the_cap():
    """I == R: cosine and P exactly 1; with skip_count NULL (all 0) every
    draw u < 1 skips; with a count equal to max_skip nothing skips."""
    w = W.get_config("c1_tiny", streams=3)
    S, E = 3, w["ssf_E"]
    f = torch.from_numpy(W.FrameWalk(w).next()).cuda()
    top = np.float32(np.nextafter(np.float32(1.0), np.float32(0.0)))
    u = torch.tensor([0.0, 0.5, top], dtype=torch.float32, device="cuda")
    c, p, k = _call(f, f, u, None, S, E, 0.98, 10)
    assert np.all(c == 1.0) and np.all(p == 1.0) and np.all(k == 1)
    at_cap = torch.full((S,), 10, dtype=torch.int64, device="cuda")
    c, p, k = _call(f, f, u, at_cap, S, E, 0.98, 10)
    assert np.all(p == 1.0) and np.all(k == 0)
    below = torch.full((S,), 9, dtype=torch.int64, device="cuda")
    assert np.all(_call(f, f, u, below, S, E, 0.98, 10)[2] == 1)


@pytest.mark.parametrize("E", [4, 12, 2 * BLOCK + 4, 3 * BLOCK])
def test_noalloc_ragged_frame_sizes_against_the_oracle(E):
    """Frames whose size leaves a partly filled last work block (or a single
    float4) reduce like the oracle's plain double sums."""
    w = W.get_config("c1_tiny", streams=2, ssf_c=1, ssf_h=1, ssf_w=E)
    S = 2
    walk = W.FrameWalk(w)
    ref_np, frame_np = walk.next(), walk.next()
    u_np = np.array([0.1, 0.9], dtype=np.float32)
    got = _call(torch.from_numpy(frame_np).cuda(), torch.from_numpy(ref_np).cuda(),
                torch.from_numpy(u_np).cuda(), None, S, E, w["eta"], w["max_skip"])
    orc = _oracle(w, ref_np, frame_np, u_np)
    for s in range(S):
        assert abs(got[0][s] - orc[s]["cos"]) <= 1e-6, (E, s)
        assert abs(got[1][s] - orc[s]["p"]) <= 5e-5, (E, s)
        if not orc[s]["near"]:
            assert got[2][s] == orc[s]["skip"], (E, s)


def test_noalloc_at_the_scratch_limit_and_beyond():
    """S * ceil(E / 8192) * 3 = 32544 <= 32736 for 113 streams of 3x512x512
    frames: accepted and correct (sampled streams against the oracle); 114
    streams exceed the scratch and are rejected before any launch."""
    E = 3 * 512 * 512
    S = MAX_PARTIALS // (3 * (E // BLOCK))
    assert S == 113
    w = W.get_config("c2_sdturbo_image", streams=1)
    walk = W.FrameWalk(w)
    base_ref, base_fr = walk.next()[0], walk.next()[0]
    ref = torch.from_numpy(base_ref).cuda().repeat(S, 1)
    frame = torch.from_numpy(base_fr).cuda().repeat(S, 1)
    frame[7] = ref[7]  # one identical pair among them
    u_np = W.uniform_f32(123, 1, (S,))
    c, p, k = _call(frame, ref, torch.from_numpy(u_np).cuda(), None, S, E, w["eta"], w["max_skip"])
    assert c[7] == 1.0 and p[7] == 1.0 and k[7] == 1
    orc = _oracle(w, base_ref[None], base_fr[None], u_np[:1])[0]
    for s in (0, 56, S - 1):
        assert c[s] == c[0] and p[s] == p[0]  # same data, same bits, whatever the stream
        assert abs(c[s] - orc["cos"]) <= 1e-6 and abs(p[s] - orc["p"]) <= 5e-5
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    o = torch.zeros(S + 1, dtype=torch.float64, device="cuda")
    kk = torch.zeros(S + 1, dtype=torch.int64, device="cuda")
    with pytest.raises(B.SdsError) as e:
        B.sds_ssf_noalloc(t, t, t, None, S + 1, E, 0.98, 10, o, o, kk)
    assert e.value.status == B.SDS_ERR_INVALID_ARG
    assert "SDS_NOALLOC_MAX_PARTIALS" in B.sds_last_error()
