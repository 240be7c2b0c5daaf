"""The allocation-free similarity filter, sds_ssf_noalloc, against sds_ssf.

sds_ssf_noalloc serves callers that cannot allocate device memory (a fixed
budget owned by another allocator, or a loop where cudaMalloc/cudaFree must
not run), so they cannot create a context.  It keeps its scratch in a static
device array.  Here it is called through the C ABI twice in a row on new
frames and must give what the context path gives for the same frame and
reference: the cosine within the 1e-6 used by the other SSF tests, the same
probability within 5e-5 and the same skip decision.  This file is collected
last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W

pytestmark = pytest.mark.gpu


def test_noalloc_matches_context_path_on_two_calls():
    w = W.get_config("c2_sdturbo_image", streams=2)
    S, E = w["streams"], w["ssf_E"]
    ctx = B.sds_create(B.config_from_workload(w))
    try:
        walk = W.FrameWalk(w)
        first = torch.from_numpy(walk.next()).cuda()
        u0 = torch.zeros(S, dtype=torch.float32, device="cuda")
        B.sds_ssf(ctx, first, u0)  # first frame: processed, becomes the reference
        ref = first.clone()
        cos_o = torch.empty(S, dtype=torch.float64, device="cuda")
        p_o = torch.empty(S, dtype=torch.float64, device="cuda")
        skip_o = torch.empty(S, dtype=torch.int64, device="cuda")
        for call in range(2):
            frame = torch.from_numpy(walk.next()).cuda()
            u = torch.from_numpy(W.gen_u(w, 50 + call)).cuda()
            before = B.sds_read_state(ctx, S)
            count = torch.tensor([st["ssf_skip_count"] for st in before], dtype=torch.int64,
                                 device="cuda")
            B.sds_ssf_noalloc(frame, ref, u, count, S, E, w["eta"], w["max_skip"], cos_o, p_o,
                              skip_o)
            B.sds_ssf(ctx, frame, u)
            after = B.sds_read_state(ctx, S)
            torch.cuda.synchronize()
            got_cos, got_p, got_skip = cos_o.cpu().numpy(), p_o.cpu().numpy(), skip_o.cpu().numpy()
            for s in range(S):
                assert abs(got_cos[s] - after[s]["ssf_cos"]) <= 1e-6, (call, s)
                assert abs(got_p[s] - after[s]["ssf_p"]) <= 5e-5, (call, s)
                assert got_skip[s] == after[s]["ssf_skip"], (call, s)
            # the context keeps a processed frame as its reference; mirror that
            keep = torch.tensor([st["ssf_skip"] == 0 for st in after], device="cuda")
            ref = torch.where(keep[:, None], frame, ref)
    finally:
        B.sds_destroy(ctx)


def test_noalloc_rejects_requests_beyond_its_scratch():
    S, E = 29, 3 * 512 * 512  # 29 * 384 * 3 partials > 32736
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    o = torch.zeros(S, dtype=torch.float64, device="cuda")
    k = torch.zeros(S, dtype=torch.int64, device="cuda")
    with pytest.raises(B.SdsError) as e:
        B.sds_ssf_noalloc(t, t, t, None, S, E, 0.98, 10, o, o, k)
    assert e.value.status == B.SDS_ERR_INVALID_ARG
    assert "SDS_NOALLOC_MAX_PARTIALS" in B.sds_last_error()
