"""Failure detection on the GPU without a fault: K1's bounded waits.

Every wait of the attention kernel on a barrier has a time limit.  The test
hook sds_test_attn_timeout shortens the limit to 1 ms and makes CTA 0 skip
the copy of one key tile, so the waits for it run out.  The launch must
return on its own (no hang, no CUDA error), record the timeout in the
stream's error word, and leave the context usable: the next launch, with
the hook off, must match the oracle again.
"""
import time

import numpy as np
import pytest
import torch

from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import GpuPipe, OraclePipe, attn_rel_err

pytestmark = pytest.mark.gpu

ERR_ATTN_WAIT_TIMEOUT = 1


@pytest.mark.parametrize("d", [64, 128])
def test_attention_wait_runs_out_reports_and_the_context_recovers(d):
    w = W.get_config("c1_tiny", d=d, steps=2)
    g, o = GpuPipe(w), OraclePipe(w)
    try:
        k, v = W.gen_kv(w, 0)
        g.push(k, v)
        o.push(k, v)
        h = W.EmbeddingWalk(w).next()
        g.refresh(h)
        o.refresh(h)
        q = W.gen_q(w, 0)
        ref = o.attend(q)
        assert attn_rel_err(g.attend(q)[0], ref[0]) <= 2e-2
        assert g.state()[0]["error_word"] == 0

        B.sds_test_attn_timeout(g.ctx, 1_000_000, 0)  # 1 ms; CTA 0 never loads key tile 0
        t0 = time.perf_counter()
        g.attend(q)  # synchronises: the launch ended by itself
        elapsed = time.perf_counter() - t0
        torch.cuda.synchronize()
        assert elapsed < 1.0, elapsed
        assert g.state()[0]["error_word"] & ERR_ATTN_WAIT_TIMEOUT

        B.sds_test_attn_timeout(g.ctx, 0, -1)  # back to the default limit, nothing withheld
        for _ in range(2):
            assert attn_rel_err(g.attend(q)[0], ref[0]) <= 2e-2
        # the other kernels of the context still run and agree with the oracle
        lat = W.gen_latents(w, 0)
        xn, out = g.step(lat)
        (xr, outr), = o.step(lat)
        assert np.max(np.abs(out[0] - outr)) <= 1e-5 * max(np.max(np.abs(outr)), 1.0)
    finally:
        g.close()


def test_timeout_hook_rejects_bad_arguments():
    w = W.get_config("c1_tiny")
    g = GpuPipe(w)
    try:
        for bad in ((-1, 0), (3_000_000_000, 0), (1000, -2)):
            with pytest.raises(B.SdsError) as e:
                B.sds_test_attn_timeout(g.ctx, *bad)
            assert e.value.status == B.SDS_ERR_INVALID_ARG
    finally:
        g.close()
