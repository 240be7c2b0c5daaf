"""Checkpoints on the device: a context restored from sds_state_export
continues exactly like the one it was taken from (bit-identical attention,
update, decisions and ring), a checkpoint without K/V restores everything
but the ring, and a corrupted checkpoint changes nothing."""
import numpy as np
import pytest
import torch

from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import GpuPipe

pytestmark = pytest.mark.gpu


def drive(g: GpuPipe, w, step, emb, lat_walk, frames):
    k, v = W.gen_kv(w, step)
    g.push(k, v)
    g.refresh(emb[step])
    att = g.attend(W.gen_q(w, step))
    xn, out = g.step(W.gen_latents(w, step), frames[step], W.gen_u(w, step), lat_walk[step])
    return att, xn, out


def inputs(w, steps):
    ew, lw, fw = W.EmbeddingWalk(w), W.LatentWalk(w), W.FrameWalk(w)
    return ([ew.next() for _ in range(steps)], [lw.next() for _ in range(steps)],
            [fw.next() for _ in range(steps)])


def same_states(x, y) -> bool:
    """Per-stream records equal field by field (NaN marks an absent motion pair)."""
    if len(x) != len(y):
        return False
    for a, b in zip(x, y):
        if a.keys() != b.keys():
            return False
        for k in a:
            if not np.array_equal(np.asarray(a[k]), np.asarray(b[k]), equal_nan=True):
                return False
    return True


@pytest.mark.parametrize("name,over", [
    ("c1_tiny", dict(streams=2, M=2, T=3, R=6, mot_k=3, emb_step=0.5)),
    ("c1_tiny", dict(rope_tau=3)),
])
def test_restored_context_continues_identically(name, over):
    w = W.get_config(name, **over)
    steps = 9
    emb, lat, frames = inputs(w, steps)
    a, b = GpuPipe(w), GpuPipe(w)
    try:
        for s in range(5):
            drive(a, w, s, emb, lat, frames)
        ck = B.sds_state_export(a.ctx, with_kv=True)
        B.sds_state_check(B.config_from_workload(w), ck)
        B.sds_state_import(b.ctx, ck)
        assert b.meta() == a.meta()
        assert same_states(b.state(), a.state())
        for s in range(5, steps):
            ra, rb = drive(a, w, s, emb, lat, frames), drive(b, w, s, emb, lat, frames)
            assert np.array_equal(ra[0], rb[0]), s      # attention, bitwise
            assert np.array_equal(ra[1], rb[1]), s      # next latents
            assert np.array_equal(ra[2], rb[2]), s      # completed frame
            assert same_states(a.state(), b.state()), s
        for x, y in zip(a.kv(), b.kv()):
            assert np.array_equal(x, y)
        assert np.array_equal(a.sink_emb(), b.sink_emb())
        # the two contexts now export the same bytes
        assert B.sds_state_export(a.ctx) == B.sds_state_export(b.ctx)
    finally:
        a.close()
        b.close()


def test_checkpoint_without_kv_and_rejected_imports():
    w = W.get_config("c1_tiny", streams=2)
    emb, lat, frames = inputs(w, 4)
    a, b = GpuPipe(w), GpuPipe(w)
    try:
        for s in range(4):
            drive(a, w, s, emb, lat, frames)
        full = B.sds_state_export(a.ctx, with_kv=True)
        small = B.sds_state_export(a.ctx, with_kv=False)
        assert len(full) > len(small)
        before = B.sds_state_export(b.ctx, with_kv=True)
        # corrupted: rejected, b unchanged
        bad = bytearray(small)
        bad[200] ^= 1
        with pytest.raises(B.SdsError) as e:
            B.sds_state_import(b.ctx, bytes(bad))
        assert e.value.status == B.SDS_ERR_STATE
        assert B.sds_state_export(b.ctx, with_kv=True) == before
        # a checkpoint of another configuration: rejected
        other = GpuPipe(W.get_config("c1_tiny", streams=2, gamma=1.2))
        try:
            with pytest.raises(B.SdsError):
                B.sds_state_import(other.ctx, small)
        finally:
            other.close()
        # without K/V: metadata and records restored, ring untouched (still zero)
        B.sds_state_import(b.ctx, small)
        assert b.meta() == a.meta() and same_states(b.state(), a.state())
        assert np.array_equal(b.sink_emb(), a.sink_emb())
        assert all(not np.any(x) for x in b.kv())
        # a buffer too small for the export is refused with the size needed
        import ctypes as C
        n = C.c_size_t(10)
        assert B.lib().sds_state_export(a.ctx, C.create_string_buffer(10), C.byref(n), 1,
                                        None) == B.SDS_ERR_INVALID_ARG
        assert n.value == len(full)
        torch.cuda.synchronize()
    finally:
        a.close()
        b.close()
