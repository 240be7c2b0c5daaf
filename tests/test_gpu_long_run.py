"""The long-run stress case at the 1.3B-DiT shape: 10,000 chunks on two
concurrent streams, with random-walk latents whose chunks take a x20 step
5 % of the time, sink refreshes from a drifting embedding walk and RoPE
resets every ~1024 frames.

Every chunk: the sink decision (index and fire / no fire; bit-exact unless
the oracle flags a near tie) and the noise rate (within 1e-5) against the
oracle.  Every 500 chunks: the host metadata, the exported checkpoint's
ring and sinks (V bit-exact, rotated K within the RoPE bound, embeddings
bit-exact) and sampled attention rows (within 2e-2) against the oracle.
The oracle runs in its lazy mode: pushes record which chunk frame each key
frame holds and the ring is rebuilt with the oracle's push arithmetic at
each check.  K/V chunks cycle through a pool of four, so the ring keeps
changing while the inputs stay on the device.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W
from tests.harness import attn_rel_err, bf16_dev, bf16_host, f32_dev, rope_k_excess

pytestmark = pytest.mark.gpu

POOL = 4
CHECK_EVERY = 500


def export_kv(ctx, w):
    """Ring and sinks as read back from a checkpoint (not from the live buffers)."""
    data = B.sds_state_export(ctx, with_kv=True)
    B.sds_state_check(B.config_from_workload(w), data)
    h = B.sds_state_header.from_buffer_copy(data[:128])
    n_kv = h.kv_elems
    off = 128 + h.payload_bytes - 4 * n_kv
    sh = (w["streams"], (w["M"] + w["R"]) * w["L"], w["H"], w["d"])
    k = np.frombuffer(data, dtype=np.uint16, count=n_kv, offset=off).reshape(sh)
    v = np.frombuffer(data, dtype=np.uint16, count=n_kv, offset=off + 2 * n_kv).reshape(sh)
    emb_off = 128 + 128 + w["streams"] * B.SDS_STATE_RECORD_BYTES
    emb = np.frombuffer(data, dtype=np.float32, count=h.emb_elems, offset=emb_off)
    return k, v, emb.reshape(w["streams"], w["M"], w["D"])


def test_c5_ten_thousand_chunks_checked_every_500():
    w = W.get_config("c5_stress", streams=2)
    S, n, chunks = w["streams"], w["n"], w["steps"]
    assert chunks == 10000
    pool = [W.gen_kv(w, i) for i in range(POOL)]
    pool_dev = [(bf16_dev(k), bf16_dev(v)) for k, v in pool]
    q_bits = W.gen_q(w, 0)
    q = bf16_dev(q_bits)
    o = torch.empty((S, w["q_rows"], w["H"], w["d"]), dtype=torch.bfloat16, device="cuda")
    lat = W.gen_latents(w, 0)
    dev = {k: f32_dev(v) for k, v in lat.items() if k != "z"}
    z = [f32_dev(lat["z"][i]) for i in range(n - 1)]
    x_next = [torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda") for _ in range(n)]
    out = torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda")
    ctx = B.sds_create(B.config_from_workload(w))
    oracle = [O.Stream(w) for _ in range(S)]
    for st in oracle:
        st.set_lazy(True)
    emb, walk = W.EmbeddingWalk(w), W.LatentWalk(w)
    fires = bursts_seen = checks = near = 0
    TL = w["T"] * w["L"]
    try:
        for c in range(chunks):
            k_bits, v_bits = pool[c % POOL]
            kd, vd = pool_dev[c % POOL]
            B.sds_kv_push(ctx, kd, vd)
            h = emb.next()
            hd = f32_dev(h)
            B.sds_sink_refresh(ctx, hd)
            chunk = walk.next()
            cd = f32_dev(chunk)
            io = B.make_step_io([dev["x"][i] for i in range(n)], [dev["x0"][i] for i in range(n)],
                                [dev["eps_c"][i] for i in range(n)], z, x_next, out,
                                dev["x0_new"], dev["eps_new"], None, None, cd)
            B.sds_step_update(ctx, io)
            ref_sink, ref_mot = [], []
            for s, st in enumerate(oracle):
                st.push(k_bits[s], v_bits[s])
                ref_sink.append(st.sink_refresh(h[s]))
                ref_mot.append(st.motion(chunk[s]))
            got = B.sds_read_state(ctx, S)
            for s in range(S):
                r, g = ref_sink[s], got[s]
                if r["near"]:
                    near += 1
                else:
                    assert (g["sink_j"], g["sink_fire"]) == (r["j"], r["fire"]), (c, s, g, r)
                    fires += r["fire"] == 1
                assert abs(g["noise_rate"] - ref_mot[s]["s"]) <= 1e-5, (c, s)
                assert g["error_word"] == 0
                bursts_seen += ref_mot[s]["dhat"] >= 1.0
            if (c + 1) % CHECK_EVERY:
                continue
            checks += 1
            m, om = B.sds_get_meta(ctx), oracle[0].meta()
            assert (m["frames_pushed"], m["rope_offset"], m["chunk_p0"], m["ring_valid"],
                    m["sinks_filled"], m["rope_resets"]) == \
                (om["F"], om["o"], om["p0"], om["valid"], om["sinks_filled"], om["resets"]), c
            gk, gv, gemb = export_kv(ctx, w)
            B.sds_attend(ctx, q, o)
            torch.cuda.synchronize()
            got_o = W.bf16_bits_to_f32(bf16_host(o)).astype(np.float64)
            rows = np.unique(np.concatenate([[0, TL - 1, TL, w["q_rows"] - 1],
                                             np.random.default_rng(c).choice(w["q_rows"], 12)]))
            for s, st in enumerate(oracle):
                prov = st.provenance()
                frames = (w["M"] + w["R"], w["L"], w["H"], w["d"])
                kf = np.zeros(frames, dtype=np.uint16)
                vf = np.zeros(frames, dtype=np.uint16)
                for f, (src, j, _) in enumerate(prov):
                    if src >= 0:
                        pk, pv = pool[src % POOL]
                        kf[f] = pk[s].reshape(w["T"], w["L"], w["H"], w["d"])[j]
                        vf[f] = pv[s].reshape(w["T"], w["L"], w["H"], w["d"])[j]
                st.materialize(kf, vf)
                ok_, ov_ = st.kv()
                assert np.array_equal(gv[s], ov_), (c, s)
                assert rope_k_excess(gk[s], ok_) <= 1.0, (c, s)
                filled = st.meta()["sinks_filled"]
                assert np.array_equal(gemb[s][:filled].astype(np.float64), st.emb()[:filled]), (c, s)
                ref_o = st.attend(q_bits[s], rows)
                assert attn_rel_err(got_o[s][rows], ref_o) <= 2e-2, (c, s)
        assert checks == chunks // CHECK_EVERY
        assert oracle[0].meta()["resets"] >= 25       # ~29 resets over 30,000 frames
        assert fires >= 10 and bursts_seen >= 10
    finally:
        B.sds_destroy(ctx)
        for st in oracle:
            st.close()
