"""Checkpoint validation on the host (no device): sds_state_check accepts a
buffer laid out as include/sds.h documents and rejects every corruption
before anything would reach a device -- a flipped payload byte, a wrong
magic, version or configuration, a truncated or resized buffer, and
metadata out of range."""
import ctypes as C
import struct

import numpy as np
import pytest

from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W


def fnv1a(data: bytes) -> int:
    h = 14695981039346656037
    for byte in data:
        h ^= byte
        h = (h * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h


def layout(w, with_kv):
    S = w["streams"]
    emb = S * w["M"] * w["D"]
    ssf = 2 * S * w["ssf_E"] if w["ssf"] else 0
    mot = 2 * S * w["N_f"] if w["motion"] else 0
    kv = S * (w["M"] + w["R"]) * w["L"] * w["HD"]
    sizes = [128, S * B.SDS_STATE_RECORD_BYTES, 4 * emb, 4 * ssf, 4 * mot]
    if with_kv:
        sizes += [2 * kv, 2 * kv]
    return dict(emb=emb, ssf=ssf, mot=mot, kv=kv, payload=sum(sizes))


def build(cfg, w, with_kv=True, meta=(12, 4, 3, 11, 1, 2, 12, 12, 12), seed=0):
    L = layout(w, with_kv)
    rng = np.random.default_rng(seed)
    payload = bytearray(rng.integers(0, 256, L["payload"], dtype=np.uint8).tobytes())
    payload[:128] = struct.pack("<16q", *(tuple(meta) + (0,) * (16 - len(meta))))
    h = B.sds_state_header()
    h.magic = B.SDS_STATE_MAGIC
    h.abi_version = B.SDS_ABI_VERSION
    h.config_hash = fnv1a(bytes(cfg))
    h.flags = 1 if with_kv else 0
    h.payload_bytes = L["payload"]
    h.payload_hash = fnv1a(bytes(payload))
    h.streams = w["streams"]
    h.devstate_bytes = B.SDS_STATE_RECORD_BYTES
    h.emb_elems, h.ssf_ref_elems, h.mot_prev_elems, h.kv_elems = L["emb"], L["ssf"], L["mot"], L["kv"]
    return bytes(h) + bytes(payload)


@pytest.fixture()
def setup():
    w = W.get_config("c1_tiny", streams=2)
    return w, B.config_from_workload(w)


def test_header_is_128_bytes():
    assert C.sizeof(B.sds_state_header) == 128


@pytest.mark.parametrize("with_kv", [True, False])
def test_well_formed_checkpoint_is_accepted(setup, with_kv):
    w, cfg = setup
    B.sds_state_check(cfg, build(cfg, w, with_kv))


def expect_reject(cfg, data, what):
    with pytest.raises(B.SdsError) as e:
        B.sds_state_check(cfg, data)
    assert e.value.status == B.SDS_ERR_STATE
    assert what in B.sds_last_error()


def test_every_corruption_is_rejected(setup):
    w, cfg = setup
    good = build(cfg, w)
    flipped = bytearray(good)
    flipped[128 + 128 + 5] ^= 0x10                    # one payload bit
    expect_reject(cfg, bytes(flipped), "hash")
    bad_magic = b"XDSSTAT1" + good[8:]
    expect_reject(cfg, bad_magic, "magic")
    expect_reject(cfg, good[:-1], "truncated")
    expect_reject(cfg, good[:100], "shorter than its header")
    other = B.config_from_workload(dict(w, gamma=1.5))
    expect_reject(other, good, "different configuration")
    h = B.sds_state_header.from_buffer_copy(good[:128])
    h.abi_version = 1
    expect_reject(cfg, bytes(h) + good[128:], "ABI version")
    h = B.sds_state_header.from_buffer_copy(good[:128])
    h.devstate_bytes = 712
    expect_reject(cfg, bytes(h) + good[128:], "section sizes")
    # metadata out of range, with a valid hash: more sinks filled than exist
    expect_reject(cfg, build(cfg, w, meta=(12, 4, 3, 11, 5, 2, 12, 12, 12)), "metadata")
    # reserved metadata words must be zero
    expect_reject(cfg, build(cfg, w, meta=(12, 4, 3, 11, 1, 2, 12, 12, 12, 7)), "metadata")


def test_null_buffer_is_an_argument_error(setup):
    w, cfg = setup
    assert B.lib().sds_state_check(C.byref(cfg), None, 0) == B.SDS_ERR_INVALID_ARG
