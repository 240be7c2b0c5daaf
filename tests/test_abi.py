"""CPU checks of the C ABI: the library loads, exports every symbol the
header declares, the ctypes structs match the C layout, and invalid
configurations are rejected on the host before any CUDA call."""
import ctypes as C
import os
import re
import subprocess

import pytest

from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import build as sds_build
from streaming_diffusion_stream_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sds.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    sds_build.build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SDS_API\s+[\w\s\*]+?\b(sds_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sds_create", "sds_destroy", "sds_attend", "sds_kv_push", "sds_sink_refresh",
              "sds_step_update", "sds_ssf", "sds_read_state", "sds_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = C.CDLL(B.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(B.SIGNATURES)
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (sds_\w+)", out))
    assert exported == set(declared_functions())
    assert B.sds_abi_version() == B.SDS_ABI_VERSION


def test_struct_layouts_match_the_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "sds.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\\n", sizeof(sds_config), sizeof(sds_step_io),
         sizeof(sds_stream_state), sizeof(sds_meta), sizeof(sds_buffers));
  printf("%zu %zu %zu %zu\\n", offsetof(sds_config, t_index), offsetof(sds_config, rope_base),
         offsetof(sds_step_io, out), offsetof(sds_stream_state, motion_d));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sizes = [int(x) for x in lines[0].split()]
    offs = [int(x) for x in lines[1].split()]
    assert sizes == [C.sizeof(B.sds_config), C.sizeof(B.sds_step_io), C.sizeof(B.sds_stream_state),
                     C.sizeof(B.sds_meta), C.sizeof(B.sds_buffers)]
    assert offs == [B.sds_config.t_index.offset, B.sds_config.rope_base.offset,
                    B.sds_step_io.out.offset, B.sds_stream_state.motion_d.offset]


def _create_status(cfg):
    out = C.c_void_p()
    return B.lib().sds_create(C.byref(cfg), C.byref(out)), out.value


@pytest.mark.parametrize("field,value,msg", [
    ("abi_version", 99, "abi_version"),
    ("head_dim", 96, "head_dim"),
    ("slots_n", 9, "slots_n"),
    ("slots_n", 0, "slots_n"),
    ("ring_R", 0, None),  # image mode with frames_T=1 is valid for c1 shapes? T=1 -> but sink_M=1 invalid
    ("grid_w", 7, "grid_h * grid_w"),
    ("slot_elems", 1022, "slot_elems"),
    ("mot_k", 65, "mot_k"),
    ("cfg_type", 3, "cfg_type"),
    ("update_kind", 2, "update_kind"),
    ("eps_c_bf16", 2, "eps_c_bf16"),
    ("txt2img", 2, "txt2img"),
    ("txt2img", 1, "cfg_type must be 0 or 2"),  # c1 runs self-negative R-CFG
    ("streams", 0, "streams"),
])
def test_invalid_configs_are_rejected_on_the_host(field, value, msg):
    cfg = B.config_from_workload(W.get_config("c1_tiny"))
    setattr(cfg, field, value)
    st, ptr = _create_status(cfg)
    assert st == B.SDS_ERR_INVALID_ARG and ptr is None
    err = B.sds_last_error()
    assert "invalid config" in err
    if msg:
        assert msg in err


def test_ring_smaller_than_a_chunk_is_rejected():
    cfg = B.config_from_workload(W.get_config("c3_dit1p3b_video"))
    cfg.ring_R = 2
    st, _ = _create_status(cfg)
    assert st == B.SDS_ERR_INVALID_ARG and "ring_R" in B.sds_last_error()


def test_t_index_outside_schedule_is_rejected():
    cfg = B.config_from_workload(W.get_config("c1_tiny"))
    cfg.t_index[0] = 50
    st, _ = _create_status(cfg)
    assert st == B.SDS_ERR_INVALID_ARG and "t_index" in B.sds_last_error()


def test_memory_cap_fails_with_oom_before_allocating():
    cfg = B.config_from_workload(W.get_config("c4_dit14b_video"), mem_cap_bytes=1 << 20)
    st, ptr = _create_status(cfg)
    assert st == B.SDS_ERR_OOM and ptr is None
    assert "mem_cap_bytes" in B.sds_last_error()


def test_calls_on_a_null_context_fail_cleanly():
    L = B.lib()
    assert L.sds_kv_push(None, None, None, None) == B.SDS_ERR_INVALID_ARG
    assert L.sds_attend(None, None, None, None, None, None) == B.SDS_ERR_INVALID_ARG
    assert L.sds_step_update(None, None, None) == B.SDS_ERR_INVALID_ARG
    assert L.sds_attention(None, None, None, None, 1, 1, 1, 1, 64, None) == B.SDS_ERR_INVALID_ARG
    L.sds_destroy(None)


def test_raw_attention_rejects_bad_sizes_without_cuda():
    L = B.lib()
    p = 1 << 12  # aligned dummy, never dereferenced: validation fails first
    assert L.sds_attention(p, p, p, p, 1, 8, 8, 1, 96, None) == B.SDS_ERR_INVALID_ARG
    assert L.sds_attention(p, p, p, p, 0, 8, 8, 1, 64, None) == B.SDS_ERR_INVALID_ARG
    assert L.sds_attention(p + 2, p, p, p, 1, 8, 8, 1, 64, None) == B.SDS_ERR_INVALID_ARG


def test_noise_rate_needs_a_rate_inside_the_unit_interval():
    """The rate places the incoming frame the fraction s of the way from slot
    1's timestep to pure noise, so with the rate applied s_min and s_max must
    lie in [0, 1]; any such config is accepted by validation, with either
    update, since the entry is never below slot 1."""
    w = W.get_config("c1_tiny", noise_rate_on=1, update_kind=1, s_min=0.0, s_max=1.0)
    for field, value in (("s_min", -0.1), ("s_max", 1.5)):
        cfg = B.config_from_workload(w)
        setattr(cfg, field, value)
        st, _ = _create_status(cfg)
        assert st == B.SDS_ERR_INVALID_ARG and "s_min <= s_max <= 1" in B.sds_last_error()
    st, ptr = _create_status(B.config_from_workload(w))
    assert st != B.SDS_ERR_INVALID_ARG  # no GPU here: creation stops later, at the device
    if ptr:
        B.lib().sds_destroy(C.c_void_p(ptr))


def test_txt2img_with_the_noise_rate_is_rejected():
    cfg = B.config_from_workload(W.get_config("c1_tiny", cfg_type=0, txt2img=1, noise_rate_on=1))
    st, _ = _create_status(cfg)
    assert st == B.SDS_ERR_INVALID_ARG and "noise_rate_on" in B.sds_last_error()
