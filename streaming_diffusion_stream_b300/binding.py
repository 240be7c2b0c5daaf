"""ctypes binding of libsds.so (include/sds.h), names as in the C ABI.

Argument marshalling only: tensors are passed as device pointers (torch
tensors' data_ptr()), streams as cudaStream_t handles.  Every step of the
path runs in the library's CUDA kernels; there is no CPU fallback.  Loading
fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsds.so")

SDS_ABI_VERSION = 5
SDS_MAX_SLOTS = 8
SDS_MAX_CHUNK_FRAMES = 8
SDS_STATE_MAGIC = b"SDSSTAT1"
SDS_STATE_RECORD_BYTES = 760

SDS_OK, SDS_ERR_INVALID_ARG, SDS_ERR_OOM, SDS_ERR_CUDA, SDS_ERR_STATE, SDS_ERR_UNSUPPORTED = range(6)
STATUS_NAMES = {0: "SDS_OK", 1: "SDS_ERR_INVALID_ARG", 2: "SDS_ERR_OOM", 3: "SDS_ERR_CUDA",
                4: "SDS_ERR_STATE", 5: "SDS_ERR_UNSUPPORTED"}

_i64 = C.c_int64
_f64 = C.c_double
_P = C.c_void_p


class sds_config(C.Structure):
    _fields_ = [("abi_version", _i64)] + [(n, _i64) for n in (
        "streams", "slots_n", "frames_T", "tokens_L", "heads_H", "head_dim", "sink_M", "ring_R",
        "rope_on", "grid_h", "grid_w", "rope_tau", "emb_dim_D")] + [
        ("t_index", _i64 * SDS_MAX_SLOTS)] + [(n, _i64) for n in (
            "num_inference_steps", "num_train_steps", "cfg_type", "slot_elems", "ssf_on",
            "ssf_elems", "max_skip_frame", "motion_on", "frame_elems", "mot_k",
            "mem_cap_bytes", "attn_ctas", "update_kind", "noise_rate_on", "eps_c_bf16",
            "txt2img")] + [(n, _f64) for n in (
                "rope_base", "s_th", "beta_start", "beta_end", "gamma", "delta", "ssf_eta",
                "mot_sigma", "mot_lambda", "s_min", "s_max")]


class sds_step_io(C.Structure):
    _fields_ = [("x", _P * SDS_MAX_SLOTS), ("x0", _P * SDS_MAX_SLOTS),
                ("eps_c", _P * SDS_MAX_SLOTS), ("z", _P * SDS_MAX_SLOTS),
                ("x_next", _P * SDS_MAX_SLOTS), ("out", _P), ("x0_new", _P), ("eps_new", _P),
                ("ssf_frame", _P), ("ssf_u", _P), ("motion_chunk", _P),
                ("eps_neg", _P * SDS_MAX_SLOTS)]


class sds_stream_state(C.Structure):
    _fields_ = [("ssf_evals", _i64), ("ssf_skip", _i64), ("ssf_skip_count", _i64),
                ("ssf_has_ref", _i64), ("ssf_cos", _f64), ("ssf_p", _f64), ("sink_j", _i64),
                ("sink_fire", _i64), ("sink_alpha_min", _f64), ("sink_alpha_2", _f64),
                ("motion_pairs", _i64), ("motion_dhat", _f64), ("noise_rate", _f64),
                ("motion_d", _f64 * SDS_MAX_CHUNK_FRAMES), ("error_word", _i64),
                ("slot0_timestep", _i64)]

    def as_dict(self) -> dict:
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["motion_d"] = list(self.motion_d)
        return d


class sds_meta(C.Structure):
    _fields_ = [(n, _i64) for n in ("frames_pushed", "rope_offset", "chunk_p0", "ring_valid",
                                    "sinks_filled", "rope_resets", "chunks")]


class sds_buffers(C.Structure):
    _fields_ = [("kv_k", _P), ("kv_v", _P), ("sink_emb", _P), ("kv_rows", _i64)]


class sds_state_header(C.Structure):
    _fields_ = [("magic", C.c_char * 8), ("abi_version", _i64), ("config_hash", C.c_uint64),
                ("flags", _i64), ("payload_bytes", _i64), ("payload_hash", C.c_uint64),
                ("streams", _i64), ("devstate_bytes", _i64), ("emb_elems", _i64),
                ("ssf_ref_elems", _i64), ("mot_prev_elems", _i64), ("kv_elems", _i64),
                ("reserved", _i64 * 4)]


class sds_slo_config(C.Structure):
    _fields_ = [("target_fps", _f64), ("forget", _f64), ("knee_gain", _f64),
                ("frames_T", _i64), ("b_min", _i64), ("b_max", _i64)]


class sds_slo_choice(C.Structure):
    _fields_ = [("batch", _i64), ("meets_slo", _i64), ("exploring", _i64), ("b_slo", _i64),
                ("b_knee", _i64), ("a", _f64), ("b", _f64), ("latency_s", _f64),
                ("per_stream_fps", _f64), ("total_fps", _f64)]


# name -> (restype, argtypes)
SIGNATURES = {
    "sds_abi_version": (C.c_int, []),
    "sds_create": (C.c_int, [C.POINTER(sds_config), C.POINTER(_P)]),
    "sds_destroy": (None, [_P]),
    "sds_last_error": (C.c_char_p, [_P]),
    "sds_kv_push": (C.c_int, [_P, _P, _P, _P]),
    "sds_sink_refresh": (C.c_int, [_P, _P, _P]),
    "sds_attend": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "sds_attention": (C.c_int, [_P, _P, _P, _P, _i64, _i64, _i64, _i64, _i64, _P]),
    "sds_step_update": (C.c_int, [_P, C.POINTER(sds_step_io), _P]),
    "sds_ssf": (C.c_int, [_P, _P, _P, _P]),
    "sds_ssf_noalloc": (C.c_int, [_P, _P, _P, _P, _i64, _i64, _f64, _i64, _P, _P, _P, _P]),
    "sds_read_state": (C.c_int, [_P, C.POINTER(sds_stream_state), _P]),
    "sds_test_attn_timeout": (C.c_int, [_P, _i64, _i64]),
    "sds_get_meta": (C.c_int, [_P, C.POINTER(sds_meta)]),
    "sds_get_buffers": (C.c_int, [_P, C.POINTER(sds_buffers)]),
    "sds_state_export": (C.c_int, [_P, _P, C.POINTER(C.c_size_t), _i64, _P]),
    "sds_state_import": (C.c_int, [_P, _P, C.c_size_t, _P]),
    "sds_state_check": (C.c_int, [C.POINTER(sds_config), _P, C.c_size_t]),
    "sds_slo_create": (C.c_int, [C.POINTER(sds_slo_config), C.POINTER(_P)]),
    "sds_slo_destroy": (None, [_P]),
    "sds_slo_observe": (C.c_int, [_P, _i64, _f64]),
    "sds_slo_choose": (C.c_int, [_P, C.POINTER(sds_slo_choice)]),
}

_lib = None


def lib() -> C.CDLL:
    """Load libsds.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m streaming_diffusion_stream_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class SdsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def check(status: int, ctx=None):
    if status != SDS_OK:
        msg = lib().sds_last_error(ctx)
        raise SdsError(status, msg.decode() if msg else "")


def config_from_workload(w: dict, mem_cap_bytes: int = 0) -> sds_config:
    """sds_config for a workload dict of streaming_diffusion_stream_b300.workloads."""
    c = sds_config()
    c.abi_version = SDS_ABI_VERSION
    c.streams, c.slots_n, c.frames_T, c.tokens_L = w["streams"], w["n"], w["T"], w["L"]
    c.heads_H, c.head_dim = w["H"], w["d"]
    video = w["mode"] == "video"
    c.sink_M, c.ring_R = (w["M"], w["R"]) if video else (0, 0)
    c.rope_on = 1 if (video and w["rope"]) else 0
    c.grid_h, c.grid_w, c.rope_tau = w["grid_h"], w["grid_w"], w["rope_tau"]
    c.emb_dim_D = w["D"]
    for i, t in enumerate(w["t_index"]):
        c.t_index[i] = t
    c.num_inference_steps, c.num_train_steps, c.cfg_type = w["n_inf"], w["n_train"], w["cfg_type"]
    c.slot_elems = w["N_s"]
    c.ssf_on, c.ssf_elems, c.max_skip_frame = int(w["ssf"]), w["ssf_E"], w["max_skip"]
    c.motion_on, c.frame_elems, c.mot_k = int(w["motion"]), w["N_f"], w["mot_k"]
    c.mem_cap_bytes = mem_cap_bytes
    c.attn_ctas = w.get("attn_ctas", 0)
    c.update_kind = w.get("update_kind", 0)
    c.noise_rate_on = w.get("noise_rate_on", 0)
    c.eps_c_bf16 = w.get("eps_c_bf16", 0)
    c.txt2img = w.get("txt2img", 0)
    c.rope_base, c.s_th = w["rope_base"], w["s_th"]
    c.beta_start, c.beta_end = w["beta_start"], w["beta_end"]
    c.gamma, c.delta, c.ssf_eta = w["gamma"], w["delta"], w["eta"]
    c.mot_sigma, c.mot_lambda, c.s_min, c.s_max = w["sigma"], w["lam"], w["s_min"], w["s_max"]
    return c


def sds_abi_version() -> int:
    return int(lib().sds_abi_version())


def sds_last_error(ctx=None) -> str:
    m = lib().sds_last_error(ctx)
    return m.decode() if m else ""


def sds_create(cfg: sds_config) -> int:
    out = _P()
    check(lib().sds_create(C.byref(cfg), C.byref(out)))
    return out.value


def sds_destroy(ctx: int) -> None:
    lib().sds_destroy(ctx)


def sds_kv_push(ctx, k, v, stream=None):
    check(lib().sds_kv_push(ctx, _ptr(k), _ptr(v), _stream(stream)), ctx)


def sds_sink_refresh(ctx, chunk_emb, stream=None):
    check(lib().sds_sink_refresh(ctx, _ptr(chunk_emb), _stream(stream)), ctx)


def sds_attend(ctx, q, o, ext_k=None, ext_v=None, stream=None):
    check(lib().sds_attend(ctx, _ptr(q), _ptr(o), _ptr(ext_k), _ptr(ext_v), _stream(stream)), ctx)


def sds_attention(q, k, v, o, S, Lq, Lk, H, head_dim, stream=None):
    check(lib().sds_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), S, Lq, Lk, H, head_dim,
                              _stream(stream)))


def make_step_io(x, x0, eps_c, z, x_next, out, x0_new, eps_new, ssf_frame=None, ssf_u=None,
                 motion_chunk=None, eps_neg=None) -> sds_step_io:
    """x, x0, eps_c, x_next: sequences of n per-slot tensors; z: n-1 tensors;
    eps_neg: n tensors (cfg_type 2) or None."""
    io = sds_step_io()
    for i, t in enumerate(x):
        io.x[i] = _ptr(t)
    for i, t in enumerate(x0):
        io.x0[i] = _ptr(t)
    for i, t in enumerate(eps_c):
        io.eps_c[i] = _ptr(t)
    for i, t in enumerate(z):
        io.z[i] = _ptr(t)
    for i, t in enumerate(x_next):
        io.x_next[i] = _ptr(t)
    io.out, io.x0_new, io.eps_new = _ptr(out), _ptr(x0_new), _ptr(eps_new)
    io.ssf_frame, io.ssf_u, io.motion_chunk = _ptr(ssf_frame), _ptr(ssf_u), _ptr(motion_chunk)
    for i, t in enumerate(eps_neg or []):
        io.eps_neg[i] = _ptr(t)
    return io


def sds_step_update(ctx, io: sds_step_io, stream=None):
    check(lib().sds_step_update(ctx, C.byref(io), _stream(stream)), ctx)


def sds_test_attn_timeout(ctx, wait_limit_ns: int, withhold_k_tile: int):
    check(lib().sds_test_attn_timeout(ctx, int(wait_limit_ns), int(withhold_k_tile)), ctx)


def sds_ssf(ctx, frame, u, stream=None):
    check(lib().sds_ssf(ctx, _ptr(frame), _ptr(u), _stream(stream)), ctx)


def sds_ssf_noalloc(frame, ref, u, skip_count, S, E, eta, max_skip, cos_out, p_out, skip_out,
                    stream=None):
    """Allocation-free similarity filter (see include/sds.h): all arguments are
    caller-owned device tensors; the library allocates nothing."""
    check(lib().sds_ssf_noalloc(_ptr(frame), _ptr(ref), _ptr(u), _ptr(skip_count), S, E, eta,
                                max_skip, _ptr(cos_out), _ptr(p_out), _ptr(skip_out),
                                _stream(stream)))


def sds_read_state(ctx, streams: int, stream=None) -> list[dict]:
    arr = (sds_stream_state * streams)()
    check(lib().sds_read_state(ctx, arr, _stream(stream)), ctx)
    return [a.as_dict() for a in arr]


def sds_get_meta(ctx) -> dict:
    m = sds_meta()
    check(lib().sds_get_meta(ctx, C.byref(m)), ctx)
    return {n: getattr(m, n) for n, _ in m._fields_}


def sds_get_buffers(ctx) -> dict:
    b = sds_buffers()
    check(lib().sds_get_buffers(ctx, C.byref(b)), ctx)
    return {n: getattr(b, n) for n, _ in b._fields_}


def sds_state_export(ctx, with_kv: bool = True, stream=None) -> bytes:
    """Checkpoint of the context (synchronises `stream`) as bytes."""
    n = C.c_size_t(0)
    check(lib().sds_state_export(ctx, None, C.byref(n), int(with_kv), _stream(stream)), ctx)
    buf = C.create_string_buffer(n.value)
    check(lib().sds_state_export(ctx, buf, C.byref(n), int(with_kv), _stream(stream)), ctx)
    return buf.raw[:n.value]


def sds_state_import(ctx, data: bytes, stream=None) -> None:
    check(lib().sds_state_import(ctx, data, len(data), _stream(stream)), ctx)


def sds_state_check(cfg: sds_config, data: bytes) -> None:
    """Validate a checkpoint against a configuration (no device access)."""
    check(lib().sds_state_check(C.byref(cfg), data, len(data)))


class SloController:
    """The library's SLO-aware stream-batch controller (host only)."""

    def __init__(self, target_fps: float, frames_T: int, b_min: int = 1, b_max: int = 8,
                 forget: float = 1.0, knee_gain: float = 0.05):
        cfg = sds_slo_config(target_fps, forget, knee_gain, frames_T, b_min, b_max)
        h = _P()
        check(lib().sds_slo_create(C.byref(cfg), C.byref(h)))
        self.h = h.value

    def observe(self, batch: int, latency_s: float) -> None:
        check(lib().sds_slo_observe(self.h, int(batch), float(latency_s)))

    def choose(self) -> dict:
        r = sds_slo_choice()
        check(lib().sds_slo_choose(self.h, C.byref(r)))
        return {n: getattr(r, n) for n, _ in r._fields_}

    def close(self) -> None:
        if self.h:
            lib().sds_slo_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
