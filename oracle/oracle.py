"""ctypes wrapper of the CPU oracle (oracle/sds_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package's smoke check
and by the benchmark's CPU-baseline leg -- never by the product path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_i64 = C.c_longlong
_f64 = C.c_double


class OrcCfg(C.Structure):
    _fields_ = [(n, _i64) for n in (
        "n", "T", "L", "H", "d", "M", "R", "image_mode", "rope_on", "grid_h", "grid_w",
        "rope_tau", "D", "n_inf", "n_train", "cfg_type", "N_s", "ssf_E", "max_skip",
        "N_f", "mot_k", "update_kind", "noise_rate_on")] + [("t_index", _i64 * 8)] + [(n, _f64) for n in (
        "rope_base", "s_th", "beta_start", "beta_end", "gamma", "delta", "eta",
        "sigma", "lam", "s_min", "s_max")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_create.restype = P
        L.orc_create.argtypes = [C.POINTER(OrcCfg)]
        L.orc_destroy.argtypes = [P]
        L.orc_set_threads.argtypes = [C.c_int]
        L.orc_max_threads.restype = C.c_int
        L.orc_bf16_round.restype = C.c_uint16
        L.orc_bf16_round.argtypes = [_f64]
        L.orc_bf16_value.restype = _f64
        L.orc_bf16_value.argtypes = [C.c_uint16]
        L.orc_alpha_bar.argtypes = [C.POINTER(OrcCfg), P]
        L.orc_slot_timestep.restype = _i64
        L.orc_slot_timestep.argtypes = [C.POINTER(OrcCfg), _i64]
        L.orc_rope_angle.restype = _f64
        L.orc_rope_angle.argtypes = [_f64, _i64, _i64, _i64]
        L.orc_rope_segments.argtypes = [_i64, P]
        L.orc_rope_rotate.argtypes = [P, P, _i64, _i64, P, _f64]
        L.orc_attention.argtypes = [P, P, P, _i64, _i64, _i64, P, _i64, P]
        L.orc_push.restype = _i64
        L.orc_push.argtypes = [P, P, P]
        L.orc_meta.argtypes = [P, P]
        L.orc_sink_refresh.argtypes = [P, P, P, P]
        L.orc_get_kv.argtypes = [P, P, P]
        L.orc_get_emb.argtypes = [P, P]
        L.orc_key_rows.restype = _i64
        L.orc_key_rows.argtypes = [P, P]
        L.orc_attend.argtypes = [P, P, P, _i64, P]
        L.orc_step_update.argtypes = [P] * 9
        L.orc_step_update2.argtypes = [P] * 10
        L.orc_ssf.argtypes = [P, P, C.c_float, P, P]
        L.orc_motion.argtypes = [P, P, P]
        L.orc_set_lazy.argtypes = [P, C.c_int]
        L.orc_provenance.argtypes = [P, P]
        L.orc_materialize.argtypes = [P, P, P]
        L.orc_slot0_timestep.restype = _i64
        L.orc_slot0_timestep.argtypes = [P]
        L.orc_noise_rate.restype = _f64
        L.orc_noise_rate.argtypes = [P]
        L.orc_skip_count.restype = _i64
        L.orc_skip_count.argtypes = [P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def make_cfg(w: dict) -> OrcCfg:
    """Oracle config from a workload dict (streaming_diffusion_stream_b300.workloads)."""
    c = OrcCfg()
    c.n, c.T, c.L, c.H, c.d = w["n"], w["T"], w["L"], w["H"], w["d"]
    c.M, c.R = w["M"], w["R"]
    c.image_mode = 1 if w["mode"] == "image" else 0
    c.rope_on = 1 if w["rope"] else 0
    c.grid_h, c.grid_w, c.rope_tau = w["grid_h"], w["grid_w"], w["rope_tau"]
    c.D, c.n_inf, c.n_train, c.cfg_type = w["D"], w["n_inf"], w["n_train"], w["cfg_type"]
    c.N_s, c.ssf_E, c.max_skip = w["N_s"], w["ssf_E"], w["max_skip"]
    c.N_f, c.mot_k = w["N_f"], w["mot_k"]
    c.update_kind = w.get("update_kind", 0)
    c.noise_rate_on = w.get("noise_rate_on", 0)
    for i, t in enumerate(w["t_index"]):
        c.t_index[i] = t
    c.rope_base, c.s_th = w["rope_base"], w["s_th"]
    c.beta_start, c.beta_end = w["beta_start"], w["beta_end"]
    c.gamma, c.delta, c.eta = w["gamma"], w["delta"], w["eta"]
    c.sigma, c.lam, c.s_min, c.s_max = w["sigma"], w["lam"], w["s_min"], w["s_max"]
    return c


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def bf16_round(x: float) -> int:
    return int(lib().orc_bf16_round(float(x)))


def bf16_value(b: int) -> float:
    return float(lib().orc_bf16_value(int(b)))


def alpha_bar(w: dict) -> np.ndarray:
    c = make_cfg(w)
    out = np.zeros(w["n_train"], dtype=np.float64)
    lib().orc_alpha_bar(C.byref(c), _p(out))
    return out


def slot_timestep(w: dict, i: int) -> int:
    c = make_cfg(w)
    return int(lib().orc_slot_timestep(C.byref(c), i))


def rope_angle(base: float, width: int, pair: int, pos: int) -> float:
    return float(lib().orc_rope_angle(base, width, pair, pos))


def rope_segments(d: int):
    seg = np.zeros(3, dtype=np.int64)
    lib().orc_rope_segments(d, _p(seg))
    return [int(s) for s in seg]


def rope_rotate(vecs: np.ndarray, pos3: np.ndarray, base: float = 10000.0) -> np.ndarray:
    vecs = np.ascontiguousarray(vecs, dtype=np.float64)
    nvec, d = vecs.shape
    pos3 = np.ascontiguousarray(pos3, dtype=np.int64).reshape(nvec, 3)
    out = np.zeros_like(vecs)
    lib().orc_rope_rotate(_p(vecs), _p(out), nvec, d, _p(pos3), base)
    return out


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows=None) -> np.ndarray:
    """Softmax attention of bf16 q rows [Lq][H][d] against bf16 k, v [Lk][H][d]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Lq, H, d = q.shape
    rows = np.arange(Lq, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), H, d), dtype=np.float64)
    lib().orc_attention(_p(q), _p(k), _p(v), H, d, k.shape[0], _p(rows), len(rows), _p(out))
    return out


class Stream:
    """One stream of the oracle's stateful path (ring, sinks, SSF, motion)."""

    def __init__(self, w: dict):
        self.w = w
        self.cfg = make_cfg(w)
        self.h = lib().orc_create(C.byref(self.cfg))

    def close(self):
        if self.h:
            lib().orc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def push(self, k: np.ndarray, v: np.ndarray) -> int:
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        return int(lib().orc_push(self.h, _p(k), _p(v)))

    def meta(self) -> dict:
        m = np.zeros(6, dtype=np.int64)
        lib().orc_meta(self.h, _p(m))
        return dict(F=int(m[0]), o=int(m[1]), p0=int(m[2]), valid=int(m[3]),
                    sinks_filled=int(m[4]), resets=int(m[5]))

    def sink_refresh(self, h: np.ndarray) -> dict:
        h = np.ascontiguousarray(h, dtype=np.float32)
        r = np.zeros(3, dtype=np.int64)
        dr = np.zeros(2, dtype=np.float64)
        lib().orc_sink_refresh(self.h, _p(h), _p(r), _p(dr))
        return dict(j=int(r[0]), fire=int(r[1]), near=int(r[2]), alpha_min=float(dr[0]),
                    alpha_2=float(dr[1]))

    def kv(self):
        w = self.w
        sh = ((w["M"] + w["R"]) * w["L"], w["H"], w["d"])
        k = np.zeros(sh, dtype=np.uint16)
        v = np.zeros(sh, dtype=np.uint16)
        lib().orc_get_kv(self.h, _p(k), _p(v))
        return k, v

    def emb(self) -> np.ndarray:
        w = self.w
        e = np.zeros((w["M"], w["D"]), dtype=np.float64)
        lib().orc_get_emb(self.h, _p(e))
        return e

    def key_rows(self) -> np.ndarray:
        n = int(lib().orc_key_rows(self.h, None))
        rows = np.zeros(n, dtype=np.int64)
        lib().orc_key_rows(self.h, _p(rows))
        return rows

    def attend(self, q: np.ndarray, rows=None) -> np.ndarray:
        """Attention of (unrotated) query rows [n*T*L][H][d]; rotation happens inside."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        w = self.w
        nrow = q.shape[0]
        rows = np.arange(nrow, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), w["H"], w["d"]), dtype=np.float64)
        lib().orc_attend(self.h, _p(q), _p(rows), len(rows), _p(out))
        return out

    def step_update(self, x, x0, eps_c, z, x0_new, eps_new, eps_neg=None):
        """Slot arrays [n][N_s] (z: [n-1][N_s]) for this stream; eps_neg [n][N_s]
        for cfg_type 2; x0_new None for txt2img; returns (x_next, out)."""
        w = self.w
        n, N = w["n"], w["N_s"]
        f = lambda a: np.ascontiguousarray(a, dtype=np.float32)
        x, x0, eps_c, eps_new = map(f, (x, x0, eps_c, eps_new))
        x0_new = f(x0_new) if x0_new is not None else None  # None: txt2img
        z = f(z) if n > 1 else np.zeros((1, N), dtype=np.float32)
        en = f(eps_neg) if eps_neg is not None else np.zeros((n, N), dtype=np.float32)
        xn = np.zeros((n, N), dtype=np.float64)
        out = np.zeros(N, dtype=np.float64)
        lib().orc_step_update2(self.h, _p(x), _p(x0), _p(eps_c), _p(z), _p(en),
                               _p(x0_new) if x0_new is not None else None, _p(eps_new), _p(xn),
                               _p(out))
        return xn, out

    def ssf(self, frame: np.ndarray, u: float) -> dict:
        frame = np.ascontiguousarray(frame, dtype=np.float32)
        r = np.zeros(3, dtype=np.int64)
        dr = np.zeros(2, dtype=np.float64)
        lib().orc_ssf(self.h, _p(frame), float(np.float32(u)), _p(r), _p(dr))
        return dict(skip=int(r[0]), skip_count=int(r[1]), near=int(r[2]), cos=float(dr[0]),
                    p=float(dr[1]))

    def motion(self, chunk: np.ndarray) -> dict:
        chunk = np.ascontiguousarray(chunk, dtype=np.float32)
        T = self.w["T"]
        dr = np.zeros(T + 2, dtype=np.float64)
        lib().orc_motion(self.h, _p(chunk), _p(dr))
        return dict(d=dr[:T].copy(), dhat=float(dr[T]), s=float(dr[T + 1]))

    def noise_rate(self) -> float:
        return float(lib().orc_noise_rate(self.h))

    def slot0_timestep(self) -> int:
        return int(lib().orc_slot0_timestep(self.h))

    def set_lazy(self, on: bool = True) -> None:
        """Pushes record provenance only; K/V are built later by materialize()."""
        lib().orc_set_lazy(self.h, int(on))

    def provenance(self) -> np.ndarray:
        """[M+R][3]: (chunk index, frame in chunk, chunk start p0) per key frame, -1 if unwritten."""
        w = self.w
        out = np.zeros((w["M"] + w["R"], 3), dtype=np.int64)
        lib().orc_provenance(self.h, _p(out))
        return out

    def materialize(self, k_frames: np.ndarray, v_frames: np.ndarray) -> None:
        """Write every key frame with a provenance from the raw frames given in
        buffer order ([M+R][L][H][d] bf16), exactly as push writes them."""
        k = np.ascontiguousarray(k_frames, dtype=np.uint16)
        v = np.ascontiguousarray(v_frames, dtype=np.uint16)
        lib().orc_materialize(self.h, _p(k), _p(v))
