"""Drive one seeded workload through the CUDA library and through the oracle.

Both sides get the same input buffers from streaming_diffusion_stream_b300.
workloads; nothing here computes any part of the method.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from streaming_diffusion_stream_b300 import binding as B
from streaming_diffusion_stream_b300 import workloads as W


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def bf16_ordered(b: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers whose difference counts ulps."""
    b = b.astype(np.int64)
    return np.where(b >= 0x8000, -(b & 0x7FFF), b)


def max_ulp_diff(a: np.ndarray, b: np.ndarray) -> int:
    return int(np.max(np.abs(bf16_ordered(a) - bf16_ordered(b)))) if a.size else 0


def rope_k_excess(gpu_bits: np.ndarray, ref_bits: np.ndarray) -> float:
    """Largest violation of the rotated-key bound (<= 1.0 means within it).

    The kernel rotates in fp32 and rounds to bf16; the oracle rotates in
    double and rounds to bf16.  Per element the difference is bounded by one
    bf16 ulp of the result plus the fp32 rounding error of the rotation,
    which is a few fp32 epsilons of the pair's norm (rotation keeps the norm):
    |g - o| <= max(ulp_bf16(o), 2^-20 * |pair|).  Near-zero results make the
    second term the larger one.  Returns max |g - o| / bound.
    """
    g = W.bf16_bits_to_f32(gpu_bits).astype(np.float64).reshape(-1, 2)
    o = W.bf16_bits_to_f32(ref_bits).astype(np.float64).reshape(-1, 2)
    norm = np.sqrt(o[:, 0] ** 2 + o[:, 1] ** 2)[:, None]
    mag = np.abs(o)
    expo = np.floor(np.log2(np.where(mag > 0, mag, 2.0 ** -126)))
    ulp = 2.0 ** (np.maximum(expo, -126) - 7)
    bound = np.maximum(ulp, 2.0 ** -20 * norm)
    return float(np.max(np.abs(g - o) / bound)) if g.size else 0.0


def attn_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """Largest per-(row-block, head) error relative to that block's max |ref|.

    gpu, ref: [rows][H][d].  Error of a head block = max |gpu - ref| /
    max(max |ref|, rms(ref)) over the rows compared.
    """
    worst = 0.0
    for h in range(ref.shape[1]):
        r = ref[:, h, :]
        g = gpu[:, h, :]
        scale = max(np.max(np.abs(r)), np.sqrt(np.mean(r * r)), 1e-30)
        worst = max(worst, float(np.max(np.abs(g - r)) / scale))
    return worst


def tensor_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max |gpu - ref| / max(max|ref|, rms(ref)) over a whole tensor."""
    scale = max(np.max(np.abs(ref)), np.sqrt(np.mean(ref * ref)), 1e-30)
    return float(np.max(np.abs(gpu.astype(np.float64) - ref)) / scale)


class _DevArray:
    """Zero-copy view of library-owned device memory for torch.as_tensor."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = dict(shape=tuple(shape), typestr=typestr,
                                             data=(int(ptr), False), version=3, strides=None)


def dev_view(ptr: int, shape, typestr: str) -> torch.Tensor:
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")


class GpuPipe:
    """The CUDA library path for one workload (S streams in one context)."""

    def __init__(self, w: dict):
        self.w = w
        self.ctx = B.sds_create(B.config_from_workload(w))
        S, HD = w["streams"], w["HD"]
        self.o = torch.empty((S, w["q_rows"], w["H"], w["d"]), dtype=torch.bfloat16, device="cuda")
        self.out = torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda")
        self.x_next = [torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda")
                       for _ in range(w["n"])]

    def close(self):
        if self.ctx:
            B.sds_destroy(self.ctx)
            self.ctx = None

    def push(self, k_bits, v_bits):
        k, v = bf16_dev(k_bits), bf16_dev(v_bits)
        B.sds_kv_push(self.ctx, k, v)
        self._keep = (k, v)

    def refresh(self, h):
        ht = f32_dev(h)
        B.sds_sink_refresh(self.ctx, ht)
        self._keep_h = ht

    def attend(self, q_bits, ext_k=None, ext_v=None) -> np.ndarray:
        q = bf16_dev(q_bits)
        ek = bf16_dev(ext_k) if ext_k is not None else None
        ev = bf16_dev(ext_v) if ext_v is not None else None
        B.sds_attend(self.ctx, q, self.o, ek, ev)
        torch.cuda.synchronize()
        return W.bf16_bits_to_f32(bf16_host(self.o)).astype(np.float64)

    def step(self, lat: dict, ssf_frame=None, u=None, motion_chunk=None):
        n = self.w["n"]
        dev = {k: f32_dev(v) for k, v in lat.items() if k not in ("z", "eps_neg")}
        if self.w.get("eps_c_bf16"):  # the predictions as bf16 tensors
            dev["eps_c"] = [bf16_dev(W.to_bf16_bits(lat["eps_c"][i])) for i in range(n)]
        z = [f32_dev(lat["z"][i]) for i in range(n - 1)]
        en = [f32_dev(lat["eps_neg"][i]) for i in range(n)] if "eps_neg" in lat else None
        sf = f32_dev(ssf_frame) if ssf_frame is not None else None
        ut = f32_dev(u) if u is not None else None
        mc = f32_dev(motion_chunk) if motion_chunk is not None else None
        io = B.make_step_io([dev["x"][i] for i in range(n)], [dev["x0"][i] for i in range(n)],
                            [dev["eps_c"][i] for i in range(n)], z, self.x_next, self.out,
                            None if self.w.get("txt2img") else dev["x0_new"], dev["eps_new"], sf,
                            ut, mc, en)
        B.sds_step_update(self.ctx, io)
        torch.cuda.synchronize()
        xn = np.stack([t.cpu().numpy() for t in self.x_next])  # [n][S][N]
        return xn, self.out.cpu().numpy()

    def ssf(self, frame, u):
        f, ut = f32_dev(frame), f32_dev(u)
        B.sds_ssf(self.ctx, f, ut)
        torch.cuda.synchronize()

    def state(self):
        return B.sds_read_state(self.ctx, self.w["streams"])

    def meta(self):
        return B.sds_get_meta(self.ctx)

    def kv(self):
        """Ring/sink K and V as bf16 bits [S][(M+R)*L][H][d]."""
        w = self.w
        buf = B.sds_get_buffers(self.ctx)
        shape = (w["streams"], buf["kv_rows"], w["H"], w["d"])
        torch.cuda.synchronize()
        return [dev_view(ptr, shape, "<i2").cpu().numpy().view(np.uint16)
                for ptr in (buf["kv_k"], buf["kv_v"])]

    def sink_emb(self):
        w = self.w
        buf = B.sds_get_buffers(self.ctx)
        torch.cuda.synchronize()
        return dev_view(buf["sink_emb"], (w["streams"], w["M"], w["D"]), "<f4").cpu().numpy()


class OraclePipe:
    """The oracle path: one oracle stream per workload stream."""

    def __init__(self, w: dict):
        self.w = w
        self.s = [O.Stream(w) for _ in range(w["streams"])]

    def push(self, k_bits, v_bits):
        return [s.push(k_bits[i], v_bits[i]) for i, s in enumerate(self.s)]

    def refresh(self, h):
        return [s.sink_refresh(h[i]) for i, s in enumerate(self.s)]

    def attend(self, q_bits, rows=None):
        return [s.attend(q_bits[i], rows) for i, s in enumerate(self.s)]

    def step(self, lat: dict):
        n = self.w["n"]
        ec = lat["eps_c"]
        if self.w.get("eps_c_bf16"):  # the values the bf16 tensors hold
            ec = W.bf16_bits_to_f32(W.to_bf16_bits(ec))
        res = []
        for i, s in enumerate(self.s):
            z = lat["z"][:, i] if n > 1 else None
            en = lat["eps_neg"][:, i] if "eps_neg" in lat else None
            x0n = None if self.w.get("txt2img") else lat["x0_new"][i]
            res.append(s.step_update(lat["x"][:, i], lat["x0"][:, i], ec[:, i], z, x0n,
                                     lat["eps_new"][i], eps_neg=en))
        return res

    def ssf(self, frame, u):
        return [s.ssf(frame[i], float(u[i])) for i, s in enumerate(self.s)]

    def motion(self, chunk):
        return [s.motion(chunk[i]) for i, s in enumerate(self.s)]
