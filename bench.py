#!/usr/bin/env python3
"""Benchmark of the stream-batch attend + update step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c4_dit14b_video|c2_sdturbo_image|c3_dit1p3b_video|c5_stress]
                    [--streams B]

One step is one pass of the whole hot path over one batch of synthetic input:
image workloads run K1 attend (external batch K/V) + K4 (R-CFG update + SSF);
video workloads run K2 push + K3 sink refresh + K1 attend + K4 (update +
motion).  Frames per step: 1 (image) or T (video), per stream.

Inputs live in HBM before the timed region; consecutive steps cycle through
enough independent input sets that their total exceeds the L2 cache.  Time is
measured with CUDA events on the launching stream, bracketed by a barrier and
a device synchronize, max over ranks.  rank 0 prints one JSON line.

--impl reference times the CPU oracle (the double-precision reference of the
same computation) on the host cores, each step a bounded sample.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from streaming_diffusion_stream_b300 import workloads as W  # noqa: E402

METRIC = "frames/s of stream-batch attend+update step"
UNIT = "frames/s"
PROFILE_DIR = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 300; 20 for --impl reference)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default 20; 3 for --impl reference)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c4_dit14b_video")
    ap.add_argument("--streams", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hbm-isolated", action="store_true",
                    help="skip the isolated K2 / K4 timing at c5 with 8 streams")
    ap.add_argument("--cfg-type", type=int, default=None,
                    help="guidance: 0 none, 1 self-negative R-CFG, 2 supplied negative prediction")
    ap.add_argument("--update-kind", type=int, default=None,
                    help="0 predict x0 and re-noise, 1 strided DDPM posterior")
    ap.add_argument("--noise-rate-on", action="store_true",
                    help="the incoming frame enters slot 0 at the motion noise rate")
    ap.add_argument("--eps-c-bf16", action="store_true",
                    help="the noise predictions eps_c arrive as bf16")
    ap.add_argument("--txt2img", action="store_true",
                    help="no input image: the incoming frame is the noise draw (cfg_type 0 unless given)")
    ap.add_argument("--sweep-streams", type=int, default=0,
                    help="print one line per stream count B = 1..N (same workload, one GPU)")
    return ap.parse_args()


def workload(args, rank: int = 0) -> dict:
    """The workload one rank serves.  Ranks are independent replicas serving
    their own streams, so each rank draws its inputs from its own seed."""
    over = {}
    if getattr(args, "streams", None):
        over["streams"] = args.streams
    if getattr(args, "cfg_type", None) is not None:
        over["cfg_type"] = args.cfg_type
    if getattr(args, "update_kind", None) is not None:
        over["update_kind"] = args.update_kind
    if getattr(args, "noise_rate_on", False):
        over["noise_rate_on"] = 1
    if getattr(args, "eps_c_bf16", False):
        over["eps_c_bf16"] = 1
    if getattr(args, "txt2img", False):
        over["txt2img"] = 1
        over.setdefault("cfg_type", 0)
    w = W.get_config(args.workload, **over)
    w["seed"] = w["seed"] + 1000 * rank
    return w


def frames_per_step(w: dict) -> int:
    return w["streams"] * (w["T"] if w["mode"] == "video" else 1)


def attn_flops(w: dict) -> float:
    """Algorithmic FLOPs of one attend launch: 4 * S * H * Lq * Lk * d (QK^T and PV)."""
    return 4.0 * w["streams"] * w["H"] * w["q_rows"] * w["key_cap"] * w["d"]


def step_bytes(w: dict, with_ssf: bool, with_motion: bool) -> float:
    """Algorithmic bytes of one K4 launch: every operand read once, every result written once."""
    n, S = w["n"], w["streams"]
    # x, eps_c, x0 or eps_neg (n each; no third without guidance), z (n-1),
    # x0_new, eps_new read | x_next (n), out written
    per_slot = 5 if w.get("cfg_type", 1) != 0 else 4
    b = 4.0 * S * w["N_s"] * (per_slot * n + 2)
    if w.get("eps_c_bf16"):
        b -= 2.0 * S * w["N_s"] * n       # eps_c read as 2-byte values
    if w.get("txt2img"):
        b -= 4.0 * S * w["N_s"]           # no x0_new
    if with_ssf:
        b += 4.0 * S * w["ssf_E"] * 3     # frame, reference | reference copy
    if with_motion:
        b += 4.0 * S * w["N_f"] * (w["T"] + 2)  # T frames + previous | previous copy
    return b


def push_bytes(w: dict) -> float:
    """Algorithmic bytes of one K2 launch: the chunk's K and V read once and
    written once into the ring (bf16)."""
    return 2.0 * 4 * w["streams"] * w["kv_rows"] * w["HD"]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


def attn_roofline(w: dict, ms: float, peaks: dict, ms_region: float, clocks=None) -> dict:
    """K1's line: algorithmic FLOPs per launch / mean launch time, against
    the measured bf16 peak.  The burst peak applies to a kernel timed at
    full clocks; when the clock samples of the timed region show the power
    cap (or clocks well below their maximum), the region ran as the
    sustained peak was measured -- under the power cap -- and that peak
    applies.  The other fraction is given beside it."""
    flops = attn_flops(w)
    achieved = flops / (ms / 1e3) / 1e12
    capped = bool(clocks) and ("sw_power_cap" in (clocks.get("reasons") or []) or (
        clocks.get("sm_mhz") and clocks.get("sm_max_mhz")
        and clocks["sm_mhz"] < 0.95 * clocks["sm_max_mhz"]))
    sustained = capped or ms_region >= 3000.0
    peak = peaks["bf16_sus"] if sustained else peaks["bf16"]
    kind = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if capped:
        kind += ", power cap seen in the timed region"
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": ncu_traffic("attn", w["name"]),
            "kernel": "attn_kernel (K1)", "ms_per_launch": round(ms, 4), "flops_per_launch": flops,
            "peak_kind": f"{kind} ({peaks['source']})",
            "timed_region_ms": round(ms_region, 1),
            "frac_of_burst": round(achieved / peaks["bf16"], 4),
            "frac_of_sustained": round(achieved / peaks["bf16_sus"], 4)}


def hbm_roofline(kernel: str, nbytes: float, ms: float, peaks: dict) -> dict:
    """An HBM-bound kernel: algorithmic bytes per launch / mean launch time,
    against the measured copy bandwidth."""
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": peaks["hbm"],
            "unit": "GB/s", "frac": round(gbs / peaks["hbm"], 4), "bytes_per_launch": nbytes,
            "ms_per_launch": round(ms, 4), "peak_kind": f"hbm_gbs ({peaks['source']})"}


def kernel_source_hash() -> str:
    """Hash of the attention kernel's sources with // comments and blank
    lines removed, so that a comment edit does not orphan an ncu capture."""
    import hashlib
    h = hashlib.sha256()
    for f in ("k_attn.cu", "ptx.cuh", "rope.cuh"):
        lines = []
        for line in open(os.path.join(ROOT, "streaming_diffusion_stream_b300", "csrc", f)):
            i = line.find("//")
            code = (line[:i] if i >= 0 else line).rstrip()
            if code.strip():
                lines.append(code)
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload_name: str):
    """Per-launch DRAM bytes recorded from an ncu capture of the current kernel source.

    Reads profiles/<kernel>_<workload>.txt (lines 'key: value'); returns None
    when absent or when the kernel source changed since the capture.
    """
    p = os.path.join(PROFILE_DIR, f"{kernel}_{workload_name}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    def __init__(self, uuid: str | None):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="sds_clocks_", suffix=".csv")
        os.close(fd)
        # Every poll costs the GPU work some throughput (a 100 ms poll of this
        # query slowed the c3 step by about 9 %), so poll every 200 ms and
        # only the fields that are reported.
        q = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def remove(self):
        try:
            os.unlink(self.path)
        except OSError:
            pass

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        n_inside = len(inside)
        if not inside and rows:
            # a timed region shorter than the poll interval: the nearest poll
            inside = [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": inside[0][2],
                "reasons": reasons, "samples": n_inside, "poll_ms": 200}


# --------------------------------------------------------------------------- our arm

class Runner:
    """Device buffers and the step sequence for one workload on one GPU."""

    def __init__(self, w: dict, pool_bytes_min: float):
        import torch
        from streaming_diffusion_stream_b300 import binding as B
        self.torch, self.B, self.w = torch, B, w
        self.ctx = B.sds_create(B.config_from_workload(w))
        S, n = w["streams"], w["n"]
        self.video = w["mode"] == "video"
        dev = "cuda"
        bf = torch.bfloat16
        self.o = torch.empty((S, w["q_rows"], w["H"], w["d"]), dtype=bf, device=dev)
        self.out = torch.empty((S, w["N_s"]), dtype=torch.float32, device=dev)
        self.x_next = [torch.empty((S, w["N_s"]), dtype=torch.float32, device=dev) for _ in range(n)]
        # pool of independent input sets larger than L2
        set_bytes = self.set_bytes()
        self.n_sets = int(max(2, min(64, np.ceil(pool_bytes_min / set_bytes))))
        # consecutive chunk embeddings are steps of one unit-norm random walk,
        # as in the workload (the sink refreshes when the walk drifts past s_th)
        self.emb_walk = W.EmbeddingWalk(w)
        self.sets = [self.make_set(i) for i in range(self.n_sets)]
        self.pool_bytes = set_bytes * self.n_sets

    def set_bytes(self) -> float:
        w = self.w
        b = 2.0 * w["streams"] * w["q_rows"] * w["HD"] + 2 * 2.0 * w["streams"] * w["kv_rows"] * w["HD"]
        b += 4.0 * w["streams"] * w["N_s"] * ((5 if w.get("cfg_type", 1) == 2 else 4) * w["n"] + 1)
        if w["ssf"]:
            b += 4.0 * w["streams"] * w["ssf_E"]
        if w["motion"]:
            b += 4.0 * w["streams"] * w["T"] * w["N_f"]
        if self.video and w["M"] > 0:
            b += 4.0 * w["streams"] * w["D"]
        return b

    def host_set(self, i: int) -> dict:
        w = self.w
        k, v = W.gen_kv(w, i)
        d = dict(q=W.gen_q(w, i), k=k, v=v)
        lat = W.gen_latents(w, i)
        if w.get("eps_c_bf16"):
            lat["eps_c"] = W.to_bf16_bits(lat["eps_c"])
        d.update(lat)
        if w["ssf"]:
            d["frame"] = W.FrameWalk(dict(w, seed=w["seed"] + 7919 * (i + 1))).next()
            d["u"] = W.gen_u(w, i)
        if w["motion"]:
            d["chunk"] = W.LatentWalk(dict(w, seed=w["seed"] + 104729 * (i + 1))).next()
        if self.video and w["M"] > 0:
            d["h"] = self.emb_walk.next()
        return d

    def make_set(self, i: int) -> dict:
        """One input set in HBM: every tensor is a view into one flat device
        buffer laid out like host_flat's pinned buffer, so the end-to-end run
        can move a whole step's inputs with a single host-to-device copy."""
        flat, views = self.flat_views(self.host_set(i))
        dev = flat.cuda()
        return self.bind(dev, views)

    def flat_views(self, hs: dict):
        """Pack a host input set into one byte buffer (16-byte aligned
        tensors); returns it and the (key, offset, dtype, shape) of each."""
        torch = self.torch
        views, off = [], 0
        for key, a in hs.items():
            bf16 = a.dtype == np.uint16
            a = a if bf16 else np.ascontiguousarray(a, dtype=np.float32)
            views.append((key, off, bf16, a.shape))
            off += -(-a.nbytes // 16) * 16
        flat = np.zeros(off, dtype=np.uint8)
        for (key, o, bf16, shape), a in zip(views, hs.values()):
            a = a if bf16 else np.ascontiguousarray(a, dtype=np.float32)
            flat[o:o + a.nbytes] = a.reshape(-1).view(np.uint8)
        return torch.from_numpy(flat), views

    def bind(self, dev, views) -> dict:
        torch = self.torch
        out = {"_flat": dev}
        for key, o, bf16, shape in views:
            n = int(np.prod(shape))
            dt = torch.bfloat16 if bf16 else torch.float32
            out[key] = dev[o:o + n * 2 if bf16 else o + n * 4].view(dt).view(shape)
        out["_io"] = self.io(out)
        return out

    def io(self, s: dict):
        n = self.w["n"]
        en = [s["eps_neg"][i] for i in range(n)] if "eps_neg" in s else None
        return self.B.make_step_io([s["x"][i] for i in range(n)], [s["x0"][i] for i in range(n)],
                                   [s["eps_c"][i] for i in range(n)],
                                   [s["z"][i] for i in range(n - 1)], self.x_next, self.out,
                                   None if self.w.get("txt2img") else s["x0_new"], s["eps_new"],
                                   s.get("frame"), s.get("u"),
                                   s.get("chunk"), en)

    def step(self, s: dict, ev=None):
        """One pass of the hot path.  ev: optional dict of (start, end) events per kernel."""
        B, ctx = self.B, self.ctx

        def rec(name, i):
            if ev is not None:
                ev[name][i].record()

        if self.video:
            rec("push", 0)
            B.sds_kv_push(ctx, s["k"], s["v"])
            rec("push", 1)
            if self.w["M"] > 0:
                rec("refresh", 0)
                B.sds_sink_refresh(ctx, s["h"])
                rec("refresh", 1)
            rec("attend", 0)
            B.sds_attend(ctx, s["q"], self.o)
            rec("attend", 1)
        else:
            rec("attend", 0)
            B.sds_attend(ctx, s["q"], self.o, s["k"], s["v"])
            rec("attend", 1)
        rec("update", 0)
        B.sds_step_update(ctx, s["_io"])
        rec("update", 1)

    def launches_per_step(self) -> int:
        """Kernels one step launches: push, sink decision + copy (with sinks),
        attend, fused update -- or attend + update in image mode."""
        if self.video:
            return 3 + (2 if self.w["M"] > 0 else 0)
        return 2

    def close(self):
        self.torch.cuda.synchronize()
        self.B.sds_destroy(self.ctx)


def dist_setup(n_gpus: int):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value (timing only: the data path has no collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(frames_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job frames/s: all ranks' frames over the slowest rank's time."""
    return frames_per_rank * world / (ms_max / 1e3)


def run_ours(args):
    import torch
    rank, world = dist_setup(args.gpus)
    w = workload(args, rank)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    run = Runner(w, pool_bytes_min=2.0 * l2)
    stream = torch.cuda.current_stream()
    steps, warm = args.steps, max(3, args.warmup)

    for i in range(warm):
        run.step(run.sets[i % run.n_sets])
    torch.cuda.synchronize()

    names = ["attend", "update"] + (["push"] + (["refresh"] if w["M"] > 0 else []) if run.video else [])
    ev = {n: [[torch.cuda.Event(enable_timing=True) for _ in range(steps)] for _ in range(2)]
          for n in names}
    # create every event now (an event is created on its first record), so
    # that the timed loop only enqueues work
    for n in names:
        for pair in ev[n]:
            for e in pair:
                e.record(stream)
    torch.cuda.synchronize()
    uuid = str(getattr(props, "uuid", "")) or None
    if uuid and not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    clk = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if clk else 0.0)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        evi = {n: (ev[n][0][i], ev[n][1][i]) for n in names}
        run.step(run.sets[(warm + i) % run.n_sets], evi)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    clocks = clk.summary(wall0, wall1) if clk else None
    if clk:
        clk.stop()
        clk.remove()
    per_kernel = {n: float(np.mean([ev[n][0][i].elapsed_time(ev[n][1][i]) for i in range(steps)]))
                  for n in names}
    ms_step = ms_total / steps
    value = aggregate(frames_per_step(w) * steps, ms_total, world)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(run, w, max(10, min(steps, 100)), world)

    peaks = load_peaks()
    a_ms = per_kernel["attend"]
    roof = attn_roofline(w, a_ms, peaks, ms_total, clocks)
    kern = {"attend": {"ms": round(a_ms, 4), "tflops": roof["achieved"]}}
    hbm = {}
    ub = step_bytes(w, w["ssf"], w["motion"])
    hbm["update"] = hbm_roofline("step_kernel (K4)", ub, per_kernel["update"], peaks)
    if run.video:
        hbm["push"] = hbm_roofline("kv_push_kernel (K2)", push_bytes(w), per_kernel["push"], peaks)
        if "refresh" in per_kernel:
            kern["refresh"] = {"ms": round(per_kernel["refresh"], 4),
                               "note": "decision every step; the copy only when a sink is replaced"}
    for k, r in hbm.items():
        kern[k] = {"ms": r["ms_per_launch"], "bytes": r["bytes_per_launch"], "gbs": r["achieved"],
                   "frac_hbm": r["frac"]}

    iso = None
    if rank == 0 and not args.no_hbm_isolated:
        iso = hbm_isolated(peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["name"], "streams_per_gpu": w["streams"], "slots_n": w["n"],
                   "heads": w["H"], "head_dim": w["d"], "q_rows": w["q_rows"],
                   "keys": w["key_cap"], "frames_per_step": frames_per_step(w),
                   "update_dtype": "fp32", "attention_dtype": "bf16 in, fp32 accumulate",
                   "l2": f"{run.n_sets} rotating input sets, {run.pool_bytes / 2**20:.0f} MiB > L2 "
                         f"{l2 / 2**20:.0f} MiB",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "roofline_hbm": hbm, "roofline_hbm_isolated": iso, "kernels": kern,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": run.launches_per_step() * steps, "clocks": clocks,
    }
    run.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def hbm_isolated(peaks: dict, launches: int = 100) -> dict:
    """K2 and K4 alone at the long-run shape with 8 streams (c5_stress), the
    configuration whose bytes exceed L2 (K2 460 MB, K4 131 MB per launch):
    back-to-back launches on rotating input sets that together exceed 2 x
    L2, CUDA events around them.  Returns a roofline entry per kernel."""
    import torch
    from streaming_diffusion_stream_b300 import binding as B
    w = W.get_config("c5_stress", streams=8)
    ctx = B.sds_create(B.config_from_workload(w))
    n, S = w["n"], w["streams"]
    out = torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda")
    x_next = [torch.empty((S, w["N_s"]), dtype=torch.float32, device="cuda") for _ in range(n)]
    sets = []
    for i in range(3):  # K4 reads ~96 MB and K2 ~230 MB per set: three sets exceed 2 x L2
        lat = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in W.gen_latents(w, i).items()}
        chunk = torch.from_numpy(W.LatentWalk(dict(w, seed=w["seed"] + 31 * (i + 1))).next()).cuda()
        kb, vb = W.gen_kv(w, i)
        k = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda()
        v = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).cuda()
        io = B.make_step_io([lat["x"][j] for j in range(n)], [lat["x0"][j] for j in range(n)],
                            [lat["eps_c"][j] for j in range(n)], [lat["z"][j] for j in range(n - 1)],
                            x_next, out, lat["x0_new"], lat["eps_new"], None, None, chunk)
        sets.append(dict(lat=lat, chunk=chunk, k=k, v=v, io=io))
    res = {"workload": "c5_stress, 8 streams", "launches": launches}
    for name, fn, nbytes in (
            ("update", lambda st: B.sds_step_update(ctx, st["io"]), step_bytes(w, False, True)),
            ("push", lambda st: B.sds_kv_push(ctx, st["k"], st["v"]), push_bytes(w))):
        for i in range(10):
            fn(sets[i % 3])
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(launches):
            fn(sets[i % 3])
        b.record()
        torch.cuda.synchronize()
        kern = "step_kernel (K4)" if name == "update" else "kv_push_kernel (K2)"
        res[name] = hbm_roofline(kern, nbytes, a.elapsed_time(b) / launches, peaks)
    torch.cuda.synchronize()
    B.sds_destroy(ctx)
    return res


def run_e2e(run: Runner, w: dict, steps: int, world: int) -> dict:
    """Same step with inputs copied from pinned host memory each step and the
    completed frame read back, all inside the timed region.  The copies of
    step i+1 run on a second stream into the other device input set while
    step i computes (double buffering, as a streaming service would run)."""
    import torch
    flat, _ = run.flat_views(run.host_set(0))
    pinned = flat.pin_memory()  # the step's inputs, packed as the device sets are
    nb = 2 if run.n_sets >= 2 else 1
    dev = [run.sets[b] for b in range(nb)]
    assert all(d["_flat"].numel() == pinned.numel() for d in dev)
    out_host = [torch.empty(run.out.shape, dtype=torch.float32).pin_memory() for _ in range(nb)]
    h2d = pinned.numel()
    d2h = out_host[0].numel() * 4
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    h2d_done = [torch.cuda.Event() for _ in range(nb)]
    free = [torch.cuda.Event() for _ in range(nb)]  # the step that read buffer b is done

    def copy_in(i):
        b = i % nb
        copy.wait_event(free[b])
        with torch.cuda.stream(copy):
            dev[b]["_flat"].copy_(pinned, non_blocking=True)  # one copy per step
        h2d_done[b].record(copy)

    def compute(i):
        b = i % nb
        main.wait_event(h2d_done[b])
        run.step(dev[b])
        free[b].record(main)
        out_host[b].copy_(run.out, non_blocking=True)

    def run_steps(n, start):
        copy.wait_event(start)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    for b in range(nb):
        free[b].record(main)
    warm = torch.cuda.Event()
    warm.record(main)
    run_steps(3, warm)
    torch.cuda.synchronize()
    barrier(world)
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    run_steps(steps, a)
    b_.record(main)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b_), world)
    value = frames_per_step(w) * steps * world / (ms / 1e3)
    return {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "overlap": "inputs of step i+1 copied on a second stream during step i",
            "copies_per_step": {"h2d": 1, "d2h": 1}}


# --------------------------------------------------------------------------- CPU oracle

ORACLE_SAMPLE_FLOPS = 3.0e10  # attention work of one sampled oracle step (a few seconds)


def oracle_sample_rows(w: dict) -> int:
    """Query rows (all heads) of the oracle's sampled step: a fixed amount
    of attention work, so the CPU baseline and the reference arm time the
    same sample of a workload."""
    per_row = 4.0 * w["H"] * w["key_cap"] * w["d"]
    return int(np.clip(ORACLE_SAMPLE_FLOPS / per_row, 16, w["q_rows"]))


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_step_time(w: dict, rows: int, seed: int = 0) -> dict:
    """Time the oracle on one sampled step of the workload: `rows` query
    rows (all heads, chosen by `seed`) of the attention, and in full the
    K/V push (video), the R-CFG update and the SSF / motion work.  Returns
    the measured time and the full-step time extrapolated from it (the
    attention linearly in the rows)."""
    from oracle import oracle as O
    S = w["streams"]
    rng = np.random.default_rng(seed)
    rows = min(rows, w["q_rows"])
    sel = np.sort(rng.choice(w["q_rows"], size=rows, replace=False)).astype(np.int64)
    q = W.gen_q(w, seed)
    k, v = W.gen_kv(w, seed)
    lat = W.gen_latents(w, seed)
    t_begin = time.perf_counter()
    st = O.Stream(w)
    t_push = 0.0
    if w["mode"] == "video":
        nchunks = max(1, -(-w["R"] // w["T"]))
        t0 = time.perf_counter()
        for c in range(nchunks):
            st.push(k[0], v[0])
        t_push = (time.perf_counter() - t0) / nchunks
        st.sink_refresh(np.ones(w["D"], dtype=np.float32))
        t0 = time.perf_counter()
        st.attend(q[0], sel)
        t_att = time.perf_counter() - t0
    else:
        t0 = time.perf_counter()
        O.attention(q[0], k[0], v[0], rows=sel)
        t_att = time.perf_counter() - t0
    t0 = time.perf_counter()
    z = lat["z"][:, 0] if w["n"] > 1 else None
    st.step_update(lat["x"][:, 0], lat["x0"][:, 0], lat["eps_c"][:, 0], z, lat["x0_new"][0],
                   lat["eps_new"][0])
    if w["ssf"]:
        f = W.FrameWalk(w).next()[0]
        st.ssf(f, 0.5)
        st.ssf(f, 0.5)
    if w["motion"]:
        lw = W.LatentWalk(w)
        st.motion(lw.next()[0])
    t_upd = time.perf_counter() - t0
    st.close()
    t_measured = time.perf_counter() - t_begin
    t_step = S * (t_push + t_att * (w["q_rows"] / rows) + t_upd)
    return {"t_step": t_step, "t_measured": t_measured, "rows": rows, "t_att": t_att,
            "t_fixed": t_push + t_upd}


def _sample_text(w: dict, rows: int) -> str:
    return (f"{rows} of {w['q_rows']} query rows (all {w['H']} heads) of one step's attention, "
            f"timed and extrapolated linearly to the full step; in full: R-CFG update"
            + (", SSF" if w["ssf"] else "") + (", motion" if w["motion"] else "")
            + (", K/V push" if w["mode"] == "video" else ""))


def cpu_baseline(w: dict) -> dict:
    """The oracle on the host cores: one sampled step on all cores, and a
    smaller sample on one thread."""
    from oracle import oracle as O
    cores = O.max_threads()
    rows = oracle_sample_rows(w)
    r = oracle_step_time(w, rows, seed=0)
    value = frames_per_step(w) / r["t_step"]
    out = {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": _sample_text(w, rows), "cpu_model": cpu_model(),
           "s_per_sampled_step": round(r["t_measured"], 3),
           "s_per_step_extrapolated": round(r["t_step"], 3)}
    rows1 = max(4, rows // 16)
    O.set_threads(1)
    try:
        r1 = oracle_step_time(w, rows1, seed=0)
    finally:
        O.set_threads(cores)
    out["one_thread"] = {"value": round(frames_per_step(w) / r1["t_step"], 5), "unit": UNIT,
                         "cores": 1, "sample": _sample_text(w, rows1),
                         "s_per_sampled_step": round(r1["t_measured"], 3),
                         "s_per_step_extrapolated": round(r1["t_step"], 3)}
    return out


def run_reference(args):
    """The oracle as the reference arm: each step is the sampled step of
    cpu_baseline (same rows), on the host cores; ms_per_step is the measured
    time of a sampled step, value the frames/s of the extrapolated full step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    w = workload(args)
    cores = O.max_threads()
    steps, warm = args.steps, args.warmup
    rows = oracle_sample_rows(w)
    for i in range(warm):
        oracle_step_time(w, rows, seed=0)
    t0 = time.perf_counter()
    rs = [oracle_step_time(w, rows, seed=0) for _ in range(steps)]
    wall = time.perf_counter() - t0
    t_full = float(np.mean([r["t_step"] for r in rs]))
    value = frames_per_step(w) / t_full
    line = {"metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": 0,
            "steps": steps, "warmup": warm, "ms_per_step": round(wall / steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w["name"], "streams_per_gpu": w["streams"]},
            "value_basis": "frames per extrapolated full step; ms_per_step is the measured "
                           "time of one sampled step",
            "ms_per_full_step_extrapolated": round(t_full * 1e3, 1),
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": _sample_text(w, rows),
                             "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Frames/s of the step for B = 1..N concurrent streams in one context:
    the throughput curve whose flattening is the roofline knee."""
    import torch
    torch.cuda.set_device(0)
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    rows = []
    for b in range(1, args.sweep_streams + 1):
        w = W.get_config(args.workload, streams=b)
        run = Runner(w, pool_bytes_min=2.0 * l2)
        for i in range(max(3, args.warmup)):
            run.step(run.sets[i % run.n_sets])
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(args.steps):
            run.step(run.sets[i % run.n_sets])
        e.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(e) / args.steps
        run.close()
        fps = frames_per_step(w) / (ms / 1e3)
        rows.append({"streams": b, "ms_per_step": round(ms, 4), "frames_per_s": round(fps, 1),
                     "per_stream_frames_per_s": round(fps / b, 1),
                     "attn_tflops": round(attn_flops(w) / (ms / 1e3) / 1e12, 1)})
        print(json.dumps({"sweep": args.workload, **rows[-1]}), flush=True)
    gains = [rows[i]["frames_per_s"] / rows[i - 1]["frames_per_s"] for i in range(1, len(rows))]
    knee = next((rows[i]["streams"] for i, g in enumerate(gains) if g < 1.05), rows[-1]["streams"])
    # the library's SLO controller fed with the measured step latencies
    from streaming_diffusion_stream_b300 import binding as B
    T = frames_per_step(W.get_config(args.workload, streams=1))
    choices = {}
    for fps in (30.0, 120.0, 1000.0, 3000.0):
        ctl = B.SloController(fps, T, 1, args.sweep_streams)
        for r in rows:
            ctl.observe(r["streams"], r["ms_per_step"] / 1e3)
        c = ctl.choose()
        ctl.close()
        choices[str(fps)] = {"streams": c["batch"], "meets_slo": c["meets_slo"],
                             "per_stream_fps": round(c["per_stream_fps"], 1),
                             "b_slo": c["b_slo"], "b_knee": c["b_knee"]}
    print(json.dumps({"sweep_summary": args.workload, "knee_streams": knee,
                      "frames_per_s": [r["frames_per_s"] for r in rows],
                      "slo_controller": choices}), flush=True)


def main():
    args = parse()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 300
    if args.warmup is None:
        args.warmup = 3 if args.impl == "reference" else 20
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep_streams:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
