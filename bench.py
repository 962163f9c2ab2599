#!/usr/bin/env python3
"""Benchmark of the Q4 dequant-in-GEMV hot path on the synthetic decode step.

One step = one pass of the whole fused path over one batch: 16 layers of
(RMSNorm+q/k/v, o+residual, RMSNorm+gate/up+SwiGLU, down+residual) then
RMSNorm + a 65536 x 2048 logits projection + argmax, all Q4_0, hidden 2048,
kv 512, intermediate 8192, nb = 1, run by ``q4_decode_step`` as one
persistent kernel and replayed from a CUDA graph.  622,854,144 weight bytes
stream from HBM per step (more than L2 holds), so every step reads cold
weights.

Prints ONE JSON line (rank 0).  ``value`` is weight GB/s of the whole job
(all ranks), ``ms_per_step`` the step time; ``e2e`` repeats the measure with
the step's inputs copied from pinned host memory and its result read back
inside the timed region; ``roofline`` is the decode-step kernel against the
measured HBM peak; ``graph_of_calls`` times the same step as 82 separate
library calls in one graph; ``cpu_baseline`` is the f64 C oracle on the
host.  ``--impl reference`` times the oracle itself as the
reference arm.  Multi-GPU (torchrun) runs independent replicas (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4 GEMV weight GB/s (fraction of GB300 HBM peak) and µs per fused decode-step"
WORKLOAD = ("synthetic 16-layer Q4_0 decode step, nb=1, hidden 2048, kv 512, intermediate 8192, "
            "logits 65536 x 2048 + argmax, one persistent kernel replayed from a CUDA graph")
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--no-kernels", action="store_true", help="skip the per-shape kernel table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--gemv", metavar="FMT:N:K:NB", default=None,
                    help="time one q4_gemv shape only (fmt q4_0, affine, q8_0, q4_k or q1; for profiling), then exit")
    ap.add_argument("--gemm", metavar="FMT:N:K:NB", default=None,
                    help="time one q4_gemm shape only (for profiling), then exit")
    ap.add_argument("--attn", metavar="H:HKV:D:CTX", default=None,
                    help="time one q4_attn_decode shape only (the token at position CTX-1, RoPE on; for "
                         "profiling), then exit")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device="cpu") -> float:
    """Maximum of a per-rank float over all ranks (the job's wall time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(bytes_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job weight GB/s: every rank streams its own replica's weights."""
    return bytes_per_step * steps * world / max_seconds / 1e9


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, power, reasons, n = [], [], [], set(), 0
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        top = max(power) if power else 0.0
        loaded = [s for s, p in zip(sm, power) if p >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": n, "power_w_max": top}


# ----------------------------------------------------------------- peaks

def measured_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources that define the persistent decode-step kernel and its launch
STEP_SOURCES = ("attn_common.cuh", "capi.cu", "gemv_kernel.cuh", "gemv_launch.cuh", "gemv_q4_0.cu", "q4_internal.h",
                "step_attn.cuh")


def kernel_source_hash(names=STEP_SOURCES) -> str:
    """Hash of the CUDA sources of a kernel (by default the decode step's): a
    profile summary taken on other sources is stale."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_weight_quantized_q4_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str) -> float | None:
    """DRAM bytes per launch from profiles/traffic.txt (lines of
    ``tag source_hash=<h> dram_bytes_per_launch=<n>``), if it was taken on the
    current kernel sources, else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(p) as f:
            for ln in f:
                parts = ln.split()
                if not parts or parts[0] != kernel_tag:
                    continue
                kv = dict(x.split("=", 1) for x in parts[1:] if "=" in x)
                if kv.get("source_hash") != kernel_source_hash():
                    return None
                return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None
    return None


# ------------------------------------------------------------ our arm

def time_replays(graph, steps: int, stream) -> float:
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


class _GraphEvent:
    """A timing event that becomes an event-record node when recorded during
    stream capture (cudaEventRecordExternal), via torch when it supports it,
    else through the CUDA runtime directly."""
    _rt = None

    def __init__(self):
        import torch
        try:
            self.ev = torch.cuda.Event(enable_timing=True, external=True)
            self.raw = None
        except TypeError:
            self.ev = None
            rt = _GraphEvent.runtime()
            h = ctypes.c_void_p()
            if rt.cudaEventCreate(ctypes.byref(h)) != 0:
                raise RuntimeError("cudaEventCreate failed")
            self.raw = h

    @classmethod
    def runtime(cls):
        if cls._rt is None:
            import glob
            import torch
            names = ["libcudart.so.13", "libcudart.so"]
            base = os.path.dirname(torch.__file__)
            names += glob.glob(os.path.join(base, "..", "nvidia", "cu13", "lib", "libcudart.so*"))
            names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
            for n in names:
                try:
                    cls._rt = ctypes.CDLL(n)
                    break
                except OSError:
                    continue
            if cls._rt is None:
                raise RuntimeError("libcudart not found")
        return cls._rt

    def record(self):
        import torch
        if self.ev is not None:
            self.ev.record()
            return
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        if self.runtime().cudaEventRecordWithFlags(self.raw, st, 1) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")

    def elapsed_ms(self, other) -> float:
        if self.ev is not None:
            return self.ev.elapsed_time(other.ev)
        ms = ctypes.c_float()
        if self.runtime().cudaEventElapsedTime(ctypes.byref(ms), self.raw, other.raw) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return ms.value


def kernel_timing(step, steps: int, fused: bool, name: str = "gus"):
    """Average duration of one kernel inside the step, from timing events
    captured around each of its launches in a graph of the step, replayed
    `steps` times: the persistent step kernel (fused) or every launch of the
    call named `name` (call-by-call step)."""
    import torch
    evs = []
    if fused:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step.run_fused()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        a, b = _GraphEvent(), _GraphEvent()
        with torch.cuda.graph(g):
            a.record()
            step.run_fused()   # includes the 16-byte clear of the barrier counter
            b.record()
        evs.append((a, b))
    else:
        def around(nm, l, fn):
            if nm != name:
                return fn()
            a, b = _GraphEvent(), _GraphEvent()
            a.record()
            fn()
            b.record()
            evs.append((a, b))
        g = step.capture(around=around)
    durs = []
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        durs += [a.elapsed_ms(b) * 1e3 for a, b in evs]
    return statistics.mean(durs), len(durs)


def e2e_timing(step, graph, steps: int, warmup: int):
    """Step inputs (x and the attention stand-ins) copied in from pinned host
    memory and the argmax read back, inside the timed region."""
    import torch
    # the inputs (x, then every layer's attention stand-in) are one device
    # buffer and come in with one copy; the results (indices, then their
    # logits) go out with one copy of the words up to the last logit
    host_in = step.inputs.cpu().pin_memory()
    res = step.results[:16 + step.nb]
    host_out = torch.empty(res.shape, dtype=res.dtype).pin_memory()
    stream = torch.cuda.current_stream()

    def one():
        step.inputs.copy_(host_in, non_blocking=True)
        graph.replay()
        host_out.copy_(res, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


KT_REPLAYS = 15  # timed graph replays per kernel-table row


class Timed(float):
    """A per-call time in seconds: the median over the timed replays (each
    replay a graph of back-to-back calls), carrying their 10th and 90th
    percentiles."""

    def __new__(cls, per_call):
        import numpy as np
        p10, p50, p90 = (float(v) for v in np.percentile(np.asarray(per_call, dtype=np.float64), [10, 50, 90]))
        self = super().__new__(cls, p50)
        self.p10, self.p90 = p10, p90
        return self


def spread(t) -> dict:
    """The p10 / p90 fields of a kernel-table row (µs), for a Timed value."""
    if not isinstance(t, Timed):
        return {}
    return {"us_p10": round(t.p10 * 1e6, 3), "us_p90": round(t.p90 * 1e6, 3)}


def stream_ceiling(Ws, bench_calls, peak: float, tag: str) -> dict:
    """What one launch of a library kernel reaches on the same packed bytes,
    over the same rotation and back-to-back graph as the GEMV rows: a
    device-to-device copy (cudaMemcpyAsync through tensor.copy_; it reads
    and writes every byte) and a library reduction that only reads them (a
    sum over their int32 view).  The per-launch ceiling for streaming this
    many bytes once, measured beside the GEMV on every run."""
    import torch
    nbytes = Ws[0].tensor.numel()
    dsts = [torch.empty_like(W.tensor) for W in Ws]
    by_id = {id(W): i for i, W in enumerate(Ws)}
    t_copy = bench_calls(Ws, lambda W: dsts[by_id[id(W)]].copy_(W.tensor))
    t_read = bench_calls(Ws, lambda W: W.tensor.view(torch.int32).sum())
    del dsts
    return {
        tag + "_copy": {"us": round(t_copy * 1e6, 3), **spread(t_copy),
                        "read_gbs": round(nbytes / t_copy / 1e9, 1),
                        "read_write_gbs": round(2 * nbytes / t_copy / 1e9, 1),
                        "frac_of_hbm": round(2 * nbytes / t_copy / 1e9 / peak, 4),
                        "what": "device-to-device copy of the packed bytes (reads and writes each byte)"},
        tag + "_library_read": {"us": round(t_read * 1e6, 3), **spread(t_read),
                                "read_gbs": round(nbytes / t_read / 1e9, 1),
                                "frac_of_hbm": round(nbytes / t_read / 1e9 / peak, 4),
                                "what": "torch int32 sum over the packed bytes: a library kernel reading each byte once"},
    }


def kernel_table(device, l2_bytes: int, peak: float, reps: int = 48) -> dict:
    """Per-shape cold timings of single calls: a graph of `reps` back-to-back
    calls over rotating weight copies whose total exceeds 3x L2, replayed
    KT_REPLAYS times; `us` is the median per call, `us_p10` / `us_p90` the
    spread over the replays."""
    import numpy as np
    import torch

    import bit_weight_quantized_q4_gb300 as q4
    import q4_workloads as wl
    out = {}
    rng = np.random.default_rng(3)
    n, k = 14336, 4096

    def bench_calls(weights, fn):
        # every copy at least once per replay, so a replay touches > 3x L2
        n_calls = max(reps, len(weights))
        g = torch.cuda.CUDAGraph()
        fn(weights[0])
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(n_calls):
                fn(weights[i % len(weights)])
        g.replay()
        torch.cuda.synchronize()
        return Timed([time_replays(g, 1, torch.cuda.current_stream()) / n_calls for _ in range(KT_REPLAYS)])

    for fmt in ("affine", "q4_0", "q8_0", "q4_k", "q1"):
        H = wl._draw_fmt(fmt)(rng, n, k)
        W0 = (q4.Q4Weight.from_affine(H.nib, H.s, H.m, n, k, device) if fmt == "affine"
              else q4.Q4Weight.from_q8_0(H.blocks8, n, k, device) if fmt == "q8_0"
              else q4.Q4Weight.from_q4_k(H.blocks_k, n, k, device) if fmt == "q4_k"
              else q4.Q4Weight.from_q1(H.blocks1, n, k, device) if fmt == "q1"
              else q4.Q4Weight.from_q4_0(H.blocks, n, k, device))
        copies = max(2, -(-3 * l2_bytes // W0.nbytes))
        host = W0.tensor.cpu().numpy()
        Ws = [W0] + [q4.Q4Weight(W0.fmt, n, k, host, device) for _ in range(copies - 1)]
        if fmt in ("affine", "q4_0"):
            # context: a vendor reduction (torch.amax) reading the same packed bytes, same rotation
            t_ref = bench_calls(Ws, lambda W: torch.amax(W.tensor))
            out["%s_n%d_k%d_vendor_read" % (fmt, n, k)] = {
                "us": round(t_ref * 1e6, 3), **spread(t_ref), "packed_gbs": round(W0.nbytes / t_ref / 1e9, 1),
                "what": "torch.amax over the packed weight bytes: a library kernel reading the same bytes"}
        for nb in ((1, 2, 4, 8, 16) if fmt == "affine" else (1,)):
            x = torch.from_numpy(wl.draw_x(rng, nb, k)).to(device)
            y = torch.empty((nb, n), dtype=torch.float32, device=device)
            t = bench_calls(Ws, lambda W: q4.q4_gemv(W, x, out=y))
            gbs = W0.weight_bytes / t / 1e9
            out["%s_n%d_k%d_nb%d" % (fmt, n, k, nb)] = {"us": round(t * 1e6, 3), **spread(t),
                                                      "weight_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4)}
            if fmt == "q4_0":
                # warm: one copy reused, its bytes resident in L2 between calls
                t = bench_calls([W0], lambda W: q4.q4_gemv(W, x, out=y))
                gbs = W0.weight_bytes / t / 1e9
                out["%s_n%d_k%d_nb%d_warm" % (fmt, n, k, nb)] = {
                    "us": round(t * 1e6, 3), **spread(t), "weight_gbs": round(gbs, 1),
                    "what": "one weight copy reused: warm, its bytes in L2 (not an HBM figure)"}
        if fmt == "affine":
            # the prefill GEMM at verify widths: one weight stream shared by a
            # 16-row activation tile (staging pass included)
            for nb in (8, 16):
                x = torch.from_numpy(wl.draw_x(rng, nb, k)).to(device)
                y = torch.empty((nb, n), dtype=torch.float32, device=device)
                wsg = torch.empty(int(q4.lib().q4_gemm_workspace_bytes(nb, k)), dtype=torch.uint8, device=device)
                t = bench_calls(Ws, lambda W: q4.q4_gemm(W, x, out=y, workspace=wsg))
                gbs = W0.weight_bytes / t / 1e9
                out["%s_n%d_k%d_nb%d_gemm" % (fmt, n, k, nb)] = {
                    "us": round(t * 1e6, 3), **spread(t), "weight_gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / peak, 4)}
            # the same matvec fed a HalfSet (f16 even/odd streams + group sums,
            # packed once): what a caller verifying several drafts per step runs
            for nb in (8, 16):
                x = torch.from_numpy(wl.draw_x(rng, nb, k)).to(device)
                xe, xo, gs = q4.q4_pack_half(x)
                y = torch.empty((nb, n), dtype=torch.float32, device=device)
                t = bench_calls(Ws, lambda W: q4.q4_gemv_half(W, xe, xo, gsum=gs, out=y))
                gbs = W0.weight_bytes / t / 1e9
                out["%s_n%d_k%d_nb%d_halfset" % (fmt, n, k, nb)] = {
                    "us": round(t * 1e6, 3), **spread(t), "weight_gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / peak, 4)}
        if fmt == "q4_0":
            out.update(stream_ceiling(Ws, bench_calls, peak, "%s_n%d_k%d" % (fmt, n, k)))
        del Ws
        torch.cuda.empty_cache()
    # the fused calls at the small workload shapes (cfg 0..2), cold: each
    # call's weights rotate over copies totalling more than 3x L2
    def copies_of(H, count):
        W0 = q4.Q4Weight.from_q4_0(H.blocks, H.n, H.k, device)
        host = W0.tensor.cpu().numpy()
        return [W0] + [q4.Q4Weight(W0.fmt, H.n, H.k, host, device) for _ in range(count - 1)]

    def count_for(*Hs):
        total = sum(wl_bytes(H) for H in Hs)
        return max(2, -(-3 * l2_bytes // total))

    def wl_bytes(H):
        return H.n * H.k // 32 * 18

    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    c0 = wl.cfg0()
    Ws = copies_of(c0.W, count_for(c0.W))
    x0, y0 = T(c0.x), torch.empty((1, c0.W.n), dtype=torch.float32, device=device)
    t = bench_calls(Ws, lambda W: q4.q4_gemv(W, x0, out=y0))
    out["cfg0_q4_gemv_1024x1024"] = {"us": round(t * 1e6, 3), **spread(t),
                                     "weight_gbs": round(Ws[0].weight_bytes / t / 1e9, 1)}
    del Ws
    c1 = wl.cfg1()
    cnt = count_for(c1.Wq, c1.Wk, c1.Wv)
    Wq, Wk, Wv = copies_of(c1.Wq, cnt), copies_of(c1.Wk, cnt), copies_of(c1.Wv, cnt)
    x1, g1 = T(c1.x), T(c1.gamma)
    yq = torch.empty((1, c1.Wq.n), dtype=torch.float32, device=device)
    yk = torch.empty((1, c1.Wk.n), dtype=torch.float32, device=device)
    yv = torch.empty((1, c1.Wv.n), dtype=torch.float32, device=device)
    t = bench_calls(list(range(cnt)), lambda i: q4.q4_nrm_gemv(Wq[i], x1, g1, c1.eps, out=yq))
    out["cfg1_q4_nrm_gemv_2048x2048"] = {"us": round(t * 1e6, 3), **spread(t),
                                         "weight_gbs": round(Wq[0].weight_bytes / t / 1e9, 1)}
    t = bench_calls(list(range(cnt)), lambda i: q4.q4_dual_gemv(Wk[i], Wv[i], x1, g1, c1.eps, out_a=yk, out_b=yv))
    out["cfg1_q4_dual_gemv_2x512x2048"] = {"us": round(t * 1e6, 3), **spread(t),
                                           "weight_gbs": round(2 * Wk[0].weight_bytes / t / 1e9, 1)}
    del Wq, Wk, Wv
    c2 = wl.cfg2()
    cnt = count_for(c2.Wg, c2.Wu)
    Wg, Wu = copies_of(c2.Wg, cnt), copies_of(c2.Wu, cnt)
    x2, g2 = T(c2.x), T(c2.gamma)
    h2 = torch.empty((1, c2.Wg.n), dtype=torch.float32, device=device)
    t = bench_calls(list(range(cnt)), lambda i: q4.q4_gus_nrm(Wg[i], Wu[i], x2, g2, c2.eps, out=h2))
    out["cfg2_q4_gus_nrm_2x8192x2048"] = {"us": round(t * 1e6, 3), **spread(t),
                                          "weight_gbs": round(2 * Wg[0].weight_bytes / t / 1e9, 1),
                                          "frac_of_hbm": round(2 * Wg[0].weight_bytes / t / 1e9 / peak, 4)}
    del Wg, Wu
    cnt = count_for(c2.Wd)
    Wd = copies_of(c2.Wd, cnt)
    r2 = T(c2.r)
    yd = torch.empty((1, c2.Wd.n), dtype=torch.float32, device=device)
    t = bench_calls(list(range(cnt)), lambda i: q4.q4_res_gemv(Wd[i], h2, r2, out=yd))
    out["cfg2_q4_res_gemv_2048x8192"] = {"us": round(t * 1e6, 3), **spread(t),
                                         "weight_gbs": round(Wd[0].weight_bytes / t / 1e9, 1),
                                         "frac_of_hbm": round(Wd[0].weight_bytes / t / 1e9 / peak, 4)}
    del Wd
    torch.cuda.empty_cache()
    # the same nb = 1 Q4_0 kernel on a 4x taller matrix (132 MB per call): the
    # per-launch ramp and tail are amortised over 4x the bytes, which shows how
    # fast the kernel streams once it is running
    n4 = 4 * n
    H = wl.draw_q4_0(rng, n4, k)
    W0 = q4.Q4Weight.from_q4_0(H.blocks, n4, k, device)
    copies = max(2, -(-3 * l2_bytes // W0.nbytes))
    host = W0.tensor.cpu().numpy()
    Ws = [W0] + [q4.Q4Weight(W0.fmt, n4, k, host, device) for _ in range(copies - 1)]
    x = torch.from_numpy(wl.draw_x(rng, 1, k)).to(device)
    y = torch.empty((1, n4), dtype=torch.float32, device=device)
    t = bench_calls(Ws, lambda W: q4.q4_gemv(W, x, out=y))
    gbs = W0.weight_bytes / t / 1e9
    out["q4_0_n%d_k%d_nb1" % (n4, k)] = {"us": round(t * 1e6, 3), **spread(t), "weight_gbs": round(gbs, 1),
                                         "frac_of_hbm": round(gbs / peak, 4),
                                         "what": "4x the rows of the 14336 x 4096 case: launch overhead amortised"}
    out.update(stream_ceiling(Ws, bench_calls, peak, "q4_0_n%d_k%d" % (n4, k)))
    del Ws
    torch.cuda.empty_cache()
    # the prefill GEMM on the 14336 x 4096 Q4_0 projection at 64, 256 and 512
    # activation rows (one weight copy reused: its 33 MB stay partly in L2,
    # which a prefill chunk also sees; the activations are new each call)
    H = wl.draw_q4_0(rng, n, k)
    Wg = q4.Q4Weight.from_q4_0(H.blocks, n, k, device)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        bf16_peak = None
    for nbg in (64, 256, 512):
        xg = torch.from_numpy(wl.draw_x(rng, nbg, k)).to(device)
        yg = torch.empty((nbg, n), dtype=torch.float32, device=device)
        wsg = torch.empty(int(q4.lib().q4_gemm_workspace_bytes(nbg, k)), dtype=torch.uint8, device=device)
        t = bench_calls([Wg], lambda W: q4.q4_gemm(W, xg, out=yg, workspace=wsg))
        tf = 2.0 * n * k * nbg / t / 1e12
        out["gemm_q4_0_n%d_k%d_nb%d" % (n, k, nbg)] = {
            "us": round(t * 1e6, 3), **spread(t), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / bf16_peak, 4) if bf16_peak else None,
            "what": ("staging pass + GEMM (tcgen05 f16 MMAs into tensor memory; weights exact as f16 hi + lo "
                     "pairs, so the tensor work is twice the algorithmic flops counted here; fp32 accumulate); "
                     "peak: measured cuBLAS bf16")}
    del Wg
    torch.cuda.empty_cache()
    # decode attention of one token (RoPE, KV append, softmax(q K^T) V) at
    # 32 query heads, 8 kv heads, head size 64, over 4096 and 32768 cached
    # positions; the f32 caches rotate over copies totalling > 3x L2
    H_, Hkv_, D_ = 32, 8, 64
    for ctx in (4096, 32768):
        kv_bytes = 2 * Hkv_ * ctx * D_ * 4
        copies = max(2, -(-3 * l2_bytes // kv_bytes))
        caches = [(torch.randn(Hkv_, ctx, D_, device=device), torch.randn(Hkv_, ctx, D_, device=device))
                  for _ in range(copies)]
        c_, s_ = q4.rope_table(ctx, D_, 10000.0)
        tables = (torch.from_numpy(c_).to(device), torch.from_numpy(s_).to(device))
        qa = torch.randn(H_, D_, device=device)
        kn_, vn_ = torch.randn(Hkv_, D_, device=device), torch.randn(Hkv_, D_, device=device)
        oa = torch.empty(H_, D_, device=device)
        ws = torch.zeros(int(q4.lib().q4_attn_workspace_bytes(H_, D_, ctx)), dtype=torch.uint8, device=device)
        t = bench_calls(caches, lambda kv: q4.q4_attn_decode(qa, kn_, vn_, kv[0], kv[1], ctx - 1, 0, None,
                                                            rope=tables, out=oa, workspace=ws))
        gbs = kv_bytes / t / 1e9
        out["attn_decode_h%d_kv%d_d%d_ctx%d" % (H_, Hkv_, D_, ctx)] = {
            "us": round(t * 1e6, 3), **spread(t), "kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
            "what": "f32 K and V rows of every kv head read once per call"}
        del caches
        torch.cuda.empty_cache()
    return out


def run_one_gemv(args) -> dict:
    """One GEMV shape, `warmup` untimed then `steps` timed calls on one weight
    (seeded synthetic, drawn like the kernel table's); for ncu captures."""
    import numpy as np
    import torch

    import bit_weight_quantized_q4_gb300 as q4
    import q4_workloads as wl
    fmt, n, k, nb = args.gemv.split(":")
    n, k, nb = int(n), int(k), int(nb)
    q4.build()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(3)
    H = wl._draw_fmt(fmt)(rng, n, k)
    W = (q4.Q4Weight.from_affine(H.nib, H.s, H.m, n, k, dev) if fmt == "affine"
         else q4.Q4Weight.from_q8_0(H.blocks8, n, k, dev) if fmt == "q8_0"
         else q4.Q4Weight.from_q4_k(H.blocks_k, n, k, dev) if fmt == "q4_k"
         else q4.Q4Weight.from_q1(H.blocks1, n, k, dev) if fmt == "q1"
         else q4.Q4Weight.from_q4_0(H.blocks, n, k, dev))
    x = torch.from_numpy(wl.draw_x(rng, nb, k)).to(dev)
    y = torch.empty((nb, n), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        q4.q4_gemv(W, x, out=y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        q4.q4_gemv(W, x, out=y)
    e1.record()
    torch.cuda.synchronize()
    q4.q4_device_check()
    return {"gemv": args.gemv, "calls": args.steps, "us_per_call_warm_l2": round(e0.elapsed_time(e1) * 1e3 / args.steps, 3),
            "note": "one weight reused: warm L2 for matrices under 129 MB; the kernel table times cold weights"}


def run_one_gemm(args) -> dict:
    """One prefill-GEMM shape, `warmup` untimed then `steps` timed calls on
    one weight; for ncu captures."""
    import numpy as np
    import torch

    import bit_weight_quantized_q4_gb300 as q4
    import q4_workloads as wl
    fmt, n, k, nb = args.gemm.split(":")
    n, k, nb = int(n), int(k), int(nb)
    q4.build()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(3)
    H = wl._draw_fmt(fmt)(rng, n, k)
    W = (q4.Q4Weight.from_affine(H.nib, H.s, H.m, n, k, dev) if fmt == "affine"
         else q4.Q4Weight.from_q8_0(H.blocks8, n, k, dev) if fmt == "q8_0"
         else q4.Q4Weight.from_q4_k(H.blocks_k, n, k, dev) if fmt == "q4_k"
         else q4.Q4Weight.from_q1(H.blocks1, n, k, dev) if fmt == "q1"
         else q4.Q4Weight.from_q4_0(H.blocks, n, k, dev))
    x = torch.from_numpy(wl.draw_x(rng, nb, k)).to(dev)
    y = torch.empty((nb, n), dtype=torch.float32, device=dev)
    ws = torch.empty(int(q4.lib().q4_gemm_workspace_bytes(nb, k)), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        q4.q4_gemm(W, x, out=y, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        q4.q4_gemm(W, x, out=y, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    q4.q4_device_check()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    return {"gemm": args.gemm, "calls": args.steps, "us_per_call": round(us, 3),
            "tflops": round(2.0 * n * k * nb / us / 1e6, 1)}


def run_one_attn(args) -> dict:
    """One decode-attention shape, `warmup` untimed then `steps` timed calls
    on one pair of caches; for ncu captures."""
    import torch

    import bit_weight_quantized_q4_gb300 as q4
    H, Hkv, D, ctx = (int(v) for v in args.attn.split(":"))
    q4.build()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(5)
    kc = torch.randn(Hkv, ctx, D, device=dev, generator=g)
    vc = torch.randn(Hkv, ctx, D, device=dev, generator=g)
    q = torch.randn(H, D, device=dev, generator=g)
    kn, vn = torch.randn(Hkv, D, device=dev, generator=g), torch.randn(Hkv, D, device=dev, generator=g)
    c, sn = q4.rope_table(ctx, D, 10000.0)
    tables = (torch.from_numpy(c).to(dev), torch.from_numpy(sn).to(dev))
    out = torch.empty(H, D, device=dev)
    ws = torch.zeros(int(q4.lib().q4_attn_workspace_bytes(H, D, ctx)), dtype=torch.uint8, device=dev)
    call = lambda: q4.q4_attn_decode(q, kn, vn, kc, vc, ctx - 1, 0, None, rope=tables, out=out, workspace=ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    q4.q4_device_check()
    kv_bytes = 2 * Hkv * ctx * D * 4
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    return {"attn": args.attn, "calls": args.steps, "us_per_call_warm_l2": round(us, 3), "kv_bytes": kv_bytes,
            "note": "one pair of caches reused: warm L2 when they fit in 129 MB; the kernel table times cold caches"}


def workload_config(args, wbytes: int, l2: int, world: int) -> dict:
    """The `config` object of both arms (same keys, same values)."""
    return {"workload": WORKLOAD, "layers": args.layers, "nb": 1, "weight_bytes_per_step": wbytes,
            "l2": "inputs larger than L2: %d weight bytes per step vs %d B L2" % (wbytes, l2),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def l2_bytes() -> int:
    try:
        import torch
        if torch.cuda.is_available():
            return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or 0)
    except Exception:
        pass
    return 0


def run_ours(args, rank, world, local):
    import torch

    import bit_weight_quantized_q4_gb300 as q4
    import q4_workloads as wl
    from bit_weight_quantized_q4_gb300.decode import DecodeStep

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    q4.build()
    q4.lib()

    cfg = wl.cfg4(layers=args.layers)
    step = DecodeStep(cfg, device)
    wbytes = step.weight_bytes
    graph = step.capture(fused=True)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    step.run_fused()
    q4.q4_decode_check(step.step_ws)  # every grid barrier completed

    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "") or "")
    uuid = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else None
    clocks = ClockSampler(uuid).start()
    barrier(world)
    secs = time_replays(graph, args.steps, stream)
    barrier(world)
    clk = clocks.stop()
    max_secs = reduce_max(secs, world, device)
    value = job_rate(wbytes, args.steps, world, max_secs)
    ms_per_step = max_secs * 1e3 / args.steps

    peak, peak_src = measured_peaks()
    k_us, k_n = kernel_timing(step, max(3, min(args.steps, 10)), fused=True)
    achieved = wbytes / (k_us * 1e-6) / 1e9

    e2e_secs, h2d, d2h = e2e_timing(step, graph, args.steps, max(1, args.warmup))
    e2e_max = reduce_max(e2e_secs, world, device)

    # the same step as 82 separate library calls in one graph
    calls_graph = step.capture()
    for _ in range(max(1, args.warmup)):
        calls_graph.replay()
    calls_secs = time_replays(calls_graph, args.steps, stream)
    gus_us, _ = kernel_timing(step, 3, fused=False, name="gus")
    del calls_graph

    # the real step: each layer's decode attention over 4096 cached positions
    # (32 / 8 heads of 64) between K+V and the o projection, as library calls
    # in one graph; it reads the weights and every layer's K and V rows
    real = None
    if rank == 0 and world == 1 and not args.no_kernels:
        spec = wl.AttnSpec(max_seq=4096, position=4095)
        astep = DecodeStep(cfg, device, attention=(spec, wl.draw_kv_caches(4, args.layers, spec)))
        ag = astep.capture()
        for _ in range(max(1, args.warmup)):
            ag.replay()
        a_secs = time_replays(ag, args.steps, stream)
        a_bytes = astep.weight_bytes + astep.kv_bytes
        real = {"kernels_per_step": astep.n_kernels, "context": spec.position + 1,
                "us_per_step": round(a_secs * 1e6 / args.steps, 2),
                "bytes_per_step": a_bytes, "gbs": round(a_bytes * args.steps / a_secs / 1e9, 2),
                "frac_of_hbm_peak": round(a_bytes * args.steps / a_secs / 1e9 / peak, 4)}
        del ag
        # the same real step as one persistent kernel (q4_decode_step_attn)
        fg = astep.capture(fused=True)
        for _ in range(max(1, args.warmup)):
            fg.replay()
        f_secs = time_replays(fg, args.steps, stream)
        q4.q4_decode_check(astep.check_ws)
        real["persistent"] = {"kernels_per_step": 1, "us_per_step": round(f_secs * 1e6 / args.steps, 2),
                              "gbs": round(a_bytes * args.steps / f_secs / 1e9, 2),
                              "frac_of_hbm_peak": round(a_bytes * args.steps / f_secs / 1e9 / peak, 4)}
        del fg, astep
        torch.cuda.empty_cache()

    l2 = int(getattr(props, "L2_cache_size", 0) or 0)
    kernels = None
    if rank == 0 and world == 1 and not args.no_kernels:
        kernels = kernel_table(device, l2 or 128 << 20, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_sample(cfg, wbytes, budget_s=8.0)

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 hi+lo activations x exact f16 nibbles, f32 accumulate",
        "precision": "Q4_0 nibbles exact in f16; activations scaled per 32-column block by a power of two and split into f16 hi+lo (about 22 significant bits); fp32 accumulate",
        "data": "synthetic (seeded PCG64; q~U{0..15}, d~U[0.005,0.02] fp16, x~N(0,1), gamma=1+0.1N(0,1))",
        "config": workload_config(args, wbytes, l2, world),
        "kernels_per_step": 1,
        "gpu_launches": 1 * args.steps,
        "clocks": clk,
        "e2e": {"value": round(job_rate(wbytes, args.steps, world, e2e_max), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_max * 1e3 / args.steps, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": {"kernel": "q4gemv_step_kernel (q4_decode_step: the whole step, one persistent kernel)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src + " (MEASURED_PEAKS hbm_gbs)",
                     "algorithmic_bytes_per_launch": wbytes, "launch_us": round(k_us, 3),
                     "launches_timed": k_n, "traffic": profiled_traffic("decode_step_16layer")},
        "graph_of_calls": {"kernels_per_step": step.n_kernels,
                           "us_per_step": round(calls_secs * 1e6 / args.steps, 2),
                           "weight_gbs": round(wbytes * args.steps / calls_secs / 1e9, 2),
                           "gus_launch_us": round(gus_us, 3)},
    }
    if real is not None:
        line["step_with_attention"] = real
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if kernels is not None:
        line["kernels"] = kernels
    return line


# ---------------------------------------------------------- oracle arms

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_steps(cfg, threads: int, budget_s: float, max_steps: int):
    import oracle
    old = oracle.set_threads(threads)
    try:
        t0 = time.perf_counter()
        n = 0
        while True:
            oracle.decode_step(cfg)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s or n >= max_steps:
                return n, el
    finally:
        oracle.set_threads(old)


def cpu_rows(cores: int) -> dict:
    """The oracle beside the kernel table's other rows, on all host cores:
    the nb = 1 matvec of the 14336 x 4096 matrix in every format, the prefill
    GEMM at 64 rows (on a 1024-row slice, scaled to the whole matrix), and
    decode attention at 4096 cached positions (32 / 8 heads of 64)."""
    import numpy as np

    import oracle
    import q4_workloads as wl
    old = oracle.set_threads(cores)
    out = {}
    try:
        rng = np.random.default_rng(3)
        n, k = 14336, 4096
        for fmt in ("q4_0", "affine", "q8_0", "q4_k", "q1"):
            H = wl._draw_fmt(fmt)(rng, n, k)
            x = wl.draw_x(rng, 1, k)
            W = oracle._hw(H)
            t0 = time.perf_counter()
            oracle.q4_gemv(W, x)
            out["%s_n%d_k%d_nb1" % (fmt, n, k)] = {"ms": round((time.perf_counter() - t0) * 1e3, 2),
                                                   "sample": "one call"}
        Hs = wl.draw_q4_0(rng, 1024, k)
        x = wl.draw_x(rng, 64, k)
        t0 = time.perf_counter()
        oracle.q4_gemv(oracle._hw(Hs), x)
        el = time.perf_counter() - t0
        out["gemm_q4_0_n%d_k%d_nb64" % (n, k)] = {"ms": round(el * 1e3 * n / 1024, 1),
                                                  "sample": "1024 of the 14336 rows, scaled by 14"}
        H_, Hkv_, D_, ctx = 32, 8, 64, 4096
        kc = rng.standard_normal((Hkv_, ctx, D_))
        vc = rng.standard_normal((Hkv_, ctx, D_))
        q = rng.standard_normal((H_, D_))
        kn, vn = rng.standard_normal((Hkv_, D_)), rng.standard_normal((Hkv_, D_))
        c, sn = oracle.rope_table(ctx, D_, 10000.0)
        t0 = time.perf_counter()
        oracle.attn_decode(q, kn, vn, kc, vc, ctx - 1, 0, 0.125, c, sn)
        out["attn_decode_h%d_kv%d_d%d_ctx%d" % (H_, Hkv_, D_, ctx)] = {
            "ms": round((time.perf_counter() - t0) * 1e3, 2), "sample": "one call, 1 thread (heads in sequence)"}
    finally:
        oracle.set_threads(old)
    return out


def cpu_baseline_sample(cfg, wbytes: int, budget_s: float = 8.0) -> dict:
    """The f64 C oracle on whole decode steps of the same workload: on all
    host cores (the output rows of every GEMV split over threads; rows are
    independent and each output is computed by the same code), and on one
    thread, each repeated until about `budget_s` seconds have passed."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    n_all, el_all = _oracle_steps(cfg, cores, budget_s, 40)
    n_one, el_one = _oracle_steps(cfg, 1, budget_s, 10)
    rows = cpu_rows(cores)
    return {"rows": rows,
            "value": round(wbytes * n_all / el_all / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d full decode step(s) (%d weight bytes each) in the f64 C oracle on %d threads, %.1f s"
                      % (n_all, wbytes, cores, el_all),
            "cpu_model": cpu_model(), "nproc": cores,
            "ms_per_step": round(el_all * 1e3 / n_all, 1),
            "single_thread": {"value": round(wbytes * n_one / el_one / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "ms_per_step": round(el_one * 1e3 / n_one, 1),
                              "sample": "%d full decode step(s) on 1 thread, %.1f s" % (n_one, el_one)}}


def run_reference(args, rank, world):
    """Reference arm: the f64 C oracle on the host, one full decode step of
    the same workload per timed step (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    import q4_workloads as wl
    oracle.build()
    cfg = wl.cfg4(layers=args.layers)
    wbytes = wl.decode_step_weight_bytes(layers=args.layers)
    for _ in range(args.warmup):
        oracle.decode_step(cfg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_step(cfg)
    el = time.perf_counter() - t0
    value = wbytes * args.steps / el / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded PCG64, same workload as the GPU arm)",
        "config": workload_config(args, wbytes, l2_bytes(), world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "one full decode step per timed step in the f64 C oracle, 1 thread "
                                   "(this arm is single-threaded; the GPU arm's cpu_baseline also reports all cores)",
                         "cpu_model": cpu_model(), "nproc": os.cpu_count() or 1},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.gemv:
        line = run_one_gemv(args) if rank == 0 else None
    elif args.gemm:
        line = run_one_gemm(args) if rank == 0 else None
    elif args.attn:
        line = run_one_attn(args) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
