"""Benchmark of the sink-attention hot path on B300.

Headline (the `value` of the JSON line): sliding-window sink-attention prefill,
bf16, B=1, T=32768, Hq=64, Hkv=8, D=128, W=128, in TFLOP/s counting unmasked
work only (4*D*Hq per visible (query, key) pair).  One step = one prefill call
over that batch.  The same line carries `parts`: the global-attention prefill
on the same shapes (TFLOP/s) and the MTP verify configurations (KV GB/s and
calls/s): 64 requests x 4 tokens with contexts ~ U[4096, 65536] against the
paged GA cache and the 131-slot SWA ring (39 SWA layers back to back), and
8 requests at context 262144 with q_len in {1, 4}.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torchrun as independent replicas (weak scaling, no data-path
collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sink-attn prefill TFLOP/s and MTP-verify KV GB/s, % of B300 roofline"
B, T, HQ, HKV, D, W = 1, 32768, 64, 8, 128, 128
QMAX, PAGE, RING = 4, 64, W + 4 - 1
SWA_LAYERS = 39   # SWA layers of the 48-layer model (39 SWA + 9 GA)


# ------------------------------------------------------------ workload math
def visible_pairs(T_: int, window: int | None) -> int:
    """Number of (query, key) pairs with 0 <= j <= i and (GA or j > i - W)."""
    if window is None or window >= T_:
        return T_ * (T_ + 1) // 2
    return window * T_ - window * (window - 1) // 2


def prefill_flop(T_: int, window: int | None) -> float:
    return 4.0 * D * HQ * visible_pairs(T_, window) * B


def prefill_min_bytes() -> float:
    return 2.0 * (2 * B * T * HQ * D + 2 * B * T * HKV * D)   # Q, O, K, V once each (bf16)


def verify_kv_bytes(ctx: np.ndarray) -> float:
    """K+V bytes of the visible cache, read once per (request, kv head)."""
    return float(np.sum(ctx.astype(np.float64))) * HKV * D * 2 * 2


# ------------------------------------------------------------ host helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def source_sha(rel: str) -> str:
    """Hash of a kernel file together with every header of the library, so
    that recorded counters go stale whenever the compiled kernel could change."""
    import glob
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "global_attention_sinks_swa_b300", "csrc")
    for path in [os.path.join(ROOT, rel)] + sorted(glob.glob(os.path.join(csrc, "*.cuh")) +
                                                   glob.glob(os.path.join(csrc, "*.h"))):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_file: str, name: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(name)
        if rec and rec.get("source_sha") == source_sha(kernel_file):
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class CtypesNvml:
    """The few read-only NVML queries the clock sampler needs, called through
    ctypes on the driver's libnvidia-ml (for hosts without the `pynvml`
    module).  Same names and constants as pynvml's; `lib` may be any object
    with the NVML C entry points (tests pass a fake)."""

    NVML_CLOCK_SM = 1
    # clock event reason bits of the NVML API
    nvmlClocksEventReasonSwPowerCap = 0x4
    nvmlClocksEventReasonHwSlowdown = 0x8
    nvmlClocksEventReasonSwThermalSlowdown = 0x20
    nvmlClocksEventReasonHwThermalSlowdown = 0x40

    def __init__(self, lib=None):
        import ctypes
        self._c = ctypes
        self._lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    def nvmlInit(self):
        self._ok(self._lib.nvmlInit_v2(), "nvmlInit_v2")

    def nvmlDeviceGetHandleByIndex(self, index):
        h = self._c.c_void_p()
        self._ok(self._lib.nvmlDeviceGetHandleByIndex_v2(self._c.c_uint(index), self._c.byref(h)),
                 "nvmlDeviceGetHandleByIndex_v2")
        return h

    def _clock(self, fn, handle, kind):
        v = self._c.c_uint()
        self._ok(getattr(self._lib, fn)(handle, self._c.c_int(kind), self._c.byref(v)), fn)
        return v.value

    def nvmlDeviceGetClockInfo(self, handle, kind):
        return self._clock("nvmlDeviceGetClockInfo", handle, kind)

    def nvmlDeviceGetMaxClockInfo(self, handle, kind):
        return self._clock("nvmlDeviceGetMaxClockInfo", handle, kind)

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle):
        v = self._c.c_ulonglong()
        fn = getattr(self._lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ok(fn(handle, self._c.byref(v)), "nvmlDeviceGetCurrentClocksEventReasons")
        return v.value


class ClockSampler:
    """SM clock and throttle reasons sampled during a timed region (read-only
    queries).  NVML is polled every ~2 ms in a thread, through the `pynvml`
    module or, without it, through ctypes on the driver's NVML library;
    failing both, `nvidia-smi -lms 20` runs for the region and the sampler
    waits for its first line before the region starts."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    NVML_REASONS = ("nvmlClocksEventReasonHwSlowdown", "nvmlClocksEventReasonHwThermalSlowdown",
                    "nvmlClocksEventReasonSwThermalSlowdown", "nvmlClocksEventReasonSwPowerCap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []      # (sm_mhz, set of active reason names)
        self.sm_max = None
        self.source = "unavailable"
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    # -- NVML
    def _nvml_poll(self):
        p = self._nvml
        while not self._stop.is_set():
            self._nvml_once()
            time.sleep(0.002)

    def _nvml_once(self):
        p = self._nvml
        try:
            mhz = float(p.nvmlDeviceGetClockInfo(self._h, p.NVML_CLOCK_SM))
            mask = int(p.nvmlDeviceGetCurrentClocksEventReasons(self._h))
        except Exception:  # noqa: BLE001
            return
        self.samples.append((mhz, {n for n, a in zip(self.NAMES, self.NVML_REASONS)
                                   if mask & getattr(p, a, 0)}))

    # -- nvidia-smi
    def _smi_read(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                mhz, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.sm_max = mx
            self.samples.append((mhz, {n for n, v in zip(self.NAMES, parts[2:6])
                                       if v.lower() == "active"}))
            self._first.set()

    def _start_nvml(self, nvml, source):
        nvml.nvmlInit()
        self._nvml = nvml
        self._h = nvml.nvmlDeviceGetHandleByIndex(self.gpu)
        self.sm_max = float(nvml.nvmlDeviceGetMaxClockInfo(self._h, nvml.NVML_CLOCK_SM))
        self.source = source
        self._thread = threading.Thread(target=self._nvml_poll, daemon=True)
        self._thread.start()

    def __enter__(self):
        notes = []
        for source in ("nvml", "nvml-ctypes"):
            try:
                if source == "nvml":
                    import pynvml as nvml
                else:
                    nvml = CtypesNvml()
                self._start_nvml(nvml, source)
                return self
            except Exception as e:  # noqa: BLE001
                notes.append(f"{source}: {type(e).__name__}: {e}")
        self.error = "; ".join(notes)
        try:
            import subprocess
            self._first = threading.Event()
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._smi_read, daemon=True)
            self._thread.start()
            self._first.wait(timeout=3.0)
            self.source = "nvidia-smi"
        except Exception as e:  # noqa: BLE001
            self.error = (self.error or "") + f"; nvidia-smi: {type(e).__name__}: {e}"
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            time.sleep(0.03)   # one more nvidia-smi line after the region
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self.source.startswith("nvml") and not self.samples:
            self._nvml_once()
        return False

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": [], "samples": len(self.samples),
               "source": self.source}
        if self.samples:
            out["sm_mhz"] = statistics.median(m for m, _ in self.samples)
            out["reasons"] = sorted(set().union(*(r for _, r in self.samples)))
        if self.error:
            out["note"] = self.error
        return out


# ----------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (the timing rule); identity for one process."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ GPU timing
class _NoSampler:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def time_region(fn, steps: int, world: int, stream, sampler=None):
    """CUDA-event time of `steps` calls of fn on `stream`, barrier + sync on
    both sides; `sampler` (a ClockSampler) runs only around the region."""
    import torch
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with (sampler or _NoSampler()):
        start.record(stream)
        for i in range(steps):
            fn(i)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(stop) / steps


def bench_prefill(A, synth, kind: str, steps: int, warmup: int, world: int, stream, seed: int,
                  sampler=None):
    import torch
    sets = []
    for s in range(2):   # two rotating input sets; each set (1.2 GB) exceeds L2
        q, k, v, sink = synth.prefill_inputs(B, T, HQ, HKV, D, seed + s, device="cuda")
        sets.append((q, k, v, sink, torch.empty_like(q)))
    window = W if kind == "swa" else None

    def step(i):
        q, k, v, sink, o = sets[i % 2]
        if kind == "swa":
            A.attn_swa_sink_prefill(q, k, v, sink, window=W, out=o, stream=stream)
        else:
            A.attn_ga_sink_prefill(q, k, v, sink, out=o, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        ms = time_region(step, steps, world, stream, sampler)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError(f"{kind} prefill reported a device error")
    return ms, prefill_flop(T, window)


PACKED_SEQS, PACKED_LO, PACKED_HI = 16, 256, 16384


def bench_prefill_packed(A, synth, steps: int, warmup: int, world: int, stream, seed: int):
    """SWA prefill of a packed serving batch: 16 prompts with log-uniform
    lengths in [256, 16384] (seeded), two rotating input sets larger than L2.
    Returns ms per call, unmasked FLOP and the Q+K+V+O bytes of one call."""
    import torch
    lens = synth.packed_lengths(PACKED_SEQS, PACKED_LO, PACKED_HI, 1006)
    sets = []
    for s in range(2):
        q, k, v, sink, cu = synth.packed_inputs(lens, HQ, HKV, D, seed + s, device="cuda")
        sets.append((q, k, v, sink, torch.from_numpy(cu).cuda(), torch.empty_like(q)))
    mx = int(lens.max())

    def step(i):
        q, k, v, sink, cu, o = sets[i % 2]
        A.attn_swa_sink_prefill_varlen(q, k, v, cu, sink, window=W, max_seqlen=mx, out=o,
                                       stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        ms = time_region(step, steps, world, stream)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError("packed prefill reported a device error")
    flop = sum(4.0 * D * HQ * visible_pairs(int(n), W) for n in lens)
    nbytes = 2.0 * float(lens.sum()) * (2 * HQ * D + 2 * HKV * D)
    return ms, flop, nbytes, lens


def bench_backward(A, synth, steps: int, warmup: int, world: int, stream, seed: int, T_=T,
                   window=W):
    """Backward (dq, dk, dv, dsink), by default the SWA layer at the headline
    sizes (window 0: global attention); FLOP = the five products over visible
    pairs (S, dP, dV, dK, dQ): 10*D*Hq per pair."""
    import torch
    q, k, v, sink = synth.prefill_inputs(B, T_, HQ, HKV, D, seed, device="cuda")
    dout = synth.normal((B, T_, HQ, D), seed + 1, device="cuda")
    lse = torch.empty(B, HQ, T_, device="cuda")
    if window:
        o = A.attn_swa_sink_prefill(q, k, v, sink, window=window, lse=lse, stream=stream)
    else:
        o = A.attn_ga_sink_prefill(q, k, v, sink, lse=lse, stream=stream)
    ws = torch.empty(A._lib.attn_sink_prefill_backward_workspace(B, T_, HQ, D), dtype=torch.uint8,
                     device="cuda")

    def step(_):
        A.attn_sink_prefill_backward(q, k, v, o, lse, dout, sink, window=window, workspace=ws,
                                     stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        ms = time_region(step, steps, world, stream)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError("backward reported a device error")
    return ms, 10.0 * D * HQ * visible_pairs(T_, window or None) * B


def bench_prefill_e2e(A, synth, steps: int, warmup: int, world: int, stream, seed: int):
    """Same metric through the public call with host buffers: every step
    copies its inputs (q, k, v, sink) from pinned host memory and its output
    o back.  Steps are double-buffered over three streams, so the upload of
    step i+1 and the download of step i overlap on the full-duplex link, as a
    serving loop would run them; the time runs from the first upload to the
    last download."""
    import torch
    q, k, v, sink = synth.prefill_inputs(B, T, HQ, HKV, D, seed, device="cuda")
    hq, hk, hv, hs = (x.cpu().pin_memory() for x in (q, k, v, sink))
    del q, k, v, sink
    ho = [torch.empty_like(hq).pin_memory() for _ in range(2)]
    dev = [[torch.empty_like(x, device="cuda") for x in (hq, hk, hv, hs, hq)] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        bi = i & 1
        dq, dk, dv, ds, do = dev[bi]
        if i >= 2:
            s_in.wait_event(comp_done[bi])      # step i-2's kernel has read these inputs
        with torch.cuda.stream(s_in):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
            in_done[bi].record(s_in)
        stream.wait_event(in_done[bi])
        if i >= 2:
            stream.wait_event(out_done[bi])     # step i-2's output has been read back
        A.attn_swa_sink_prefill(dq, dk, dv, ds, window=W, out=do, stream=stream)
        comp_done[bi].record(stream)
        s_out.wait_event(comp_done[bi])
        with torch.cuda.stream(s_out):
            ho[bi].copy_(do, non_blocking=True)
            out_done[bi].record(s_out)

    def run(n, first):
        for i in range(n):
            step(first + i)

    run(max(2, warmup), 0)
    torch.cuda.synchronize()
    barrier(world)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    run(steps, 2 * max(2, warmup))   # even offset: buffer parity continues
    stop.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(stop) / steps
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hs))
    d2h = ho[0].numel() * ho[0].element_size()
    return ms, h2d, d2h


def _paged_problem(ctx, q_lens, seed, device="cuda", fp8=False):
    import torch
    import synth
    npages = (ctx + PAGE - 1) // PAGE
    nb = len(ctx)
    num_pages = int(npages.sum())
    perm = synth.page_permutation(num_pages, seed)
    pt = np.zeros((nb, int(npages.max())), np.int32)
    o = 0
    for b in range(nb):
        pt[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
    if fp8:   # E4M3 codes and per-kv-head scales
        kp = synth.e4m3_codes((num_pages, HKV, PAGE, D), seed + 1, device=device)
        vp = synth.e4m3_codes((num_pages, HKV, PAGE, D), seed + 2, device=device)
    else:
        kp = synth.normal((num_pages, HKV, PAGE, D), seed + 1, device=device)
        vp = synth.normal((num_pages, HKV, PAGE, D), seed + 2, device=device)
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), HQ, D), seed + 3, device=device)
    sink = synth.sink_logits(HQ, seed + 4, device=device)
    return dict(kp=kp, vp=vp, pt=torch.from_numpy(pt).to(device), ctx=torch.from_numpy(ctx).to(device),
                cu_q=torch.from_numpy(cu_q).to(device), q=q, sink=sink, max_ctx=int(ctx.max()),
                ks=synth.kv_scales(HKV, seed + 5, device=device),
                vs=synth.kv_scales(HKV, seed + 6, device=device))


def bench_verify_ga(A, ctx, q_lens, steps, warmup, world, stream, seed, fp8=False):
    """GA paged verify; fp8=True reads 8-bit (E4M3) pages: half the bytes."""
    import torch
    P = _paged_problem(ctx, q_lens, seed, fp8=fp8)
    ws_bytes = A.attn_ga_sink_verify_workspace(len(ctx), HQ, HKV, D, QMAX, P["max_ctx"])
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(P["q"])

    def step(_):
        if fp8:
            A.attn_ga_sink_verify_fp8(P["q"], P["cu_q"], P["kp"], P["vp"], P["pt"], P["ctx"],
                                      P["sink"], P["ks"], P["vs"], max_ctx=P["max_ctx"], q_max=QMAX,
                                      out=out, workspace=ws, stream=stream)
        else:
            A.attn_ga_sink_verify(P["q"], P["cu_q"], P["kp"], P["vp"], P["pt"], P["ctx"], P["sink"],
                                  max_ctx=P["max_ctx"], q_max=QMAX, out=out, workspace=ws,
                                  stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
        ms = time_region(step, steps, world, stream)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError("GA verify reported a device error")
    return ms, verify_kv_bytes(ctx) / (2 if fp8 else 1)


def bench_verify_swa(A, nreq, steps, warmup, world, stream, seed):
    """39 SWA layers back to back (distinct rings), replayed as one CUDA graph."""
    import torch
    import synth
    rings = [(synth.normal((nreq, HKV, RING, D), seed + 2 * i, device="cuda"),
              synth.normal((nreq, HKV, RING, D), seed + 2 * i + 1, device="cuda"))
             for i in range(SWA_LAYERS)]
    ctx = synth.context_lengths(nreq, 4096, 65536, seed + 99)
    q_lens = np.full(nreq, QMAX, np.int32)
    cu_q = torch.from_numpy(synth.cu_seqlens(q_lens)).cuda()
    sl = torch.from_numpy(ctx).cuda()
    q = synth.normal((nreq * QMAX, HQ, D), seed + 100, device="cuda")
    sink = synth.sink_logits(HQ, seed + 101, device="cuda")
    outs = [torch.empty_like(q) for _ in range(SWA_LAYERS)]

    def layers():
        for i, (rk, rv) in enumerate(rings):
            A.attn_swa_sink_verify(q, cu_q, rk, rv, sl, sink, window=W, q_max=QMAX, out=outs[i],
                                   stream=stream)

    with torch.cuda.stream(stream):
        layers()   # warm (tensor-map encode, function attributes)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layers()
        for _ in range(warmup):
            graph.replay()
        ms = time_region(lambda _: graph.replay(), steps, world, stream)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError("SWA verify reported a device error")
    kv = float(nreq) * RING * HKV * D * 2 * 2 * SWA_LAYERS
    return ms, kv


# ------------------------------------------------- one MTP step, model order
def model_step_problem(A, nreq, lo, hi, seed, q_lens=None, ctx=None):
    """The attention of one MTP verify step over the 48-layer hybrid stack in
    model order (synth.hybrid_layer_kinds: GA at layers 0, 5, 11, .., 47):
    every layer owns its cache (a 131-slot ring per SWA layer, a paged pool
    per GA layer), its queries, its new keys/values and its sink logits.
    nreq requests with contexts ~ U[lo, hi] (seeded), 4 new tokens each
    unless q_lens is given (contexts too, when ctx is given)."""
    import torch
    import synth
    kinds = synth.hybrid_layer_kinds()
    ctx = (synth.context_lengths(nreq, lo, hi, seed) if ctx is None
           else np.asarray(ctx, np.int32))
    q_lens = np.full(nreq, QMAX, np.int32) if q_lens is None else np.asarray(q_lens, np.int32)
    cu_q = synth.cu_seqlens(q_lens)
    nq = int(cu_q[-1])
    npages = (ctx + PAGE - 1) // PAGE
    num_pages, max_pages = int(npages.sum()), int(npages.max())
    layers = []
    for li, kind in enumerate(kinds):
        base = seed + 1000 * (li + 1)
        d = {"kind": kind,
             "q": synth.normal((nq, HQ, D), base, device="cuda"),
             "k_new": synth.normal((nq, HKV, D), base + 1, device="cuda"),
             "v_new": synth.normal((nq, HKV, D), base + 2, device="cuda"),
             "sink": synth.sink_logits(HQ, base + 3, device="cuda"),
             "out": torch.empty(nq, HQ, D, dtype=torch.bfloat16, device="cuda")}
        if kind == "swa":
            d["rk"] = synth.normal((nreq, HKV, RING, D), base + 4, device="cuda")
            d["rv"] = synth.normal((nreq, HKV, RING, D), base + 5, device="cuda")
        else:
            perm = synth.page_permutation(num_pages, base + 6)
            pt = np.zeros((nreq, max_pages), np.int32)
            o = 0
            for b in range(nreq):
                pt[b, :npages[b]] = perm[o:o + npages[b]]
                o += npages[b]
            d["pt"] = torch.from_numpy(pt).cuda()
            d["kp"] = synth.normal((num_pages, HKV, PAGE, D), base + 7, device="cuda")
            d["vp"] = synth.normal((num_pages, HKV, PAGE, D), base + 8, device="cuda")
        layers.append(d)
    max_ctx = int(ctx.max())
    ws_bytes = A.attn_ga_sink_verify_workspace(nreq, HQ, HKV, D, QMAX, max_ctx)
    return {"layers": layers, "ctx": ctx, "q_lens": q_lens, "cu_q_np": cu_q,
            "cu_q": torch.from_numpy(cu_q).cuda(), "seq_lens": torch.from_numpy(ctx).cuda(),
            "max_ctx": max_ctx,
            "ws": torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")}


def model_step(A, P, stream):
    """Enqueue the step: for each layer in order, append its new keys/values
    to its cache, then verify.  Every kernel is launched as a programmatic
    dependent of the one before it, so a layer's verify can set up and
    prefetch its cache into L2 while the previous kernel finishes."""
    cu, sl = P["cu_q"], P["seq_lens"]
    for d in P["layers"]:
        if d["kind"] == "swa":
            A.attn_swa_ring_append(d["k_new"], d["v_new"], cu, sl, d["rk"], d["rv"], q_max=QMAX,
                                   stream=stream)
            A.attn_swa_sink_verify(d["q"], cu, d["rk"], d["rv"], sl, d["sink"], window=W,
                                   q_max=QMAX, out=d["out"], stream=stream)
        else:
            A.attn_ga_paged_append(d["k_new"], d["v_new"], cu, sl, d["kp"], d["vp"], d["pt"],
                                   q_max=QMAX, stream=stream)
            A.attn_ga_sink_verify(d["q"], cu, d["kp"], d["vp"], d["pt"], sl, d["sink"],
                                  max_ctx=P["max_ctx"], q_max=QMAX, out=d["out"],
                                  workspace=P["ws"], stream=stream)


def model_step_kv_bytes(P) -> float:
    """K+V bytes the step's verifies read: the ring of every SWA layer and the
    visible pages of every GA layer, once per (request, kv head)."""
    n_swa = sum(d["kind"] == "swa" for d in P["layers"])
    n_ga = len(P["layers"]) - n_swa
    return n_swa * float(len(P["ctx"])) * RING * HKV * D * 2 * 2 + n_ga * verify_kv_bytes(P["ctx"])


def bench_verify_step(A, nreq, steps, warmup, world, stream, seed):
    """One MTP step over the 48 layers (39 SWA ring + 9 GA paged verifies, each
    after its cache append) replayed as one CUDA graph."""
    import torch
    P = model_step_problem(A, nreq, 4096, 65536, seed)
    with torch.cuda.stream(stream):
        model_step(A, P, stream)   # warm (tensor-map encode, function attributes)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            model_step(A, P, stream)
        for _ in range(warmup):
            graph.replay()
        ms = time_region(lambda _: graph.replay(), steps, world, stream)
    if A.attn_check_device_error(stream) != 0:
        raise RuntimeError("model step reported a device error")
    kv = model_step_kv_bytes(P)
    del P, graph
    torch.cuda.empty_cache()
    return ms, kv


# --------------------------------------------------------------- CPU baseline
def cpu_baseline(seconds_target: float = 15.0):
    """The fp64 oracle on a bounded sample of the headline workload (rows of
    the SWA prefill), timed on the host cores; value in unmasked TFLOP/s."""
    import oracle
    import synth
    import torch
    cores = len(os.sched_getaffinity(0))
    q, k, v, sink = synth.prefill_inputs(B, T, HQ, HKV, D, 2024, dtype=torch.float32)
    rng = np.random.default_rng(0)
    n = 4096
    total_rows, total_flop, total_s = 0, 0.0, 0.0
    while total_s < seconds_target and total_rows < B * T * HQ:
        rows = np.stack([np.zeros(n, np.int64), rng.integers(W, T, n), rng.integers(0, HQ, n)], 1)
        t0 = time.perf_counter()
        oracle.prefill_rows(q, k, v, sink, rows, W)
        total_s += time.perf_counter() - t0
        total_rows += n
        total_flop += 4.0 * D * W * n   # rows past the first W see exactly W keys
        n *= 2
    return {"value": total_flop / total_s / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{total_rows} random rows (i >= W) of the SWA prefill, {total_s:.1f} s; "
                      f"fp64 C loops, OpenMP over rows"}


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-parts", action="store_true", help="headline only")
    ap.add_argument("--profile", default="",
                    help="comma list of swa,ga,verify_ga,verify_ga_fp8,verify_swa,verify_step,backward,ga_backward: run only these kernels "
                         "(warmup + steps), no JSON line; for ncu captures")
    args = ap.parse_args()
    world, rank, local = dist_env()
    warmup = max(3, args.warmup)

    if args.impl == "reference":
        return run_reference(args, world, rank, warmup)

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    import global_attention_sinks_swa_b300 as A
    import synth
    stream = torch.cuda.Stream()
    hbm, tf_burst, tf_sus, peak_src = load_peaks()

    if args.profile:
        return run_profile(A, synth, args, warmup, stream)
    clocks = ClockSampler(local)
    ms, flop = bench_prefill(A, synth, "swa", args.steps, warmup, world, stream, 1002 + 10 * rank,
                             clocks)
    ms_max = reduce_max(ms, world, torch.device("cuda", local))
    value = world * flop / (ms_max * 1e-3) / 1e12
    achieved = prefill_min_bytes() / (ms * 1e-3) / 1e9

    parts = {}
    launches = args.steps
    if not args.no_parts:
        steps_p = max(3, args.steps // 2)
        ms_ga, flop_ga = bench_prefill(A, synth, "ga", steps_p, warmup, world, stream, 1003 + 10 * rank)
        parts["ga_prefill"] = {"config": "B=1 T=32768 Hq=64 Hkv=8 D=128 full causal bf16",
                               "value": flop_ga / (ms_ga * 1e-3) / 1e12, "unit": "TFLOP/s",
                               "ms": ms_ga, "roofline": {"bound": "tensor",
                                                         "peak": tf_burst, "unit": "TFLOP/s",
                                                         "frac": flop_ga / (ms_ga * 1e-3) / 1e12 / tf_burst,
                                                         "frac_sustained": flop_ga / (ms_ga * 1e-3) / 1e12 / tf_sus}}
        ms_pk, flop_pk, bytes_pk, lens_pk = bench_prefill_packed(A, synth, steps_p, warmup, world,
                                                                 stream, 1007 + 10 * rank)
        parts["swa_prefill_packed_16seq"] = {
            "config": f"{PACKED_SEQS} packed prompts, lengths log-uniform in "
                      f"[{PACKED_LO}, {PACKED_HI}] (total {int(lens_pk.sum())} tokens), "
                      "Hq=64 Hkv=8 D=128 W=128 bf16, cu_seqlens",
            "value": flop_pk / (ms_pk * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": ms_pk,
            "roofline": {"bound": "hbm", "achieved": bytes_pk / (ms_pk * 1e-3) / 1e9,
                         "peak": hbm, "unit": "GB/s",
                         "frac": bytes_pk / (ms_pk * 1e-3) / 1e9 / hbm}}
        ms_bw, flop_bw = bench_backward(A, synth, max(3, steps_p // 2), warmup, world, stream,
                                        1008 + 10 * rank)
        parts["swa_backward"] = {
            "config": "B=1 T=32768 Hq=64 Hkv=8 D=128 W=128 bf16: dq, dk, dv, dsink",
            "value": flop_bw / (ms_bw * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": ms_bw,
            "flop": "10*D*Hq per visible pair (five products)",
            "roofline": {"bound": "tensor", "peak": tf_burst, "unit": "TFLOP/s",
                         "frac": flop_bw / (ms_bw * 1e-3) / 1e12 / tf_burst}}
        ms_gb, flop_gb = bench_backward(A, synth, 3, warmup, world, stream, 1009 + 10 * rank,
                                        window=0)
        parts["ga_backward"] = {
            "config": "B=1 T=32768 Hq=64 Hkv=8 D=128 full causal bf16: dq, dk, dv, dsink",
            "value": flop_gb / (ms_gb * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": ms_gb,
            "flop": "10*D*Hq per visible pair (five products)",
            "roofline": {"bound": "tensor", "peak": tf_burst, "unit": "TFLOP/s",
                         "frac": flop_gb / (ms_gb * 1e-3) / 1e12 / tf_burst,
                         "frac_sustained": flop_gb / (ms_gb * 1e-3) / 1e12 / tf_sus}}
        ctx4 = synth.context_lengths(64, 4096, 65536, 1004)
        ms4, kv4 = bench_verify_ga(A, ctx4, np.full(64, QMAX, np.int32), args.steps, warmup, world,
                                   stream, 1004 + 10 * rank)
        parts["verify_ga_64req"] = {"config": "64 req x q4, ctx~U[4096,65536], page 64",
                                    "value": kv4 / (ms4 * 1e-3) / 1e9, "unit": "GB/s",
                                    "calls_per_s": 1e3 / ms4, "ms": ms4,
                                    "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                                                 "frac": kv4 / (ms4 * 1e-3) / 1e9 / hbm}}
        ms8, kv8 = bench_verify_ga(A, ctx4, np.full(64, QMAX, np.int32), args.steps, warmup, world,
                                   stream, 1004 + 10 * rank, fp8=True)
        parts["verify_ga_fp8_64req"] = {"config": "64 req x q4, ctx~U[4096,65536], page 64, E4M3 pages",
                                        "value": kv8 / (ms8 * 1e-3) / 1e9, "unit": "GB/s",
                                        "calls_per_s": 1e3 / ms8, "ms": ms8,
                                        "speedup_vs_bf16_pages": ms4 / ms8,
                                        "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                                                     "frac": kv8 / (ms8 * 1e-3) / 1e9 / hbm}}
        ms_s, kv_s = bench_verify_swa(A, 64, args.steps, warmup, world, stream, 2004 + 10 * rank)
        parts["verify_swa_64req_39layers"] = {
            "config": "64 req x q4, 131-slot ring, 39 layers in one CUDA graph",
            "value": kv_s / (ms_s * 1e-3) / 1e9, "unit": "GB/s", "calls_per_s": SWA_LAYERS * 1e3 / ms_s,
            "ms_per_39_layers": ms_s,
            "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                         "frac": kv_s / (ms_s * 1e-3) / 1e9 / hbm}}
        torch.cuda.empty_cache()
        ms_st, kv_st = bench_verify_step(A, 64, max(3, args.steps // 5), warmup, world, stream,
                                         3004 + 10 * rank)
        parts["verify_step_48layers"] = {
            "config": "one MTP step in model order: 48 layers (GA at 0,5,11,..,47; 39 SWA ring + "
                      "9 GA paged), append + verify per layer, 64 req x q4, ctx~U[4096,65536], "
                      "distinct caches, one CUDA graph, programmatic dependent launches",
            "value": kv_st / (ms_st * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_st,
            "layers_per_s": 48 * 1e3 / ms_st, "kv_bytes_per_step": kv_st,
            "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                         "frac": kv_st / (ms_st * 1e-3) / 1e9 / hbm}}
        for ql, name in ((4, "verify_ga_8x262144_q4"), (1, "verify_ga_8x262144_q1")):
            ctx5 = np.full(8, 262144, np.int32)
            ms5, kv5 = bench_verify_ga(A, ctx5, np.full(8, ql, np.int32), args.steps, warmup, world,
                                       stream, 1005 + ql + 10 * rank)
            parts[name] = {"config": f"8 req x q{ql}, ctx 262144, page 64",
                           "value": kv5 / (ms5 * 1e-3) / 1e9, "unit": "GB/s",
                           "calls_per_s": 1e3 / ms5, "ms": ms5,
                           "roofline": {"bound": "hbm", "peak": hbm, "unit": "GB/s",
                                        "frac": kv5 / (ms5 * 1e-3) / 1e9 / hbm}}
        torch.cuda.empty_cache()

    e2e_ms, h2d, d2h = bench_prefill_e2e(A, synth, max(3, args.steps // 4), warmup, world, stream,
                                         1002 + 10 * rank)
    e2e_ms = reduce_max(e2e_ms, world, torch.device("cuda", local))

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": warmup,
            "ms_per_step": ms_max,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic: Q,K,V ~ N(0,1) bf16, sink ~ N(0,1) fp32, seeded",
            "config": {"workload": "SWA sink prefill B=1 T=32768 Hq=64 Hkv=8 D=128 W=128",
                       "global_batch": B * world, "seq_len": T, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (1.2 GB per set, 2 rotating sets)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": peak_src,
                         "traffic": ncu_traffic("global_attention_sinks_swa_b300/csrc/prefill_swa.cu",
                                                "prefill_swa_stream_kernel"),
                         "algorithmic_bytes": prefill_min_bytes(),
                         "tensor_frac": flop / (ms * 1e-3) / 1e12 / tf_burst},
            "clocks": clocks.summary(),
            "e2e": {"value": world * flop / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "overlap": "steps double-buffered on three streams: the upload of step i+1 "
                               "overlaps the download of step i; each step moves its own data"},
            "gpu_launches": launches,
            "parts": parts,
        }
        line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile(A, synth, args, warmup, stream):
    """Only the named kernels, for profiler captures (sizes: the headline and
    GA prefill at full size, 1.2 GB each; GA verify on 16 requests ~ 2.3 GB,
    half that with 8-bit pages)."""
    for name in args.profile.split(","):
        if name in ("swa", "ga"):
            bench_prefill(A, synth, name, args.steps, warmup, 1, stream, 1002)
        elif name == "backward":   # a quarter of the headline length: a small capture
            bench_backward(A, synth, args.steps, warmup, 1, stream, 1008, T_=T // 4)
        elif name == "ga_backward":
            bench_backward(A, synth, args.steps, warmup, 1, stream, 1009, T_=T // 4, window=0)
        elif name in ("verify_ga", "verify_ga_fp8"):
            ctx = synth.context_lengths(16, 4096, 65536, 1004)
            bench_verify_ga(A, ctx, np.full(16, QMAX, np.int32), args.steps, warmup, 1, stream, 1004,
                            fp8=name.endswith("fp8"))
        elif name == "verify_swa":
            bench_verify_swa(A, 64, args.steps, warmup, 1, stream, 2004)
        elif name == "verify_step":
            bench_verify_step(A, 64, args.steps, warmup, 1, stream, 3004)
        else:
            raise SystemExit(f"unknown profile target {name}")
    print(json.dumps({"profile": args.profile, "ok": True}), flush=True)


def run_reference(args, world, rank, warmup):
    """The oracle as it stands on the host cores, on a bounded sample of the
    headline workload per step."""
    if rank != 0:
        return
    import oracle
    import synth
    import torch
    q, k, v, sink = synth.prefill_inputs(B, T, HQ, HKV, D, 2024, dtype=torch.float32)
    rng = np.random.default_rng(0)
    n = 2048
    def step():
        rows = np.stack([np.zeros(n, np.int64), rng.integers(W, T, n), rng.integers(0, HQ, n)], 1)
        oracle.prefill_rows(q, k, v, sink, rows, W)
    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = 4.0 * D * W * n / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "SWA sink prefill B=1 T=32768 Hq=64 Hkv=8 D=128 W=128",
                   "sample": f"{n} random rows per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} random rows (i >= W) of the SWA prefill per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
