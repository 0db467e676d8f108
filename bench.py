"""Benchmark of the attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  The headline workload is the largest single-GPU
configuration, the long ragged causal prefill (B=1, H=32, N=16381, d=128,
causal, bf16): one step is one fa_fwd_ex call over it (one launch of the fused
forward, 2048 blocks of 256 query rows, longest first), timed with CUDA events
on the launching stream; its inputs (402 MB) exceed L2, so nothing is flushed.
``extra`` carries the other workloads of the target (prefill N=2048 d=64 with
L2 flushed between steps, causal N=8192 d=128 with x8 key spikes, split-KV
decode L=32768) and of the library's further paths (backward and FP8 forward on
the causal workload, the decode over a paged cache, the causal workload in four
key shards merged by the combine), each with its roofline fraction.  ``e2e``
repeats the headline through the C ABI with pinned host buffers and the
host<->device copies inside the timed region.  ``cpu_baseline`` is the fp64
oracle timed on the host cores (one thread and all of them) over a bounded
sample of the headline's rows, with a labelled extrapolation to the whole
workload.  ``--impl reference`` times that oracle as the reference arm (there
is no runnable reference implementation).

Multi-GPU: the work does not shard across GPUs in this design; under torchrun
every rank runs an independent replica ("scaling": "weak") and the slowest
rank's time is reported.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "ragged"
EXTRA = ("prefill", "causal", "decode")
E2E_CHUNKS = 8  # host<->device pipeline stages of the e2e step
L2_FLUSH_BYTES = 256 << 20
METRIC = "attention fwd TFLOPS (bf16, causal/non-causal) and decode GB/s vs GB300 roofline"


# ----------------------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from ncu captures summarised
# under profiles/, keyed by kernel and workload, valid only while the kernel sources are unchanged.
_FWD = "bf5065744ca54e1b253c2dc98ec99b932f320522aa698fdb3178cb9e91562e04"
_BWD = "3100608144e05a1479f6d4eec6fe754549bc5e11c799049f40b136280dca76b6"
_DEC = "238a9c1b2ffecb15b22cb24a1544220a197fcbdb2c867899597a0c8e4fa65d64"
NCU_TRAFFIC = {
    ("fwd_kernel", "ragged"): {"sources": {"fa_fwd.cu": _FWD}, "bytes": 559.377e6},
    ("fwd_kernel", "causal"): {"sources": {"fa_fwd.cu": _FWD}, "bytes": 263.888e6},
    ("fwd_kernel_fp8", "causal"): {"sources": {"fa_fwd.cu": _FWD}, "bytes": 136.481e6},
    ("fwd_persist_kernel", "prefill"): {"sources": {"fa_fwd.cu": _FWD}, "bytes": 50.483e6},
    # backward: the dominant kernel (dK/dV) on the causal workload
    ("bwd_dkdv_kernel", "causal"): {"sources": {"fa_bwd.cu": _BWD}, "bytes": 372.482e6},
    # the four-shard step: four forward launches over the key shards and the combine, summed
    ("causal_sharded4", "causal"): {"sources": {"fa_fwd.cu": _FWD, "fa_decode.cu": _DEC}, "bytes": 1108.970e6},
    # decode: captured on the B4 slice (decode_small) and scaled by 16 to B64 (K/V streamed once)
    ("decode_split_kernel", "decode"): {"sources": {"fa_decode.cu": _DEC}, "bytes": 16 * 2151.001e6},
    ("decode_split_kernel_paged", "decode"): {"sources": {"fa_decode.cu": _DEC}, "bytes": 16 * 2150.928e6},
}


def _traffic(kernel: str, workload: str):
    rec = NCU_TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    for src, sha in rec["sources"].items():
        try:
            with open(os.path.join(ROOT, "exact_attention_06_gb300", "csrc", src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None
        except OSError:
            return None
    return rec["bytes"]


def _workload_label(w):
    if w.kind == "decode":
        return f"decode B{w.B} H{w.H} L{w.N} d{w.d}"
    return (f"{w.name} B{w.B} H{w.H} N{w.N} d{w.d} {'causal' if w.causal else 'non-causal'}"
            f"{' x8 key spikes' if w.spike else ''}")


def _headline_config(w, world):
    """The headline's config object, the same for both arms."""
    l2 = "flushed between timed steps (256 MiB write)" if _fits_l2(w) else (
        f"inputs larger than L2 ({3 * w.B * w.H * w.N * w.d * 2 / 1e6:.0f} MB of q, k, v): not flushed")
    return {"workload": _workload_label(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": w.scale, "global_batch": w.B * world, "seq_len": w.N, "parallelism": f"replicas x{world}",
            "l2": l2}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock event reasons)."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        c = self.c
        mhz, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(mhz)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, c.byref(mx))
        self.reasons_fn(self.h, c.byref(rs))
        return float(mhz.value), float(mx.value), [n for b, n in self.REASONS.items() if rs.value & b]


class ClockSampler:
    """SM clock and throttle reasons while a region runs: NVML polled every ~2 ms when the library
    loads (enough samples for a timed region of tens of milliseconds), else nvidia-smi samples."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.device_index = device_index
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.nvml = _Nvml(self.device_index)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.stop_flag = False
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        while not self.stop_flag:
            smp = self.nvml.sample()
            if smp is not None:
                mhz, mx, reasons = smp
                parts = ["", str(mhz), str(mx), ""] + ["" for _ in range(5)]
                for i, name in enumerate(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                          "sw_power_cap")):
                    parts[5 + i] = "Active" if name in reasons else "Not Active"
                self.samples.append((time.time(), parts))
            time.sleep(0.002)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if getattr(self, "nvml", None) is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        inside = [p for t, p in self.samples if self.t_start and self.t_end and self.t_start <= t <= self.t_end]
        window = "timed"
        if len(inside) < 3:
            inside = [p for _, p in self.samples]
            window = "warmup+timed"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for p in inside:
            for name, val in zip(names, p[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window,
                "source": "nvml" if getattr(self, "nvml", None) is not None else "nvidia-smi"}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's time (replicas: every rank runs the same step on its own GPU)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- our arm

def _fits_l2(w):
    """Whether a prefill workload's q, k, v fit in L2 (then L2 is flushed between timed steps)."""
    return w.kind == "prefill" and 3 * w.B * w.H * w.N * w.d * 2 < L2_FLUSH_BYTES


def _fwd_kernel_name(w):
    """The forward kernel fa_fwd_ex launches for a workload (bf16)."""
    return "fwd_persist_kernel" if (not w.causal and w.d == 64) else "fwd_kernel"


def _prefill_step_fn(w, dev, stream):
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    ws = _tail_workspace(w, dev)

    def step():
        fattn.fa_fwd_ex(q, k, v, o, lse, w.scale, w.causal, stream=stream, workspace=ws)
    return step, 1 if ws is None else 2


def _tail_workspace(w, dev):
    """The workspace of the forward's key split for this workload on this device (None: no key
    split planned, one launch; otherwise the forward and the combine of the split blocks)."""
    import torch
    from exact_attention_06_gb300 import fattn
    nbytes = fattn.fa_fwd_workspace_bytes(w.B, w.H, w.N, w.d, w.causal)
    return torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None


def _decode_step_fn(w, dev, stream):
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    o = torch.empty(w.B, w.H, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, dtype=torch.float32, device=dev)
    ws = torch.empty(fattn.fa_decode_workspace_bytes(w.B, w.H, w.N, w.d, 128, 0), dtype=torch.uint8, device=dev)

    def step():
        fattn.fa_decode_splitkv(q, k, v, o, lse, w.scale, ws, 128, 0, stream=stream)
    return step, 2


def _backward_step_fn(w, dev, stream):
    """One backward (D, dK/dV, dQ kernels) over the workload, from a forward done once beforehand."""
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    do = inputs.normal_bf16(q.shape, seed=9, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    fattn.fa_fwd(q, k, v, o, lse, w.scale, w.causal, stream=stream)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fattn.fa_bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)

    def step():
        fattn.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, w.causal, workspace=ws, stream=stream)
    return step, 3


def _paged_decode_step_fn(w, dev, stream, page_size=128):
    """Split-KV decode over a paged cache: the workload's K/V written into pools of 128-key pages
    in a seeded random order, every sequence at full length."""
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    n = -(-w.N // page_size)
    assert w.N == n * page_size
    perm = torch.randperm(w.B * n, generator=torch.Generator().manual_seed(3)).to(dev)
    table = perm.view(w.B, n).to(torch.int32)
    pools = []
    for x in (k, v):
        pool = torch.empty((w.B * n, w.H, page_size, w.d), dtype=torch.bfloat16, device=dev)
        pool[perm] = x.view(w.B, w.H, n, page_size, w.d).permute(0, 2, 1, 3, 4).reshape(w.B * n, w.H, page_size, w.d)
        pools.append(pool)
    del k, v, x
    kp, vp = pools
    lens = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    o = torch.empty(w.B, w.H, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, dtype=torch.float32, device=dev)
    ws = torch.empty(fattn.fa_decode_paged_workspace_bytes(w.B, w.H, w.N, w.d, page_size, n, 0), dtype=torch.uint8,
                     device=dev)

    def step():
        fattn.fa_decode_paged(q, kp, vp, table, lens, o, lse, w.scale, w.N, workspace=ws, stream=stream)
    return step, 2


def _sharded_step_fn(w, dev, stream, shards=4):
    """Sequence-sharded prefill: the keys cut into equal shards, one fa_fwd_partial_ex per shard
    reading its key range from the whole K/V tensors, then fa_combine."""
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    cuts = [w.N * i // shards for i in range(shards + 1)]
    R = w.B * w.H * w.N
    u = torch.empty((R, shards, w.d), dtype=torch.float32, device=dev)
    m = torch.empty((R, shards), dtype=torch.float32, device=dev)
    l = torch.empty((R, shards), dtype=torch.float32, device=dev)
    o = torch.empty((R, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(R, dtype=torch.float32, device=dev)

    side = [torch.cuda.Stream(device=dev) for _ in range(shards)]

    def step():
        # the shards are independent: each on its own stream, joined before the combine
        for s in range(shards):
            side[s].wait_stream(stream)
            fattn.fa_fwd_partial(q, k, v, u, m, l, w.scale, cuts[s], s, w.causal, stream=side[s],
                                 nk=cuts[s + 1] - cuts[s])
        for s in range(shards):
            stream.wait_stream(side[s])
        fattn.fa_combine(u, m, l, o, lse, stream=stream)
    return step, shards + 1


def _fp8_step_fn(w, dev, stream):
    """One FP8 forward (fa_fwd_fp8) over the workload; Q, K, V quantized to E4M3 once beforehand
    (the FP8 path keeps its inputs in HBM as codes plus block scales)."""
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    q, k, v = inputs.workload_inputs(w, seed=0, device=dev)
    nb = (w.N + 127) // 128
    packed = []
    for x in (q, k, v):
        c = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        s = torch.empty(w.B, w.H, nb, dtype=torch.float32, device=dev)
        fattn.fa_quantize_e4m3(x, c, s, stream=stream)
        packed += [c, s]
    stream.synchronize()
    del q, k, v
    (q8, sq, k8, sk, v8, sv) = packed
    o = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)

    def step():
        fattn.fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, w.scale, w.causal, stream=stream)
    return step, 1


def _time_steps(step, steps, warmup, stream, flush=None, sampler=None, dist_sync=None):
    """Per-step CUDA-event times (ms) of exactly `steps` steps after `warmup` untimed ones."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if dist_sync:
        dist_sync()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t_start")
    with torch.cuda.stream(stream):
        for a, b in evs:
            if flush is not None:
                flush()
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t_end")
    if dist_sync:
        dist_sync()
    return [a.elapsed_time(b) for a, b in evs]


def _roofline(kind, work_per_launch, launch_ms, peaks, traffic):
    if kind in ("tensor", "tensor_fp8"):
        achieved = work_per_launch / (launch_ms * 1e-3) / 1e12
        # E4M3 dense rate = the measured bf16 rate x the nominal fp8/bf16 ratio (4.5 / 2.25 PFLOP/s)
        peak = peaks["bf16_tflops"] * (2.0 if kind == "tensor_fp8" else 1.0)
        unit = "TFLOP/s"
    else:
        achieved = work_per_launch / (launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    src = {"tensor": "bf16 burst", "tensor_fp8": "bf16 burst x 2, the nominal fp8/bf16 ratio",
           "hbm": "copy bandwidth"}[kind]
    return {"bound": "tensor" if kind == "tensor_fp8" else kind, "achieved": round(achieved, 2), "peak": peak,
            "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{peaks['source']} ({src})"}


def _e2e_prefill(w, dev, stream, steps, warmup):
    """Headline metric through the C ABI from pinned host buffers (copies timed).

    The B*H heads are processed in E2E_CHUNKS chunks of consecutive heads on three streams: the
    host-to-device copies of q, k, v for chunk c+1 run while chunk c's fa_fwd_ex computes and
    chunk c-1's o, lse travel back, so that the step costs about the copies plus one chunk's
    compute (the copies alone take longer than the forward)."""
    import torch
    from exact_attention_06_gb300 import fattn, inputs
    bh = w.B * w.H
    n_chunks = E2E_CHUNKS if bh % E2E_CHUNKS == 0 else w.B
    hc = bh // n_chunks  # heads per chunk
    qh, kh, vh = (t.pin_memory().view(bh, w.N, w.d) for t in inputs.workload_inputs(w, seed=0, device="cpu"))
    oh = torch.empty((bh, w.N, w.d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((bh, w.N), dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
    od = torch.empty_like(qd)
    ld = torch.empty((bh, w.N), dtype=torch.float32, device=dev)
    ws = _tail_workspace(inputs.Workload(w.name, w.kind, 1, hc, w.N, w.d, w.causal), dev)
    s_in, s_fwd, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def step():
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        for c in range(n_chunks):
            sl = slice(c * hc, (c + 1) * hc)
            with torch.cuda.stream(s_in):
                qd[sl].copy_(qh[sl], non_blocking=True)
                kd[sl].copy_(kh[sl], non_blocking=True)
                vd[sl].copy_(vh[sl], non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            s_fwd.wait_event(e_in)
            fattn.fa_fwd_ex(qd[sl].unsqueeze(0), kd[sl].unsqueeze(0), vd[sl].unsqueeze(0), od[sl].unsqueeze(0),
                            ld[sl].unsqueeze(0), w.scale, w.causal, stream=s_fwd, workspace=ws)
            e_fwd = torch.cuda.Event()
            e_fwd.record(s_fwd)
            s_out.wait_event(e_fwd)
            with torch.cuda.stream(s_out):
                oh[sl].copy_(od[sl], non_blocking=True)
                lh[sl].copy_(ld[sl], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)

    ms = _time_steps(step, steps, warmup, stream)
    t = statistics.mean(ms)
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return {"value": round(w.flops() / (t * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "ms_per_step": round(t, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": f"{n_chunks} chunks of {hc} heads; H2D, fa_fwd_ex and D2H on three streams"}


def run_ours(args):
    import torch
    world, rank, local = _dist()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from exact_attention_06_gb300 import build as _build, inputs
    if rank == 0 or world == 1:
        _build.build()
    if dist is not None:
        dist.barrier()
    peaks = _peaks()
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.zero_()

    def dist_sync():
        if dist is not None:
            dist.barrier()

    if args.only:
        return run_only(args, inputs.WORKLOADS[args.only], dev, stream, peaks, flush)
    w = inputs.WORKLOADS[HEADLINE]
    step, launches = _prefill_step_fn(w, dev, stream)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    ms = _time_steps(step, args.steps, args.warmup, stream, flush=flush if _fits_l2(w) else None, sampler=sampler,
                     dist_sync=dist_sync)
    sampler.stop()
    t_local = statistics.mean(ms)
    t = max_over_ranks(t_local, dist, dev)
    flops = w.flops()
    value = flops * world / (t * 1e-3) / 1e12

    extra = {}
    if not args.no_extra:
        for name in EXTRA:
            we = inputs.WORKLOADS[name]
            if we.kind == "decode":
                st_fn, nl = _decode_step_fn(we, dev, stream)
            else:
                st_fn, nl = _prefill_step_fn(we, dev, stream)
            small = _fits_l2(we)
            ems = _time_steps(st_fn, args.extra_steps, max(3, args.warmup), stream, flush=flush if small else None,
                              dist_sync=dist_sync)
            et = statistics.mean(ems)
            if we.kind == "decode":
                work, kind, kern = we.kv_bytes(), "hbm", "decode_split_kernel"
                val = work / (et * 1e-3) / 1e9
                unit = "GB/s"
            else:
                work, kind, kern = we.flops(), "tensor", _fwd_kernel_name(we)
                val = work / (et * 1e-3) / 1e12
                unit = "TFLOP/s"
            extra[name] = {"value": round(val * world, 3), "unit": unit, "ms_per_step": round(et, 4),
                           "steps": args.extra_steps, "gpu_launches": nl * args.extra_steps,
                           "config": {"B": we.B, "H": we.H, "N" if we.kind == "prefill" else "L": we.N, "d": we.d,
                                      "causal": we.causal, "spike_every_64th_key_x8": we.spike},
                           "roofline": _roofline(kind, work, et, peaks, _traffic(kern, name)),
                           "l2": "flushed between timed steps (256 MiB write)" if small else "inputs larger than L2"}
            if we.kind == "decode":
                extra[name]["roofline"]["note"] = "duration covers the split kernel and the combine kernel"
            del st_fn
            torch.cuda.empty_cache()
        # backward on the causal workload (NEXT row of the plan): 2.5x the forward's flops by the usual
        # count (five N^2 d products); the dQ pass recomputes two of them, which is not counted
        wb = inputs.WORKLOADS["causal"]
        bst, nl = _backward_step_fn(wb, dev, stream)
        bms = _time_steps(bst, args.extra_steps, max(3, args.warmup), stream, dist_sync=dist_sync)
        bt = statistics.mean(bms)
        bflops = 2.5 * wb.flops()
        extra["backward_causal"] = {
            "value": round(bflops / (bt * 1e-3) / 1e12 * world, 3), "unit": "TFLOP/s", "ms_per_step": round(bt, 4),
            "steps": args.extra_steps, "gpu_launches": nl * args.extra_steps,
            "config": {"B": wb.B, "H": wb.H, "N": wb.N, "d": wb.d, "causal": True, "spike_every_64th_key_x8": True},
            "roofline": _roofline("tensor", bflops, bt, peaks, _traffic("bwd_dkdv_kernel", "causal")),
            "note": "fa_bwd: rowsum(O*dO), dK/dV pass, dQ pass; flops = 2.5 x forward (algorithmic); "
                    "traffic is the dominant dK/dV kernel's"}
        del bst
        torch.cuda.empty_cache()
        # split-KV decode over a paged cache (128-key pages, shuffled pool) on the decode workload
        wd = inputs.WORKLOADS["decode"]
        pst, nl = _paged_decode_step_fn(wd, dev, stream)
        pms = _time_steps(pst, args.extra_steps, max(3, args.warmup), stream, dist_sync=dist_sync)
        pt = statistics.mean(pms)
        extra["decode_paged"] = {
            "value": round(wd.kv_bytes() / (pt * 1e-3) / 1e9 * world, 3), "unit": "GB/s",
            "ms_per_step": round(pt, 4), "steps": args.extra_steps, "gpu_launches": nl * args.extra_steps,
            "config": {"B": wd.B, "H": wd.H, "L": wd.N, "d": wd.d, "page_size": 128, "pool": "shuffled pages"},
            "roofline": _roofline("hbm", wd.kv_bytes(), pt, peaks, _traffic("decode_split_kernel_paged", "decode")),
            "note": "fa_decode_paged: split kernel through the block table, then the combine kernel"}
        del pst
        torch.cuda.empty_cache()
        # sequence-sharded prefill of the causal workload: four key shards, then the combine
        sst, nl = _sharded_step_fn(wb, dev, stream)
        sms_ = _time_steps(sst, args.extra_steps, max(3, args.warmup), stream, dist_sync=dist_sync)
        stt = statistics.mean(sms_)
        extra["causal_sharded4"] = {
            "value": round(wb.flops() / (stt * 1e-3) / 1e12 * world, 3), "unit": "TFLOP/s",
            "ms_per_step": round(stt, 4), "steps": args.extra_steps, "gpu_launches": nl * args.extra_steps,
            "config": {"B": wb.B, "H": wb.H, "N": wb.N, "d": wb.d, "causal": True, "shards": 4,
                       "spike_every_64th_key_x8": True},
            "roofline": _roofline("tensor", wb.flops(), stt, peaks, _traffic("causal_sharded4", "causal")),
            "note": "4 x fa_fwd_partial_ex (one per 2048-key range of the whole K/V, concurrent streams) + fa_combine; "
                    "flops of the unsharded forward; traffic the DRAM bytes of the step's five launches"}
        del sst
        torch.cuda.empty_cache()
        # FP8 forward on the causal workload (E4M3 inputs with per-128-row block scales)
        fst, nl = _fp8_step_fn(wb, dev, stream)
        fms = _time_steps(fst, args.extra_steps, max(3, args.warmup), stream, dist_sync=dist_sync)
        ft = statistics.mean(fms)
        extra["fp8_causal"] = {
            "value": round(wb.flops() / (ft * 1e-3) / 1e12 * world, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ft, 4), "steps": args.extra_steps, "gpu_launches": nl * args.extra_steps,
            "dtype": "e4m3 (fp32 softmax and accumulation)",
            "config": {"B": wb.B, "H": wb.H, "N": wb.N, "d": wb.d, "causal": True, "spike_every_64th_key_x8": True},
            "roofline": _roofline("tensor_fp8", wb.flops(), ft, peaks, _traffic("fwd_kernel_fp8", "causal")),
            "l2": "inputs larger than L2"}
        del fst
        torch.cuda.empty_cache()

    e2e = _e2e_prefill(w, dev, stream, max(3, min(args.steps, 50)), max(3, args.warmup))
    if world > 1:
        e2e["value"] = round(e2e["value"] * world, 3)

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    cpu = None if (args.no_cpu_baseline or world > 1) else cpu_baseline(w, budget_s=args.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded iid N(0,1) bf16)",
        "config": _headline_config(w, world),
        "gpu_launches": launches * args.steps,
        "roofline": dict(_roofline("tensor", flops, t_local, peaks, _traffic(_fwd_kernel_name(w), HEADLINE)),
                         note=f"one {_fwd_kernel_name(w)} launch per step; flops 4*B*H*N^2*d"
                              f"{' / 2 (causal)' if w.causal else ''}, traffic its DRAM bytes per launch"),
        "clocks": sampler.summary(),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_only(args, w, dev, stream, peaks, flush):
    """One workload alone (profiler captures and sweeps): its step timed like the headline."""
    fn = (_paged_decode_step_fn if args.paged else _decode_step_fn) if w.kind == "decode" else (
        (lambda w_, d_, s_: _sharded_step_fn(w_, d_, s_, args.shards)) if args.shards else (
        _backward_step_fn if args.backward else (_fp8_step_fn if args.fp8 else _prefill_step_fn)))
    step, launches = fn(w, dev, stream)
    small = w.kind == "prefill" and 3 * w.B * w.H * w.N * w.d * 2 < L2_FLUSH_BYTES
    ms = _time_steps(step, args.steps, args.warmup, stream, flush=flush if small else None)
    t = statistics.mean(ms)
    if w.kind == "decode":
        work, kind, kern, unit = w.kv_bytes(), "hbm", "decode_split_kernel", "GB/s"
        value = work / (t * 1e-3) / 1e9
    else:
        work = w.flops() * (2.5 if args.backward else 1.0)
        kind = "tensor_fp8" if args.fp8 else "tensor"
        kern = "bwd" if args.backward else ("fwd_kernel_fp8" if args.fp8 else (
            "fwd_persist_kernel" if (not w.causal and w.d == 64) else "fwd_kernel"))
        unit = "TFLOP/s"
        value = work / (t * 1e-3) / 1e12
    tag = (" backward" if args.backward else "") + (" fp8" if args.fp8 else "") + (" paged" if args.paged else "")
    tag += f" sharded{args.shards}" if args.shards else ""
    print(json.dumps({"workload": w.name + tag, "value": round(value, 3), "unit": unit, "steps": args.steps,
                      "warmup": args.warmup, "ms_per_step": round(t, 5), "ms_min": round(min(ms), 5),
                      "gpu_launches": launches * args.steps,
                      "roofline": _roofline(kind, work, t, peaks, _traffic(kern, w.name))}), flush=True)


# ----------------------------------------------------------------------------- oracle (CPU) arm

_CPU_SAMPLE_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle
from exact_attention_06_gb300 import inputs
w = inputs.WORKLOADS[{name!r}]
steps, per_step, rows_per_call = {steps!r}, {per_step!r}, {rows!r}
heads = min(w.H, 2)  # rows are sampled from the first heads: every head has the same shape
q, k, v = inputs.prefill_inputs(1, heads, w.N, w.d, seed=0, device="cpu", spike=w.spike)
out = []
calls = 0
for _ in range(steps):
    done_rows, flops = 0, 0.0
    t0 = time.perf_counter()
    while True:
        h = calls % heads
        rows = inputs.sample_rows(w.N, rows_per_call, seed=calls).numpy()
        oracle.attention_head(q[0, h], k[0, h], v[0, h], w.scale, w.causal, rows=rows)
        done_rows += len(rows)
        # algorithmic flops of the evaluated rows: 4*d per admissible key
        flops += 4.0 * w.d * float(np.sum(rows + 1 if w.causal else np.full(len(rows), w.N)))
        calls += 1
        el = time.perf_counter() - t0
        if el >= per_step:
            break
    out.append({{"seconds": el, "rows": done_rows, "flops": flops}})
print(json.dumps(out))
"""


def _oracle_steps(w, steps, per_step_s, rows, threads=None):
    """Run the fp64 oracle as it stands in a fresh process with `threads` BLAS threads (default: every
    core of this process's affinity): `steps` bounded samples of the workload's rows."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = threads or cores
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    script = _CPU_SAMPLE_SCRIPT.format(root=ROOT, name=w.name, steps=int(steps), per_step=float(per_step_s),
                                       rows=int(rows))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, env=env,
                       timeout=180 + steps * (per_step_s + 30))
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-500:])
    return json.loads(r.stdout.strip().splitlines()[-1]), threads


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return None


def cpu_baseline(w, budget_s=12.0, rows=256):
    """The fp64 oracle on the host cores over bounded samples (~budget_s seconds each) of the
    workload's rows: once on every core of the affinity mask (the reported value) and once on one
    thread, each with seconds per row and a labelled extrapolation to the whole workload."""
    legs = {}
    try:
        for label, threads in (("all_cores", None), ("one_thread", 1)):
            res, used = _oracle_steps(w, 1, budget_s, rows, threads)
            r = res[0]
            rate = r["flops"] / r["seconds"]
            legs[label] = {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": used,
                           "seconds": round(r["seconds"], 2), "rows": r["rows"],
                           "seconds_per_row": round(r["seconds"] / r["rows"], 6),
                           "extrapolated_full_workload_s": round(w.flops() / rate, 1)}
    except (RuntimeError, subprocess.TimeoutExpired) as e:
        return {"value": None, "unit": "TFLOP/s", "kind": "oracle", "error": str(e)[-300:]}
    a = legs["all_cores"]
    return {"value": a["value"], "unit": "TFLOP/s", "cores": a["cores"], "kind": "oracle",
            "sample": f"{a['rows']} seeded query rows of the {_workload_label(w)} workload ({rows} rows per call, "
                      f"explicit fp64 score rows, drawn from its first heads) in {a['seconds']:.1f} s on "
                      f"{a['cores']} numpy/BLAS threads; the same for one thread below",
            "seconds": a["seconds"], "seconds_per_row": a["seconds_per_row"],
            "extrapolated_full_workload_s": a["extrapolated_full_workload_s"],
            "extrapolation": "labelled extrapolation: the whole workload's algorithmic flops at the sampled rate",
            "one_thread": legs["one_thread"], "cpu_model": _cpu_model()}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    from exact_attention_06_gb300 import inputs
    w = inputs.WORKLOADS[HEADLINE]
    total = args.steps + args.warmup
    per_step = max(0.05, min(20.0, args.ref_seconds / total))  # one 64-row call takes ~0.05 s
    res, cores = _oracle_steps(w, total, per_step, 64)
    timed = res[args.warmup:]
    secs = sum(r["seconds"] for r in timed)
    flops = sum(r["flops"] for r in timed)
    value = flops / secs / 1e12
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000.0 * secs / len(timed), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1) bf16)",
        "config": _headline_config(w, world),
        "arm": "the fp64 oracle as it stands, single process on the host cores",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: seeded query rows of the {_workload_label(w)} workload for "
                                   f"{per_step:.2f} s (64 rows per call, explicit fp64 score rows); "
                                   f"numpy/BLAS threads={cores}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # ~30 ms timed at the headline's ~1.45 ms a step: a burst like the measured bf16 peak the
    # roofline divides by (the best of ten back-to-back GEMMs); longer runs settle under the power
    # cap, which the clocks record names (sw_power_cap)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--only", default=None, help="time one named workload alone (e.g. causal, decode_small)")
    ap.add_argument("--backward", action="store_true", help="with --only: time fa_bwd instead of the forward")
    ap.add_argument("--fp8", action="store_true", help="with --only: time the FP8 forward (fa_fwd_fp8)")
    ap.add_argument("--paged", action="store_true", help="with --only and a decode workload: time fa_decode_paged")
    ap.add_argument("--shards", type=int, default=0, help="with --only and a prefill workload: key shards + combine")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
