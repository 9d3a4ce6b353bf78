#!/usr/bin/env python
"""Benchmark of the fused quantized LM-head on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step is one pass of the whole hot path over one batch of synthetic input:
  * training configs (gemma8k_masked, the default; gemma512, mid8, tiny):
    forward (logp, lse, argmax) + backward (dh) over all rows;
  * verify (the gamma+1 speculative-decode window): one forward (lse + argmax
    of every position) over M = 5 rows.
The default line is the 8192-row masked Gemma-class training step; it also
carries, under "verify_window", the verify window measured in the same run on
the same head, with its own HBM roofline.
`value` is tokens/s over all ranks with inputs already resident in HBM;
`e2e` is the same metric through the C ABI with the step's inputs copied from
pinned host memory and its results read back inside the timed region.
Multi-GPU runs are replicas (weak scaling): every rank runs the same
workload on its own GPU, timed between barriers, max over ranks.
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from verify_vocab_blocked_gb300 import synth  # noqa: E402

METRIC = "fused qhead logp tokens/s (fwd, fwd+bwd) + % of tensor-core / HBM roofline"
UNIT = "tokens/s"
DEFAULT_CONFIG = "gemma8k_masked"
EVENT_STRIDE = 16
# The pages' own timing, for context only (another machine, another precision,
# a real head): the e4b-class head at M = 512, forward 180 ms + backward 754 ms
# on an Apple M1 Max with fp32 operands.  It is not a baseline for any
# workload here, so vs_baseline stays null.
PAGES_CONTEXT = {"workload": "e4b-class head (V=262144, H=2560, 4-bit), M=512, fwd+bwd",
                 "hardware": "Apple M1 Max (Metal), fp32 operands",
                 "ms_fwd": 180.0, "ms_bwd": 754.0, "tokens_per_s": 512 / (0.180 + 0.754),
                 "note": "context only, not a baseline"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def code_of(text: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed: what a
    recorded measurement depends on (edits to comments keep it valid)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(sources) -> str | None:
    """sha256 (16 hex digits) of the code of the named csrc files (comments
    and whitespace left out), concatenated in order."""
    h = hashlib.sha256()
    for name in sources:
        src = os.path.join(ROOT, "verify_vocab_blocked_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        with open(src, encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel: str, workload: str):
    """ncu DRAM bytes per launch of `kernel` on `workload`, if recorded for the
    current sources of the kernel (its .cu and the headers it includes)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or source_hash(e["sources"]) != e["sha256_16"]:
        return None
    return e


def workload_desc(name: str, cfg: dict) -> dict:
    d = {"workload": f"{name}: {cfg['desc']}", "M": cfg["M"], "H": cfg["H"], "V": cfg["V"],
         "bits": cfg["bits"], "group": cfg["group"], "softcap": cfg["softcap"],
         "pass": "fwd+bwd" if cfg["bwd"] else "fwd",
         "l2": "inputs larger than L2 (packed head %.1f MB > 129 MB L2)"
               % (cfg["V"] * (cfg["H"] * cfg["bits"] / 8 + 4 * cfg["H"] / 64) / 1e6),
         "parallelism": "replicas"}
    if cfg.get("mask"):
        d["mask"] = "30%% masked: prompt prefix of %d tokens per %d-token sequence" % (
            round(cfg["mask"][1] * cfg["mask"][0]), cfg["mask"][0])
    return d


def head_bytes(cfg: dict) -> int:
    """Algorithmic bytes of one pass over the head: packed codes + fp16 scales and biases."""
    V, H = cfg["V"], cfg["H"]
    return V * (H * cfg["bits"] // 8 + 2 * 2 * (H // 64))


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sms.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------ our arm

class Runner:
    """Device buffers for one workload and the C-ABI calls of one step."""

    def __init__(self, wl: synth.Workload, device, with_dw: bool = False,
                 blockskip: float | None = None, filter_eps: float | None = None,
                 head=None):
        import ctypes

        import torch
        from verify_vocab_blocked_gb300 import qhead
        self.torch, self.q = torch, qhead
        self.wl = wl
        self.dev = device
        # `head`: the same head already resident on the device (another
        # workload's with identical head parameters), shared instead of copied.
        self.head = head if head is not None else qhead.Head.from_numpy(
            wl.head.wq, wl.head.scales, wl.head.biases, wl.head.bits, wl.head.group,
            wl.head.softcap, device=device)
        M = wl.M
        self.M = M
        self.h_host = torch.from_numpy(wl.h.astype(np.int16)).view(torch.bfloat16).pin_memory()
        self.h = self.h_host.to(device)
        self.bwd = bool(wl.cfg["bwd"])
        self.with_dw = with_dw and self.bwd  # the backward also returns the head gradient
        # approximate backward: the blockMax early exit with this eps
        self.blockskip = blockskip if self.bwd else None
        # approximate backward: the coefficient filter with this eps
        self.filter_eps = filter_eps if self.bwd and blockskip is None else None
        self.t_host = (torch.from_numpy(wl.targets).pin_memory()
                       if wl.targets is not None else None)
        self.t = self.t_host.to(device) if self.t_host is not None else None
        self.m_host = torch.from_numpy(wl.mask).pin_memory() if wl.mask is not None else None
        self.mk = self.m_host.to(device) if self.m_host is not None else None
        self.g_host = torch.from_numpy(wl.dlogp).pin_memory()
        self.g = self.g_host.to(device)
        f32, i32 = torch.float32, torch.int32
        # The per-row results (logp, lse, argmax) share one device buffer, so
        # the end-to-end leg reads them back with a single copy.
        self.rows_out = torch.empty(3, M, dtype=i32, device=device)
        self.logp = self.rows_out[0].view(f32) if self.t is not None else None
        self.lse = self.rows_out[1].view(f32)
        self.am = self.rows_out[2]
        self.dh = torch.empty(M, wl.head.H, dtype=f32, device=device) if self.bwd else None
        self.dw = (torch.empty(wl.head.V, wl.head.H, dtype=f32, device=device)
                   if self.with_dw else None)
        n = qhead.fwd_workspace(self.head, M)
        if self.bwd:
            n = max(n, qhead.bwd_dw_workspace(self.head, M) if self.with_dw
                    else qhead.bwd_workspace(self.head, M))
        self.bm = None
        if self.blockskip is not None:
            self.bm = torch.full((M, (wl.head.V + 255) // 256), float("-inf"), dtype=f32,
                                 device=device)
            L0 = qhead.lib()
            n = max(n, L0.qhead_fwd_blockmax_workspace(ctypes.byref(self.head.c()), M),
                    L0.qhead_bwd_blockskip_workspace(ctypes.byref(self.head.c()), M))
        if self.filter_eps is not None:
            L0 = qhead.lib()
            n = max(n, L0.qhead_bwd_filter_workspace(ctypes.byref(self.head.c()), M))
        self.ws = qhead.alloc_workspace(n, device)
        self.chead = self.head.c()
        self.stream = torch.cuda.current_stream(device)
        # pinned outputs for the end-to-end leg
        self.out_host = {k: torch.empty_like(v, device="cpu").pin_memory()
                         for k, v in (("rows", self.rows_out), ("dh", self.dh), ("dw", self.dw))
                         if v is not None}
        self.launches_per_step = None  # counted on the device by count_launches()
        self.active = int(wl.mask.sum()) if wl.mask is not None else M

    def _ptr(self, t):
        return None if t is None else t.data_ptr()

    def step(self, ev_fwd=None, ev_bwd=None):
        import ctypes
        L = self.q.lib()
        if ev_fwd is not None:
            L.qhead_time_next_head_kernel(ev_fwd[0].cuda_event, ev_fwd[1].cuda_event)
        if self.bm is not None:
            rc = L.qhead_fwd_blockmax(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                                      self._ptr(self.t), self._ptr(self.mk), self._ptr(self.logp),
                                      self.lse.data_ptr(), self.am.data_ptr(), self.bm.data_ptr(),
                                      self.ws.data_ptr(), self.ws.numel(), self.stream.cuda_stream)
        else:
            rc = L.qhead_fwd(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                             self._ptr(self.t), self._ptr(self.mk), self._ptr(self.logp),
                             self.lse.data_ptr(), self.am.data_ptr(), self.ws.data_ptr(),
                             self.ws.numel(), self.stream.cuda_stream)
        if rc:
            raise RuntimeError(self.q.last_error())
        if self.bwd:
            if ev_bwd is not None:
                L.qhead_time_next_head_kernel(ev_bwd[0].cuda_event, ev_bwd[1].cuda_event)
            if self.bm is not None:
                rc = L.qhead_bwd_blockskip(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                                           self.t.data_ptr(), self._ptr(self.mk),
                                           self.lse.data_ptr(), self.g.data_ptr(),
                                           self.bm.data_ptr(), float(self.blockskip),
                                           self.dh.data_ptr(), self.ws.data_ptr(),
                                           self.ws.numel(), self.stream.cuda_stream)
            elif self.filter_eps is not None:
                rc = L.qhead_bwd_filter(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                                        self.t.data_ptr(), self._ptr(self.mk),
                                        self.lse.data_ptr(), self.g.data_ptr(),
                                        ctypes.c_float(self.filter_eps), self.dh.data_ptr(),
                                        None, self.ws.data_ptr(), self.ws.numel(),
                                        self.stream.cuda_stream)
            elif self.with_dw:
                rc = L.qhead_bwd_dw(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                                    self.t.data_ptr(), self._ptr(self.mk), self.lse.data_ptr(),
                                    self.g.data_ptr(), self.dh.data_ptr(), self.dw.data_ptr(),
                                    self.ws.data_ptr(), self.ws.numel(), self.stream.cuda_stream)
            else:
                rc = L.qhead_bwd(ctypes.byref(self.chead), self.h.data_ptr(), self.M,
                                 self.t.data_ptr(), self._ptr(self.mk), self.lse.data_ptr(),
                                 self.g.data_ptr(), self.dh.data_ptr(), self.ws.data_ptr(),
                                 self.ws.numel(), self.stream.cuda_stream)
            if rc:
                raise RuntimeError(self.q.last_error())

    def h2d(self):
        n = 0
        for src, dst in ((self.h_host, self.h), (self.t_host, self.t), (self.m_host, self.mk),
                         (self.g_host if self.bwd else None, self.g)):
            if src is not None:
                dst.copy_(src, non_blocking=True)
                n += src.numel() * src.element_size()
        return n

    def d2h(self):
        n = 0
        # logp (when targets are given), lse and argmax in one copy; dh and dW
        for k, dev in (("rows", self.rows_out if self.t is not None else self.rows_out[1:]),
                       ("dh", self.dh), ("dw", self.dw)):
            if dev is not None:
                dst = self.out_host[k] if k != "rows" or self.t is not None else self.out_host[k][1:]
                dst.copy_(dev, non_blocking=True)
                n += dev.numel() * dev.element_size()
        return n


def count_launches(R: Runner) -> tuple[int, dict]:
    """This library's kernel launches in one step, counted by the CUDA activity
    profiler (CUPTI) from its exported trace: returns the total and the
    per-kernel counts."""
    import re
    import tempfile
    import torch
    from torch.profiler import ProfilerActivity, profile
    from torch.profiler import record_function
    torch.cuda.synchronize()
    # Kernel records appear in the trace only when CPU activity is traced too;
    # the step itself is a CPU range so the trace has a parent for them.
    # The first profiling session of a process records no device activity
    # (the activity tracer attaches lazily): open and discard one first.
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]):
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
        with record_function("qhead_step"):
            R.step()
            torch.cuda.synchronize()
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "trace.json")
        prof.export_chrome_trace(path)
        with open(path) as f:
            trace = json.load(f)
    counts: dict = {}
    for e in trace.get("traceEvents", []):
        name = e.get("name", "")
        if e.get("cat") != "kernel" or ("qh::" not in name and "_ZN2qh" not in name):
            continue
        m = re.search(r"(\w+_kernel)", name)
        short = m.group(1) if m else name
        counts[short] = counts.get(short, 0) + 1
    if not counts:
        cats: dict = {}
        for e in trace.get("traceEvents", []):
            cats[str(e.get("cat"))] = cats.get(str(e.get("cat")), 0) + 1
        return None, {"note": "no kernel of this library in the CUDA activity trace",
                      "trace_categories": cats}
    return sum(counts.values()), counts


def aggregate(elapsed_ms: float, units: float, world: int, dist=None) -> tuple[float, float]:
    """Max of the ranks' elapsed time and the sum of their units (replicas)."""
    if world > 1 and dist is not None:
        import torch
        t = torch.tensor([elapsed_ms], dtype=torch.float64)
        u = torch.tensor([units], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t, u = t.cuda(), u.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        return float(t.item()), float(u.item())
    return elapsed_ms, units


def cpu_baseline(wl: synth.Workload, budget_s: float = 12.0, max_reps: int = 64,
                 with_dw: bool = False) -> dict:
    """The fp64 oracle, as it stands, on a bounded sample: one row of the
    workload (full vocab), forward (+ backward, and the head gradient with
    with_dw, for training configs), repeated until the budget is spent."""
    import oracle
    oh = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, wl.head.bits, wl.head.group,
                     wl.head.softcap)
    bwd = bool(wl.cfg["bwd"])
    act = np.nonzero(wl.mask)[0] if wl.mask is not None else np.arange(wl.M)
    t0 = time.perf_counter()
    reps = 0
    while reps < max_reps:
        r = act[reps % len(act):reps % len(act) + 1]
        tg = wl.targets[r] if wl.targets is not None else None
        f = oracle.forward(wl.h[r], oh, tg)
        if bwd:
            oracle.backward(wl.h[r], oh, tg, wl.dlogp[r].astype(np.float64), lse=f.lse)
            if with_dw:
                oracle.grad_head(wl.h[r], oh, tg, wl.dlogp[r].astype(np.float64), lse=f.lse)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": reps / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} x 1 row of the workload (full V={wl.head.V}), "
                      f"{('fwd+bwd+dW' if with_dw else 'fwd+bwd') if bwd else 'fwd'}, fp64, "
                      f"{el:.1f} s"}


def event_stride(K: int) -> int:
    """Every how many timed steps the head kernel is bracketed by events: a
    stream event between two launches costs the step the overlap of the next
    launch (~9 us of a 90 us verify step when every step carries a pair)."""
    return EVENT_STRIDE if K >= 4 * EVENT_STRIDE else 4 if K >= 8 else 1


def timed_region(R: Runner, K: int, W: int, dist=None, local: int = 0):
    """W untimed steps, then K steps timed on the device between barriers and
    synchronizes, with the head kernel (and the backward chain) timed by CUDA
    events on every event_stride(K)-th step.  Returns (elapsed ms, forward
    kernel ms per sample, backward chain ms per sample, clock summary)."""
    import torch
    mk_ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    stride = event_stride(K)
    sampled = [i % stride == 0 for i in range(K)]
    ev_f = [(mk_ev(), mk_ev()) if sampled[i] else None for i in range(K)]
    ev_b = [(mk_ev(), mk_ev()) if sampled[i] and R.bwd else None for i in range(K)]
    for pair in [p for p in ev_f + ev_b if p]:  # create the events before timing
        pair[0].record()
        pair[1].record()
    for _ in range(W):
        R.step()
    torch.cuda.synchronize()
    t0, t1 = mk_ev(), mk_ev()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record()
        for i in range(K):
            R.step(ev_f[i], ev_b[i])
        t1.record()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return (t0.elapsed_time(t1), [p[0].elapsed_time(p[1]) for p in ev_f if p],
            [p[0].elapsed_time(p[1]) for p in ev_b if p], clk.summary())


def e2e_region(R: Runner, K: int, dist=None):
    """K steps through the C ABI from pinned host inputs to host outputs, the
    copies inside the timed region.  Returns (elapsed ms, h2d bytes per step,
    d2h bytes per step)."""
    import torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record()
    h2d = d2h = 0
    for _ in range(K):
        h2d = R.h2d()
        R.step()
        d2h = R.d2h()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), h2d, d2h


def hbm_roofline(cfg: dict, kms: float, hbm: float, peak_src: str, workload: str) -> dict:
    """The weight-streaming kernel against the measured copy bandwidth."""
    nbytes = head_bytes(cfg)
    achieved = nbytes / (kms / 1e3) / 1e9
    tr = _traffic("stream_fwd_kernel", workload)
    return {"kernel": "stream_fwd_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm,
            "unit": "GB/s", "frac": achieved / hbm,
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "work_per_launch": f"{nbytes} bytes (packed head + fp16 scales/biases)",
            "ms_per_launch": kms, "traffic": tr["dram_bytes_per_launch"] if tr else None}


def verify_window(dev, head_dev, head_np, local: int, count: bool = True, steps: int = 2000,
                  warmup: int = 50):
    """The gamma+1 verify window on the same head, measured in the same run:
    tokens/s, the step time and the streaming kernel's HBM roofline."""
    cfg = synth.CONFIGS["verify"]
    wl = synth.make_workload("verify", seed=0, head=head_np)
    R = Runner(wl, dev, head=head_dev)
    el, fwd_ms, _, clk = timed_region(R, steps, warmup, None, local)
    hbm, _, _, peak_src = _peaks()
    launches = count_launches(R)[1] if count else {"note": "not counted (--no-launch-count)"}
    return {"workload": workload_desc("verify", cfg)["workload"], "metric": "tokens/s",
            "value": R.active * steps / (el / 1e3), "ms_per_step": el / steps, "steps": steps,
            "warmup": warmup,
            "roofline": dict(hbm_roofline(cfg, statistics.mean(fwd_ms), hbm, peak_src, "verify"),
                             kernel_timing=f"CUDA events around the kernel on every "
                                           f"{event_stride(steps)}th timed step"),
            "launches_per_step": launches, "clocks": clk}


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = synth.CONFIGS[args.config]
    wl = synth.make_workload(args.config, seed=0)
    R = Runner(wl, dev, with_dw=args.with_dw, blockskip=args.blockskip,
               filter_eps=args.filter)
    K, W = args.steps, args.warmup
    stride = event_stride(K)

    # launches of one step, counted after a first warm-up step
    R.step()
    torch.cuda.synchronize()
    if args.no_launch_count:
        n_launch, launch_list = None, {"note": "not counted (--no-launch-count)"}
    else:
        n_launch, launch_list = count_launches(R)
    R.launches_per_step = n_launch

    # device-resident timed region
    el, fwd_ms, bwd_ms, clocks = timed_region(R, K, W, dist, local)
    el_max, units = aggregate(el, R.active * K, world, dist)
    value = units / (el_max / 1e3)

    # end-to-end timed region: pinned host inputs -> C ABI -> host outputs
    el_e, h2d, d2h = e2e_region(R, K, dist)
    el_e_max, units_e = aggregate(el_e, R.active * K, world, dist)

    hbm, tf_burst, tf_sus, peak_src = _peaks()
    timing = ("CUDA events around the head kernel on every "
              + (f"{stride}th timed step" if stride > 1 else "timed step"))
    if R.bwd:
        # dominant work: the backward head phase (logits recomputed, 2*Ma*V*H,
        # and the dh contraction, 2*Ma*V*H): a chain of two tensor-core kernels
        # per vocab chunk, timed as one region.  With the head gradient
        # (--with-dw) a third contraction per chunk, 2*Ma*V*H more, joins it.
        # The kernels are event-timed inside a run of well under a second, so
        # the denominator is the burst GEMM rate, not the power-capped
        # sustained one (which needs seconds of back-to-back work).
        dom = "tc_bwd_chain_dw" if R.with_dw else "tc_bwd_chain"
        nmul = 6.0 if R.with_dw else 4.0
        flops = nmul * R.active * cfg["V"] * cfg["H"]
        kms = statistics.mean(bwd_ms)
        achieved = flops / (kms / 1e3) / 1e12
        kname = "tc_fwd_kernel<coefficient epilogue> + tc_dh_kernel"
        if R.with_dw:
            kname += " + tc_dw_kernel"
        if R.blockskip is not None:
            dom = "tc_bwd_chain_blockskip"
        if R.filter_eps is not None:
            dom = "tc_bwd_chain_filter"
        psrc = (f"{peak_src} bf16_tflops (burst; dense, the same rate as fp16): the kernels "
                f"are event-timed inside a {el_max / 1e3:.2f} s run")
        roof = {"kernel": kname + " per vocab chunk",
                "bound": "tensor", "achieved": achieved, "peak": tf_burst,
                "unit": "TFLOP/s", "frac": achieved / tf_burst, "peak_source": psrc,
                "work_per_launch": f"{flops:.3e} flop ({int(nmul)}*Ma*V*H, Ma = active rows; "
                                   "one launch = one backward call's kernel chain)",
                "ms_per_launch": kms, "kernel_timing": timing}
        fms = statistics.mean(fwd_ms)
        ff = 2.0 * R.active * cfg["V"] * cfg["H"]
        roof["fwd_kernel"] = {"kernel": "tc_fwd_kernel" if R.M >= 17 else "stream_fwd_kernel",
                              "ms_per_launch": fms,
                              "achieved_tflops": ff / (fms / 1e3) / 1e12,
                              "frac": ff / (fms / 1e3) / 1e12 / tf_burst}
        step_ms = el_max / K
        sf = (nmul + 2.0) * R.active * cfg["V"] * cfg["H"]
        roof["step"] = {"flop": sf, "ms": step_ms,
                        "achieved_tflops": sf / (step_ms / 1e3) / 1e12,
                        "frac": sf / (step_ms / 1e3) / 1e12 / tf_burst}
        tr = _traffic(dom, args.config)
        roof["traffic"] = tr["dram_bytes_per_launch"] if tr else None
    else:
        roof = dict(hbm_roofline(cfg, statistics.mean(fwd_ms), hbm, peak_src, args.config),
                    kernel_timing=timing)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": el_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16", "data": "synthetic (seeded; no real weights or data)",
        "config": dict(workload_desc(args.config, cfg),
                       **({"pass": "fwd+bwd (dh and dW)"} if R.with_dw else {}),
                       **({"pass": "fwd+bwd, approximate: blockMax early exit",
                           "blockskip_eps": R.blockskip,
                           "flop_accounting": "exact-equivalent (skipped blocks counted as "
                                              "done): an effective rate"}
                          if R.blockskip is not None else {}),
                       **({"pass": "fwd+bwd, approximate: coefficient filter",
                           "filter_eps": R.filter_eps,
                           "flop_accounting": "exact-equivalent (skipped dh steps counted as "
                                              "done): an effective rate"}
                          if R.filter_eps is not None else {})),
        "roofline": roof,
        "e2e": {"value": units_e / (el_e_max / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": R.launches_per_step * K if R.launches_per_step is not None else None,
        "launches_per_step": launch_list,
        "clocks": clocks,
        "pages_context": PAGES_CONTEXT,
        "impl": "ours",
    }
    if (R.bwd and not args.no_verify and world == 1 and rank == 0
            and synth.CONFIGS["verify"]["H"] == cfg["H"] and cfg.get("peaked") is None):
        try:
            line["verify_window"] = verify_window(dev, R.head, wl.head, local,
                                                  count=not args.no_launch_count)
        except ValueError:  # a head with other parameters: no shared verify line
            pass
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, with_dw=R.with_dw)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_reference(args):
    """The fp64 oracle on the host cores, each step a bounded sample (one row of
    the workload over the full vocab), stopped early past a time cap."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = synth.CONFIGS[args.config]
    wl = synth.make_workload(args.config, seed=0)
    oracle.build()
    oh = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, wl.head.bits, wl.head.group,
                     wl.head.softcap)
    bwd = bool(cfg["bwd"])
    act = np.nonzero(wl.mask)[0] if wl.mask is not None else np.arange(wl.M)

    def one(i):
        r = act[i % len(act):i % len(act) + 1]
        tg = wl.targets[r] if wl.targets is not None else None
        f = oracle.forward(wl.h[r], oh, tg)
        if bwd:
            oracle.backward(wl.h[r], oh, tg, wl.dlogp[r].astype(np.float64), lse=f.lse)
            if args.with_dw:
                oracle.grad_head(wl.h[r], oh, tg, wl.dlogp[r].astype(np.float64), lse=f.lse)

    cap_s = 180.0
    w0 = time.perf_counter()
    for i in range(args.warmup):
        one(i)
        if time.perf_counter() - w0 > cap_s / 4:
            break
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        one(i)
        done += 1
        if time.perf_counter() - t0 > cap_s:
            break
    el = time.perf_counter() - t0
    value = done / el
    sample = (f"{done} of {args.steps} steps (time cap {cap_s:.0f} s), each 1 row of the workload "
              f"(full V={cfg['V']}), "
              f"{('fwd+bwd+dW' if args.with_dw else 'fwd+bwd') if bwd else 'fwd'}, fp64")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", 1)),
        "steps": done, "warmup": args.warmup, "ms_per_step": el / max(done, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no real weights or data)",
        "config": workload_desc(args.config, cfg), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--blockskip", type=float, default=None, metavar="EPS",
                    help="training configs: the approximate backward (blockMax early exit "
                         "with this eps; e.g. with --config gemma8k_peaked)")
    ap.add_argument("--filter", type=float, default=None, metavar="EPS",
                    help="training configs: the approximate backward (coefficient filter "
                         "with this eps; e.g. with --config gemma8k_peaked)")
    ap.add_argument("--with-dw", action="store_true",
                    help="training configs: the backward also returns the head gradient dW "
                         "(qhead_bwd_dw)")
    ap.add_argument("--no-launch-count", action="store_true",
                    help="skip the CUPTI launch count (for runs under a profiler)")
    ap.add_argument("--no-verify", action="store_true",
                    help="training configs: leave out the verify-window measurement on the "
                         "same head")
    args = ap.parse_args(argv)
    if (args.blockskip is not None) + (args.filter is not None) + args.with_dw > 1:
        ap.error("--blockskip, --filter and --with-dw select different backward entry points: "
                 "give at most one")
    fwd_only = not synth.CONFIGS[args.config]["bwd"]
    if args.steps is None:
        args.steps = 3000 if fwd_only else 20
    if args.warmup is None:
        args.warmup = 50 if fwd_only else 5
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
