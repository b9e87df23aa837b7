"""Throughput of exact attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gpt2_small] [--no-sweep]

One "step" is one pass of the hot path over one batch of the workload: the
forward kernel, then the backward's preprocess, main and dQ-convert kernels.
The headline workload is the largest single-GPU configuration: long-context
non-causal attention with B=1, H=16, N=16384, d=128 (bf16 Q, K, V, dO drawn
N(0, 0.5^2) from a seed, plus a per-head rank-8 bias on Q and K). The other
configurations (GPT-2 small, BERT-large with key padding, N = 4K/8K
causal and not, block-sparse at 16K, dropout, [B,N,H,d] storage, and the
one-tile case) are timed in the sweep. FLOPs per step follow the usual
count: forward 4*B*H*N^2*d, backward 2.5x that, both halved for causal.

Timing: inputs resident in HBM; W untimed warm-up steps; then K steps, each
bracketed by CUDA events on the launching stream, with a 256 MiB buffer
written between steps (outside the events) to flush the 126 MiB L2. Under
torchrun every rank runs the same workload (independent (b, h) problems, no
collective) and rank 0 prints the max-over-ranks time. The `e2e` leg repeats
the step through the public API with pinned host buffers and the host<->
device copies inside the timed region. `cpu_baseline` times the CPU fp64
oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


# DRAM bytes (read + write) per launch from one ncu capture, keyed by kernel and
# workload, valid only while the kernel's sources are unchanged (first 16 hex
# digits of the SHA-256 of the kernel's source followed by the shared device
# headers when it was captured; see profiles/).
NCU_TRAFFIC = {
    ("bwd_main", "long_n16384_noncausal"): (633_911_168, "fa_bwd_kernel.cuh", "616966a460650ff0"),
    ("fwd", "long_n16384_noncausal"): (245_179_392, "fa_fwd_kernel.cuh", "bf39e8e345d091cf"),
    ("bwd_main", "gpt2_small"): (78_426_624, "fa_bwd_kernel.cuh", "616966a460650ff0"),
    ("fwd", "gpt2_small"): (37_825_536, "fa_fwd_kernel.cuh", "bf39e8e345d091cf"),
}
_SHARED_HEADERS = ("fa_ptx.cuh", "fa_philox.cuh", "fa_internal.h", "fa_sched.cuh")


def source_digest(src: str):
    import hashlib
    csrc = os.path.join(ROOT, "exact_io_aware_11_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for name in (src, *_SHARED_HEADERS):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    entry = NCU_TRAFFIC.get((kernel, workload))
    if entry is None:
        return None
    nbytes, src, digest = entry
    return nbytes if source_digest(src) == digest else None


def flops(w: W.Workload):
    """Nominal fwd and bwd FLOPs: 4 B H N^2 d (halved for causal) and 2.5x that."""
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        f /= 2
    return f, 2.5 * f


def effective_flops(w: W.Workload, kv_len) -> tuple:
    """FLOPs over the visible keys only, for key padding (non-causal):
    sum over b of 4 H N len_b d, and 2.5x that."""
    f = sum(4.0 * w.H * w.N * min(w.N, int(n)) * w.d for n in kv_len.tolist())
    return f, 2.5 * f


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self, window=None):
        """Median SM clock and throttle reasons over the samples taken inside
        `window` (monotonic start, end), or over all samples."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if window is not None and not (window[0] <= t <= window[1] + 0.25):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
               "samples": len(sm), "reasons": sorted(reasons)}
        if window is not None:
            out["window"] = "1 s of untimed steps of the same workload, then the timed steps"
        return out


# --------------------------------------------------------------------------- our arm
class Step:
    """Buffers and the staged calls of one fwd+bwd step on one workload."""

    def __init__(self, fa, w: W.Workload, seed: int, dev):
        self.fa, self.w = fa, w
        x = W.make_inputs(w, seed)
        self.host = x
        def place(t):  # [B, H, N, d] view of the workload's storage order
            t = t.to(dev)
            return t.transpose(1, 2).contiguous().transpose(1, 2) if w.layout == "bnhd" else t

        self.q, self.k, self.v = (place(x[n]) for n in ("q", "k", "v"))
        self.do = place(x["dout"]) if x["dout"] is not None else None
        self.kv = x["kv_len"].to(dev) if x["kv_len"] is not None else None
        self.mask = x["block_mask"].to(dev) if x["block_mask"] is not None else None
        B, H, N, d = w.B, w.H, w.N, w.d
        def like():
            return torch.empty_strided(self.q.shape, self.q.stride(), dtype=self.q.dtype, device=dev)

        self.o = like()
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (like() for _ in range(3))
        self.opt = None
        if w.layout != "bhnd" or w.dropout > 0:  # the general entry points take strides, dropout
            self.opt = fa.AttentionOptions()
            self.opt.stride_b, self.opt.stride_h, self.opt.stride_n = self.q.stride()[:3]
            self.opt.causal, self.opt.scale = int(w.causal), w.scale
            self.opt.dropout_p, self.opt.dropout_seed = w.dropout, w.dropout_seed
            self.opt.block_size = 128
        # backward workspace with room for the split of the last wave, and the
        # forward's split workspace, where these sizes gain from the split
        plain = self.kv is None and self.mask is None
        base = fa.bwd_workspace_bytes(B, H, N, d)
        self.ws_bytes = fa.bwd_split_workspace_bytes(B, H, N, d, w.causal) if plain else base
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.fws_bytes = fa.fwd_workspace_bytes(B, H, N, d, w.causal) if plain else 0
        self.fws = (torch.empty(self.fws_bytes, dtype=torch.uint8, device=dev)
                    if self.fws_bytes else None)
        self.fwd_split = self.fws_bytes > 0
        self.bwd_split = self.ws_bytes > base
        self.L = fa.lib()
        self.offset = 0  # dropout counter offset, advanced once per step

    def launches(self):
        """Kernels of one step: the forward, then the backward's preprocess,
        main and dQ conversion. A pass split over its last wave runs its whole
        rounds on the plain kernel (when there is at least one), the tail on
        the split kernel and the merge of the cut items (counted as present)."""
        w = self.w
        G = torch.cuda.get_device_properties(self.q.device).multi_processor_count
        nt = (w.N + 127) // 128

        def split_pass(n_items):
            return (1 if n_items >= G else 0) + 2

        n = split_pass(w.B * w.H * ((nt + 1) // 2)) if self.fwd_split else 1
        if w.backward:
            n += 2 + (split_pass(w.B * w.H * nt) if self.bwd_split else 1)
        return n

    def fwd(self, stream):
        w, L = self.w, self.L
        fws = None if self.fws is None else self.fws.data_ptr()
        if self.opt is not None:
            import ctypes
            self.opt.dropout_offset = self.offset  # a fresh mask every step
            rc = L.fa_attention_fwd_split(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                                          self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.N,
                                          w.d, ctypes.byref(self.opt), fws, self.fws_bytes, stream)
        elif self.mask is not None:
            rc = L.fa_blocksparse_fwd(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                                      self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.N, w.d,
                                      w.scale, self.mask.data_ptr(), 128, stream)
        else:
            rc = L.fa_fwd_split(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                                self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.N, w.d,
                                int(w.causal), w.scale,
                                None if self.kv is None else self.kv.data_ptr(), fws,
                                self.fws_bytes, stream)
        assert rc == 0, rc

    def bwd_stages(self, stream):
        w, L = self.w, self.L
        if self.opt is not None:  # one call runs all three kernels
            import ctypes
            yield L.fa_attention_bwd(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                                     self.o.data_ptr(), self.do.data_ptr(), self.lse.data_ptr(),
                                     self.dq.data_ptr(), self.dk.data_ptr(), self.dv.data_ptr(),
                                     w.B, w.H, w.N, w.d, ctypes.byref(self.opt),
                                     self.ws.data_ptr(), self.ws_bytes, stream)
            self.offset += 1
            yield 0
            yield 0
            return
        if self.mask is not None:  # block-sparse: one call runs all three kernels
            yield L.fa_blocksparse_bwd(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                                       self.o.data_ptr(), self.do.data_ptr(), self.lse.data_ptr(),
                                       self.dq.data_ptr(), self.dk.data_ptr(), self.dv.data_ptr(),
                                       w.B, w.H, w.N, w.d, w.scale, self.mask.data_ptr(), 128,
                                       self.ws.data_ptr(), self.ws_bytes, stream)
            yield 0
            yield 0
            return
        kv = None if self.kv is None else self.kv.data_ptr()
        yield L.fa_bwd_preprocess(self.o.data_ptr(), self.do.data_ptr(), self.lse.data_ptr(),
                                  w.B, w.H, w.N, w.d, self.ws.data_ptr(), self.ws_bytes, stream)
        yield L.fa_bwd_main(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(),
                            self.do.data_ptr(), self.dk.data_ptr(), self.dv.data_ptr(), w.B, w.H,
                            w.N, w.d, int(w.causal), w.scale, kv, self.ws.data_ptr(),
                            self.ws_bytes, stream)
        yield L.fa_bwd_dq_convert(self.dq.data_ptr(), w.B, w.H, w.N, w.d, self.ws.data_ptr(),
                                  self.ws_bytes, stream)


KERNELS = ["fwd", "bwd_pre", "bwd_main", "dq_convert"]


def time_steps(step: Step, steps: int, warmup: int, flush, backward=True, split=True,
               soak_s: float = 0.0):
    """Times `steps` steps (L2 flushed before each). split=False: one pair of
    events around each whole step, so consecutive kernels overlap their
    launches (programmatic dependent launch); returns {"step": [ms, ...]}.
    split=True: an event between every two kernels (which stops that
    overlap); returns per-kernel lists. soak_s: seconds of untimed steps run
    right before the timed ones, so that clock samples see the GPU under load."""
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    n_ev = (5 if backward else 2) if split else 2
    times = ({k: [] for k in KERNELS[:n_ev - 1]} if split else {"step": []})

    def one(record):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] if record else None
        if record:
            evs[0].record(stream)
        step.fwd(sp)
        if record and split:
            evs[1].record(stream)
        if backward:
            for i, rc in enumerate(step.bwd_stages(sp)):
                assert rc == 0, rc
                if record and split:
                    evs[2 + i].record(stream)
        if record and not split:
            evs[1].record(stream)
        return evs

    if soak_s > 0:
        t_end = time.monotonic() + soak_s
        while time.monotonic() < t_end:
            for _ in range(20):
                flush.zero_()
                one(False)
            torch.cuda.synchronize()

    for _ in range(warmup):
        one(False)
    torch.cuda.synchronize()
    all_evs = []
    for _ in range(steps):
        flush.zero_()
        all_evs.append(one(True))
    torch.cuda.synchronize()
    for evs in all_evs:
        for i, name in enumerate(list(times)):
            times[name].append(evs[i].elapsed_time(evs[i + 1]))
    return times


def e2e_serial(fa, step: Step, steps: int, warmup: int):
    """Same step through the public API with pinned host buffers, one step
    after the other on one stream: H2D of the inputs, forward + backward, D2H
    of O, LSE, dQ, dK, dV, all inside the timed region."""
    w = step.w
    names = ["q", "k", "v", "dout"]
    host_in = {n: step.host[n].pin_memory() for n in names}
    dev = step.q.device
    dev_in = {n: torch.empty(host_in[n].shape, dtype=host_in[n].dtype, device=dev) for n in names}
    outs = [torch.empty(t.shape, dtype=t.dtype, device=dev)
            for t in (step.o, step.lse, step.dq, step.dk, step.dv)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    kv = step.kv
    stream = torch.cuda.current_stream()

    def one():
        for n in names:
            dev_in[n].copy_(host_in[n], non_blocking=True)
        o, lse = fa.forward(dev_in["q"], dev_in["k"], dev_in["v"], causal=w.causal, scale=w.scale,
                            kv_len=kv, out=outs[0], lse=outs[1], workspace=step.fws,
                            split=step.fwd_split)
        fa.backward(dev_in["q"], dev_in["k"], dev_in["v"], o, dev_in["dout"], lse,
                    causal=w.causal, scale=w.scale, kv_len=kv, workspace=step.ws, dq=outs[2],
                    dk=outs[3], dv=outs[4])
        for h, t in zip(host_out, outs):
            h.copy_(t, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in names)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    return ms, h2d, d2h


def e2e_pipelined(fa, step: Step, steps: int, warmup: int):
    """The same steps through the public API, software-pipelined as a training
    or serving loop runs them: while step i computes on the compute stream, the
    inputs of step i+1 upload on a copy stream and the results of step i-1
    download on another (two sets of device buffers). Every step still copies
    its inputs H2D from pinned memory and its O, LSE, dQ, dK, dV back D2H;
    events order upload -> compute -> download of each step and keep a buffer
    set from being overwritten before the step that used it is done. The timed
    region runs from before the first upload to after the last download."""
    w = step.w
    dev = step.q.device
    names = ["q", "k", "v", "dout"]
    host_in = {n: step.host[n].pin_memory() for n in names}
    dev_in = [{n: torch.empty(host_in[n].shape, dtype=host_in[n].dtype, device=dev)
               for n in names} for _ in range(2)]
    outs = [[torch.empty(t.shape, dtype=t.dtype, device=dev)
             for t in (step.o, step.lse, step.dq, step.dk, step.dv)] for _ in range(2)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs[0]]
                for _ in range(2)]
    kv = step.kv
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n, start=None, end=None):
        uploaded, computed, downloaded = [None] * n, [None] * n, [None] * n
        if start is not None:
            start.record(comp)
        up.wait_stream(comp)
        down.wait_stream(comp)
        for i in range(n + 2):
            if i < n:                                   # upload step i
                s = i % 2
                if i >= 2:
                    up.wait_event(computed[i - 2])      # its buffers' last reader is done
                with torch.cuda.stream(up):
                    for nm in names:
                        dev_in[s][nm].copy_(host_in[nm], non_blocking=True)
                uploaded[i] = torch.cuda.Event()
                uploaded[i].record(up)
            j = i - 1
            if 0 <= j < n:                              # compute step j
                s = j % 2
                comp.wait_event(uploaded[j])
                if j >= 2:
                    comp.wait_event(downloaded[j - 2])  # its outputs were copied out
                o, lse, dq, dk, dv = outs[s]
                x = dev_in[s]
                fa.forward(x["q"], x["k"], x["v"], causal=w.causal, scale=w.scale, kv_len=kv,
                           out=o, lse=lse, stream=comp, workspace=step.fws, split=step.fwd_split)
                fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=w.causal,
                            scale=w.scale, kv_len=kv, workspace=step.ws, dq=dq, dk=dk, dv=dv,
                            stream=comp)
                computed[j] = torch.cuda.Event()
                computed[j].record(comp)
            j = i - 2
            if 0 <= j < n:                              # download step j
                s = j % 2
                down.wait_event(computed[j])
                with torch.cuda.stream(down):
                    for h, t in zip(host_out[s], outs[s]):
                        h.copy_(t, non_blocking=True)
                downloaded[j] = torch.cuda.Event()
                downloaded[j].record(down)
        comp.wait_event(downloaded[n - 1])
        if end is not None:
            end.record(comp)

    run(warmup)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(steps, a, b)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in names)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    # the last step downloaded the O of its own uploaded inputs
    last = (steps - 1) % 2
    o_chk, _ = fa.forward(dev_in[last]["q"], dev_in[last]["k"], dev_in[last]["v"],
                          causal=w.causal, scale=w.scale, kv_len=kv)
    torch.cuda.synchronize()
    if not torch.equal(host_out[last][0], o_chk.cpu()):
        raise RuntimeError("pipelined end-to-end step produced a different O")
    return ms, h2d, d2h


def copy_rates(step: Step, reps: int = 5):
    """Plain pinned-memory copy rates (GB/s) of the same tensors the
    end-to-end leg moves each step: the inputs H2D alone, the outputs D2H
    alone, and both at once on two streams (as the pipelined schedule
    overlaps them), one cudaMemcpyAsync per tensor."""
    dev = step.q.device
    ins = [step.host[n] for n in ("q", "k", "v", "dout")]
    h_in = [t.pin_memory() for t in ins]
    d_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in ins]
    d_out = [step.o, step.lse, step.dq, step.dk, step.dv]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_out]
    nb_in = sum(t.numel() * t.element_size() for t in ins)
    nb_out = sum(t.numel() * t.element_size() for t in d_out)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(do_up, do_down):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            if do_up:
                with torch.cuda.stream(up):
                    for d, h in zip(d_in, h_in):
                        d.copy_(h, non_blocking=True)
            if do_down:
                with torch.cuda.stream(down):
                    for h, d in zip(h_out, d_out):
                        h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    run(True, True)  # warm-up
    t_up, t_down, t_both = run(True, False), run(False, True), run(True, True)
    return {"h2d_gbs": round(nb_in / t_up / 1e9, 1), "d2h_gbs": round(nb_out / t_down / 1e9, 1),
            "both_ms": round(t_both * 1e3, 4),
            "both_gbs": round((nb_in + nb_out) / t_both / 1e9, 1)}


def e2e(fa, step: Step, steps: int, warmup: int):
    """End-to-end timing through the public API: the pipelined schedule, or the
    serial one if the pipelined run fails. Returns (ms per step, H2D bytes,
    D2H bytes, schedule)."""
    try:
        return (*e2e_pipelined(fa, step, steps, warmup), "pipelined")
    except Exception as exc:  # noqa: BLE001 -- report the serial schedule instead
        torch.cuda.synchronize()
        return (*e2e_serial(fa, step, steps, warmup), f"serial (pipelined failed: {exc})")


def cpu_baseline(w: W.Workload, budget_s: float = 12.0):
    """Times the fp64 oracle (as it stands) on a bounded sample of the
    workload, about `budget_s` seconds of CPU work; returns TFLOP/s.

    Short sequences (N <= 2048): whole (b, h) heads, forward and backward.
    Longer ones, where one head's backward alone would take minutes: the
    forward of blocks of 256 query rows of a head of the workload (exact rows
    of its attention), and the backward of the leading 2048 x 2048 problem of
    that head, alternately."""
    import numpy as np

    import oracle
    x = W.make_inputs(w.with_(B=1, H=min(w.H, 4)), 0)
    done, t0, heads, parts = 0.0, time.perf_counter(), 0, []
    if w.N <= 2048:
        f_fwd, f_bwd = flops(w.with_(B=1, H=1))
        while True:
            h = heads % x["q"].shape[1]
            kv = None if x["kv_len"] is None else int(x["kv_len"][0])
            oracle.head_forward(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.scale, w.causal, kv)
            done += f_fwd
            if w.backward:
                oracle.head_backward(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["dout"][0, h],
                                     w.scale, w.causal, kv)
                done += f_bwd
            heads += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        sample = (f"{heads} whole (b,h) heads of {w.name} (N={w.N}, d={w.d}, "
                  f"{'fwd+bwd' if w.backward else 'fwd'}), numpy fp64, {el:.1f} s")
    else:
        q, k, v, do = (x[n][0, 0] for n in ("q", "k", "v", "dout"))
        ns, r0, nrows, nbwd = 2048, 0, 0, 0
        while True:
            rows = np.arange(r0, r0 + 256) % w.N
            oracle.head_forward(q, k, v, w.scale, w.causal, rows=rows)
            seen = (rows + 1) if w.causal else np.full(len(rows), w.N)
            done += float(4.0 * w.d * seen.sum())
            r0 += 256
            nrows += 256
            if w.backward:
                oracle.head_backward(q[:ns], k[:ns], v[:ns], do[:ns], w.scale, w.causal)
                done += 2.5 * 4.0 * ns * ns * w.d / (2 if w.causal else 1)
                nbwd += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        sample = (f"{w.name}: forward of {nrows} query rows of one head (N={w.N}, d={w.d}) and "
                  f"{nbwd} backward passes of its leading {ns}x{ns} problem, numpy fp64, {el:.1f} s")
    return {"value": done / el / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": sample, "seconds": el}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, step_flops: float, ms_local: float):
    """Whole-job TFLOP/s of `world` ranks that each ran steps of `step_flops`
    in `ms_local` ms per step: the slowest rank's time sets the job's pace.
    Returns (TFLOP/s over all ranks, max ms per step)."""
    ms = max_over_ranks(world, ms_local)
    return world * step_flops / (ms * 1e-3) / 1e12, ms


def run_ours(args, world, rank, local):
    import exact_io_aware_11_gb300 as fa
    from exact_io_aware_11_gb300 import build
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    w = W.WORKLOADS[args.workload]
    step = Step(fa, w, 0, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    # timed region: K whole steps, events only around each step
    t_region = [time.monotonic()]
    whole = time_steps(step, args.steps, args.warmup, flush, backward=w.backward, split=False,
                       soak_s=args.soak)
    t_region.append(time.monotonic())
    torch.cuda.synchronize()
    barrier(world)
    ms_local = sum(whole["step"]) / len(whole["step"])
    # the same steps again with an event between kernels: per-kernel split and
    # the dominant kernel's roofline
    times = time_steps(step, args.steps, 3, flush, backward=w.backward, split=True)
    per_kernel = {k: sum(v) / len(v) for k, v in times.items()}
    f_fwd, f_bwd = flops(w)
    step_flops = f_fwd + (f_bwd if w.backward else 0.0)
    value, ms_step = whole_job_tflops(world, step_flops, ms_local)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "device watchdog fired during the bench"

    # dominant kernel: roofline against the dense bf16 tensor peak
    dom = max(per_kernel, key=per_kernel.get)
    dom_flops = {"fwd": f_fwd, "bwd_main": f_bwd}.get(dom)
    peak_tf = pk["bf16_tflops"]
    # The kernel is timed inside a long run of steps, so its roofline takes the
    # sustained bf16 figure; the fraction of the burst figure is given beside it.
    peak_sus = pk.get("bf16_tflops_sustained", peak_tf)
    roofline = None
    if dom_flops is not None:
        ach = dom_flops / (per_kernel[dom] * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 2),
                    "peak": peak_sus, "unit": "TFLOP/s", "frac": round(ach / peak_sus, 4),
                    "peak_kind": f"{pk_kind} bf16 dense, sustained (kernel timed inside a long run "
                                 f"of steps)",
                    "frac_of_burst": round(ach / peak_tf, 4),
                    "traffic": ncu_traffic(dom, w.name)}

    e2e_ms, h2d, d2h, e2e_sched = (e2e(fa, step, max(3, args.steps // 4), 3) if w.backward
                                   else (None, 0, 0, None))
    copies = copy_rates(step) if w.backward else None
    clk = clocks.stop(window=tuple(t_region))

    out = {
        "metric": "attention fwd/bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded i.i.d. N(0,1) bf16 Q,K,V,dO)",
        "config": {"workload": f"{w.name}: {'causal' if w.causal else 'non-causal'} fwd+bwd, "
                               f"B={w.B} H={w.H} N={w.N} d={w.d}",
                   "pass": "fwd + bwd (preprocess, main, dQ convert)",
                   "launch": "programmatic dependent launch between the kernels",
                   "split": {"fwd": step.fwd_split, "bwd": step.bwd_split},
                   "l2": "flushed between timed steps (256 MiB write)",
                   "parallelism": f"replicas x{world} (independent (b,h) problems, no collective)"},
        "pct_of_bf16_peak": round(value / world / peak_tf, 4),
        "per_kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()},
        "per_kernel_timing": "second pass of the same steps with an event between kernels "
                             "(no launch overlap); ms_per_step is the whole-step timing",
        "fwd_tflops": round(f_fwd / (per_kernel["fwd"] * 1e-3) / 1e12, 2),
        "gpu_launches": args.steps * step.launches(),
        "roofline": roofline,
        "clocks": clk,
    }
    if e2e_ms is not None:
        e2e_value, e2e_ms = whole_job_tflops(world, step_flops, e2e_ms)
        out["e2e"] = {"value": round(e2e_value, 3),
                      "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": round(e2e_ms, 4), "schedule": e2e_sched,
                      "copy_gbs": round((h2d + d2h) / (e2e_ms * 1e-3) / 1e9, 1),
                      "plain_copy": copies}
    if args.sweep and rank == 0:
        out["sweep"] = sweep(fa, dev, flush, pk, w.name)
    if rank == 0 and world == 1:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    return out


def sweep(fa, dev, flush, pk, headline):
    """Fwd and bwd TFLOP/s of every other workload (few steps each)."""
    res = {}
    for name, w in W.WORKLOADS.items():
        if name == headline:
            continue
        st = Step(fa, w, 0, dev)
        t = time_steps(st, 10, 3, flush, backward=w.backward)
        whole = time_steps(st, 10, 3, flush, backward=w.backward, split=False)["step"]
        f_fwd, f_bwd = flops(w)
        if w.sparse:  # effective work: kept blocks only
            f_fwd = 4.0 * w.B * w.H * w.d * 128 * 128 * int(st.host["block_mask"].sum())
            f_bwd = 2.5 * f_fwd
        r = {"fwd_ms": round(statistics.median(t["fwd"]), 4),
             "fwd_tflops": round(f_fwd / (statistics.median(t["fwd"]) * 1e-3) / 1e12, 2),
             "split": {"fwd": st.fwd_split, "bwd": st.bwd_split}}
        step_ms = statistics.median(whole)
        r["step_ms"] = round(step_ms, 4)  # whole step, kernels chained by dependent launch
        r["step_tflops"] = round((f_fwd + (f_bwd if w.backward else 0.0)) / (step_ms * 1e-3) / 1e12, 2)
        r["fwd_pct_peak"] = round(r["fwd_tflops"] / pk["bf16_tflops"], 4)
        eff = None
        if st.host["kv_len"] is not None and not w.causal:  # the kernels skip padded key tiles
            eff = effective_flops(w, st.host["kv_len"])
            r["fwd_tflops_effective"] = round(eff[0] / (r["fwd_ms"] * 1e-3) / 1e12, 2)
        if w.backward:
            mb = statistics.median([a + b + c for a, b, c in zip(t["bwd_pre"], t["bwd_main"],
                                                                   t["dq_convert"])])
            r["bwd_ms"] = round(mb, 4)
            r["bwd_tflops"] = round(f_bwd / (mb * 1e-3) / 1e12, 2)
            r["bwd_pct_peak"] = round(r["bwd_tflops"] / pk["bf16_tflops"], 4)
            if eff is not None:
                r["bwd_tflops_effective"] = round(eff[1] / (mb * 1e-3) / 1e12, 2)
            if w.sparse:
                r["bwd_timing"] = "one fa_blocksparse_bwd call (preprocess, main, dQ convert)"
            elif w.dropout > 0 or w.layout != "bhnd":
                r["bwd_timing"] = "one fa_attention_bwd call (preprocess, main, dQ convert)"
            else:
                r["bwd_main_ms"] = round(statistics.median(t["bwd_main"]), 4)
        res[name] = r
        del st
        torch.cuda.empty_cache()
    return res


def run_reference(args, world, rank):
    """The CPU fp64 oracle, timed on the host cores as it stands."""
    if rank != 0:
        return None
    w = W.WORKLOADS[args.workload]
    budget = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, budget)
        if i >= args.warmup:
            vals.append(r)
    value = statistics.mean(v["value"] for v in vals)
    secs = sum(v["seconds"] for v in vals)
    return {
        "impl": "reference",
        "metric": "attention fwd/bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / len(vals) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {'causal' if w.causal else 'non-causal'} fwd+bwd, "
                               f"B={w.B} H={w.H} N={w.N} d={w.d}",
                   "sample": "each step is a bounded sample of whole heads"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": vals[-1]["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_n16384_noncausal", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed steps right before the timed ones (clock samples)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        out = run_ours(args, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
