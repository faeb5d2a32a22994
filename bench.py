"""Benchmark of the causal GQA flash-attention hot path on GB300.

Default run (one JSON line on stdout):
  * headline: prefill of 8192 tokens, 16 q heads / 2 kv heads, head_dim 256,
    fp32 KV cache, full causal. One step = fa_kv_append (K, V rows into the
    cache) + fa_prefill (fp16 staging + tensor-core kernel). value = causal
    attention TFLOP/s (4 * head_dim * n_q_heads * sum_p |S(p)| per step).
    The prefill steps (headline and prefill workloads) are captured once in a
    CUDA graph and replayed, one replay per timed step; the decode steps are
    timed as plain calls (replay measured 2-3% slower for them).
  * "workloads": the windowed prefill (sink 4, win 1024), the Q4_0-KV prefill
    (fp16 shadow of 4 sinks + 256 recent rows) and the multi-slot decode
    (32 slots x 32768 keys, Q4_0, 4 fp16 sinks, 256-key splits + combine),
    each with its own throughput and kernel roofline.
  * roofline: the dominant kernel's algorithmic work per launch over its
    CUDA-event duration, against MEASURED_PEAKS.json.
  * e2e: the same metric with host buffers: every step copies its q, k, v in
    from pinned host memory and its out back. value: the copies in, kernels
    and copy out of consecutive steps overlap on three streams (a serving
    loop); serial_value: each step's copies and kernels back to back.
  * cpu_baseline: the C oracle on a bounded sample, on this host's cores.

--impl reference times the oracle (the only reference this repository has)
on a bounded sample of the headline workload.
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

METRIC = "prefill attn TFLOP/s & decode KV GB/s at 1 GB300, % of roofline, oracle-exact"
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def visible_pairs(n, sink, win):
    """sum over queries p < n of |S(p)| (closed form of the attended-set size)."""
    p = np.arange(n, dtype=np.int64)
    if win <= 0:
        return int(np.sum(p + 1))
    lo = np.maximum(0, p - win + 1)
    recent = p - lo + 1
    sinks = np.minimum(sink, lo)          # sink keys below the window start
    return int(np.sum(recent + sinks))


def src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "causal_gqa_flash_attn_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, source_hash):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(kernel)
    if not e or e.get("source_hash") != source_hash:
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm = [float(s[0]) for s in self.samples if len(s) >= 7 and s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if len(s) >= 7 and s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples if len(s) >= 7
                          for i in range(4) if s[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# ------------------------------------------------- multi-rank (replicas)

def reduce_max_over_ranks(x, dist=None, device="cpu"):
    """Largest value of x over all ranks of the default process group (x
    itself when running alone). The job time is the slowest rank's time."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_rank, ms_max, world):
    """Whole-job throughput when every rank runs the same workload on its own
    GPU (replicas, weak scaling): all ranks' work over the slowest rank's time."""
    return world * work_per_rank / (ms_max * 1e-3)


# ------------------------------------------------------------ GPU arm

class GpuBench:
    def __init__(self, dev):
        import torch
        import causal_gqa_flash_attn_gb300 as fa
        self.torch, self.fa, self.dev = torch, fa, dev
        self.stream = torch.cuda.current_stream(dev)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_sink = torch.empty((), dtype=torch.float32, device=dev)
        self.launches = 0
        self.graph_steps = None  # True once a step was timed as graph replays
        self.graph_error = None

    def flush_l2(self):
        """Outside the timed region: write a 256 MB buffer (every line of the
        129 MB L2 replaced), then read another 256 MB buffer, so that the lines
        the write left dirty are written back here and the timed step starts
        with an L2 of clean lines that hold none of its data."""
        self.flush_buf.zero_()
        self.torch.sum(self.flush_read, dim=0, out=self.flush_sink)

    def timed_steps(self, step, warmup, steps, kernel_events=True, graph=False):
        """Run warmup + steps of `step`; each timed step between CUDA events on
        the launching stream, L2 flushed in between (outside the events).
        With graph, the step is captured once in a CUDA graph and each timed
        step is one replay (the same launches, without the host's launch gaps);
        if the capture fails the steps run as plain calls. Returns (step ms
        list, dominant-kernel ms list)."""
        torch, fa = self.torch, self.fa
        for _ in range(warmup):
            self.flush_l2()
            step()
        torch.cuda.synchronize(self.dev)
        if graph:
            try:
                out = self._timed_graph(step, steps, kernel_events)
                self.graph_steps = True
                return out
            except Exception as exc:  # a refused capture: time the plain calls
                self.graph_steps = False
                self.graph_error = str(exc)[:200]
                torch.cuda.synchronize(self.dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e in ev:  # create the underlying CUDA events
            for x in e:
                x.record(self.stream)
        torch.cuda.synchronize(self.dev)
        for s0, s1, k0, k1 in ev:
            self.flush_l2()
            if kernel_events:
                fa.set_kernel_events(k0, k1)
            s0.record(self.stream)
            step()
            s1.record(self.stream)
        fa.set_kernel_events(None, None)
        torch.cuda.synchronize(self.dev)
        st = fa.get_device_error()
        if st != fa.OK:
            raise RuntimeError(f"device error {fa.status_string(st)}")
        step_ms = [a.elapsed_time(b) for a, b, _, _ in ev]
        kern_ms = [a.elapsed_time(b) for _, _, a, b in ev] if kernel_events else []
        return step_ms, kern_ms

    def _timed_graph(self, step, steps, kernel_events):
        torch, fa = self.torch, self.fa
        s0, s1, k0, k1 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        for x in (s0, s1, k0, k1):  # create the underlying CUDA events
            x.record(self.stream)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        if kernel_events:  # recorded as event nodes on every replay
            fa.set_kernel_events(k0, k1)
        try:
            with torch.cuda.graph(g):
                step()
        finally:
            fa.set_kernel_events(None, None)
        g.replay()  # one untimed replay
        torch.cuda.synchronize(self.dev)
        step_ms, kern_ms = [], []
        for _ in range(steps):
            self.flush_l2()
            s0.record(self.stream)
            g.replay()
            s1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            step_ms.append(s0.elapsed_time(s1))
            if kernel_events:
                kern_ms.append(k0.elapsed_time(k1))
        st = fa.get_device_error()
        if st != fa.OK:
            raise RuntimeError(f"device error {fa.status_string(st)}")
        return step_ms, kern_ms

    # ---- prefill workloads
    def prefill_setup(self, w):
        torch, fa = self.torch, self.fa
        from workloads import FMT_CODES, prefill_inputs
        q, k, v = prefill_inputs(w.n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed)
        code = FMT_CODES[w.kv_fmt]
        S = dict(w=w, code=code, q_host=q, k_host=k, v_host=v)
        S["q"] = torch.from_numpy(q).to(self.dev)
        S["k"] = torch.from_numpy(k[None]).to(self.dev)
        S["v"] = torch.from_numpy(v[None]).to(self.dev)
        S["kp"] = fa.alloc_planes(1, code, w.n_kv_heads, w.n, w.head_dim, device=self.dev,
                                  scale=w.k_scale)
        S["vp"] = fa.alloc_planes(1, code, w.n_kv_heads, w.n, w.head_dim, device=self.dev,
                                  scale=w.v_scale)
        S["pos0"] = torch.zeros(1, dtype=torch.int32, device=self.dev)
        S["out"] = torch.empty((w.n, w.n_q_heads, w.head_dim), dtype=torch.float32,
                               device=self.dev)
        S["ws"] = torch.empty(fa.prefill_workspace_bytes(w.n, w.n_q_heads, w.n_kv_heads,
                                                         w.head_dim),
                              dtype=torch.uint8, device=self.dev)
        return S

    def prefill_step(self, S, q=None, k=None, v=None, out=None):
        fa, w = self.fa, S["w"]
        fa.kv_append(S["k"] if k is None else k, S["v"] if v is None else v, S["kp"], S["vp"],
                     S["pos0"], n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, max_seq=w.n,
                     kv_fmt=S["code"], shadow_sink=w.shadow_sink, shadow_win=w.shadow_win)
        fa.prefill(S["q"] if q is None else q, S["kp"], S["vp"], S["out"] if out is None else out,
                   w.n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.sink, w.win, S["code"],
                   max_seq=w.n, shadow_sink=w.shadow_sink, shadow_win=w.shadow_win,
                   workspace=S["ws"])

    def prefill_e2e(self, S, warmup, steps):
        """Same step from pinned host buffers: H2D of q, k, v and D2H of out
        inside the timed region (CUDA events on the same stream)."""
        torch = self.torch
        qh = torch.from_numpy(S["q_host"]).pin_memory()
        kh = torch.from_numpy(S["k_host"][None]).pin_memory()
        vh = torch.from_numpy(S["v_host"][None]).pin_memory()
        oh = torch.empty(S["out"].shape, dtype=torch.float32).pin_memory()
        qd, kd, vd = torch.empty_like(S["q"]), torch.empty_like(S["k"]), torch.empty_like(S["v"])
        od = torch.empty_like(S["out"])

        def step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            self.prefill_step(S, q=qd, k=kd, v=vd, out=od)
            oh.copy_(od, non_blocking=True)
        ms, _ = self.timed_steps(step, warmup, steps, kernel_events=False)
        h2d = qh.numel() * 4 + kh.numel() * 4 + vh.numel() * 4
        return ms, h2d, oh.numel() * 4

    def prefill_e2e_pipelined(self, S, warmup, steps):
        """The e2e step as a serving loop runs it. Every step still copies its
        own q, k, v from pinned host memory and its out back, but the copies in,
        the kernels and the copy out run on three streams with two sets of
        device buffers, so that step i+1's inputs and step i-1's output move
        while step i computes. Returns the mean ms per step: CUDA events around
        the whole run of `steps` steps, after `warmup` untimed ones."""
        torch = self.torch
        qh = torch.from_numpy(S["q_host"]).pin_memory()
        kh = torch.from_numpy(S["k_host"][None]).pin_memory()
        vh = torch.from_numpy(S["v_host"][None]).pin_memory()
        oh = torch.empty(S["out"].shape, dtype=torch.float32).pin_memory()
        sets = [(torch.empty_like(S["q"]), torch.empty_like(S["k"]), torch.empty_like(S["v"]),
                 torch.empty_like(S["out"])) for _ in range(2)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(self.dev) for _ in range(3))
        in_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def run(n):
            for i in range(n):
                b = i % 2
                qd, kd, vd, od = sets[b]
                with torch.cuda.stream(s_in):
                    if i >= 2:  # step i-2's kernels are done with this input set
                        s_in.wait_event(cmp_done[b])
                    qd.copy_(qh, non_blocking=True)
                    kd.copy_(kh, non_blocking=True)
                    vd.copy_(vh, non_blocking=True)
                    in_done[b].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(in_done[b])
                    if i >= 2:  # step i-2's output has left this buffer
                        s_cmp.wait_event(out_done[b])
                    self.prefill_step(S, q=qd, k=kd, v=vd, out=od)
                    cmp_done[b].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(cmp_done[b])
                    oh.copy_(od, non_blocking=True)
                    out_done[b].record(s_out)

        run(warmup)
        torch.cuda.synchronize(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        run(steps)
        e1.record(s_out)  # after the last copy out, which follows everything else
        torch.cuda.synchronize(self.dev)
        st = self.fa.get_device_error()
        if st != self.fa.OK:
            raise RuntimeError(f"device error {self.fa.status_string(st)}")
        return e0.elapsed_time(e1) / steps

    # ---- decode workload
    def decode_setup(self, w):
        torch, fa = self.torch, self.fa
        from workloads import FMT_CODES
        code = FMT_CODES[w.kv_fmt]
        L = w.n
        g = torch.Generator(device=self.dev)
        g.manual_seed(w.seed)
        S = dict(w=w, code=code, L=L)
        S["kp"] = fa.alloc_planes(w.nslots, code, w.n_kv_heads, L, w.head_dim, device=self.dev,
                                  scale=w.k_scale)
        S["vp"] = fa.alloc_planes(w.nslots, code, w.n_kv_heads, L, w.head_dim, device=self.dev,
                                  scale=w.v_scale)
        # cache rows 0..L-2 appended once (untimed), slot by slot chunks
        chunk = 4
        pos0 = torch.zeros(chunk, dtype=torch.int32, device=self.dev)
        pb = fa.kv_plane_bytes(code, w.n_kv_heads, L, w.head_dim)
        for u0 in range(0, w.nslots, chunk):
            k = torch.randn((chunk, L - 1, w.n_kv_heads, w.head_dim), generator=g,
                            device=self.dev)
            v = torch.randn((chunk, L - 1, w.n_kv_heads, w.head_dim), generator=g,
                            device=self.dev)
            fa.kv_append(k, v, S["kp"][u0 * pb:(u0 + chunk) * pb],
                         S["vp"][u0 * pb:(u0 + chunk) * pb], pos0, n_kv_heads=w.n_kv_heads,
                         head_dim=w.head_dim, max_seq=L, kv_fmt=code,
                         shadow_sink=w.shadow_sink, shadow_win=w.shadow_win)
            del k, v
        # the step's new token: row L-1 of every slot, and one query per slot
        S["k_new"] = torch.randn((w.nslots, 1, w.n_kv_heads, w.head_dim), generator=g,
                                 device=self.dev)
        S["v_new"] = torch.randn((w.nslots, 1, w.n_kv_heads, w.head_dim), generator=g,
                                 device=self.dev)
        S["q"] = torch.randn((w.nslots, w.n_q_heads, w.head_dim), generator=g, device=self.dev)
        S["pos"] = torch.full((w.nslots,), L - 1, dtype=torch.int32, device=self.dev)
        S["max_splits"] = -(-L // w.split_keys)
        S["ws"] = torch.empty(fa.decode_workspace_bytes(w.nslots, w.n_q_heads, w.head_dim,
                                                        S["max_splits"]),
                              dtype=torch.uint8, device=self.dev)
        S["out"] = torch.empty((w.nslots, w.n_q_heads, w.head_dim), dtype=torch.float32,
                               device=self.dev)
        torch.cuda.synchronize(self.dev)
        return S

    def decode_step(self, S):
        fa, w = self.fa, S["w"]
        fa.kv_append(S["k_new"], S["v_new"], S["kp"], S["vp"], S["pos"], n_kv_heads=w.n_kv_heads,
                     head_dim=w.head_dim, max_seq=S["L"], kv_fmt=S["code"],
                     shadow_sink=w.shadow_sink, shadow_win=w.shadow_win)
        fa.decode(S["q"], S["kp"], S["vp"], S["pos"], n_q_heads=w.n_q_heads,
                  n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, max_seq=S["L"], sink=w.sink,
                  win=w.win, kv_fmt=S["code"], shadow_sink=w.shadow_sink,
                  shadow_win=w.shadow_win, split_keys=w.split_keys,
                  max_splits=S["max_splits"], workspace=S["ws"])
        fa.decode_combine(S["ws"], S["out"], nslots=w.nslots, n_q_heads=w.n_q_heads,
                          head_dim=w.head_dim, max_splits=S["max_splits"])


def decode_kv_bytes(w):
    """KV bytes a decode step must read: per (slot, kv head) the fp16 sink
    rows (K and V, 2*hd bytes each) and the Q4_0 (fp32, fp16, fp8) rows of
    the rest."""
    L = w.n
    row = {"q4_0": w.head_dim // 32 * 18, "f32": w.head_dim * 4, "f16": w.head_dim * 2,
           "fp8_e4m3": w.head_dim}[w.kv_fmt]
    fp16_rows = min(w.shadow_sink, L) if w.kv_fmt == "q4_0" else 0
    if w.kv_fmt == "q4_0" and w.shadow_win > 0:
        fp16_rows = min(L, fp16_rows + w.shadow_win)
    per = fp16_rows * 2 * (2 * w.head_dim) + (L - fp16_rows) * 2 * row
    return w.nslots * w.n_kv_heads * per


def append_q4_bytes(w):
    """Bytes fa_kv_append must move to append all n rows of a Q4_0 workload:
    the fp32 K and V rows read, their Q4_0 blocks written, and the fp16
    mirrors of the shadow sink rows and of the ring's rows written."""
    rows = w.n * w.n_kv_heads
    read = 2 * rows * w.head_dim * 4
    body = 2 * rows * (w.head_dim // 32 * 18)
    mirrored = min(w.shadow_sink, w.n) + (min(256, w.n) if w.shadow_win > 0 else 0)
    shadows = 2 * w.n_kv_heads * mirrored * w.head_dim * 2
    return read + body + shadows


# ---------------------------------------------------------- CPU baseline

def oracle_prefill_sample(q, k, v, w, budget_s=12.0):
    """Time the C oracle on growing samples of query rows (all heads) until
    about budget_s of CPU work; returns (TFLOP/s, threads, description)."""
    from oracle import oracle
    kk = oracle.KVValues(k, w.kv_fmt)
    vv = oracle.KVValues(v, w.kv_fmt)
    rng = np.random.default_rng(1)
    rows_n = 4
    spent = 0.0
    flops = 0.0
    nrows = 0
    while spent < budget_s:
        rows = np.sort(rng.choice(w.n, rows_n, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attention(q[rows], rows, kk, vv, sink=w.sink, win=w.win,
                         shadow_sink=w.shadow_sink, shadow_win=w.shadow_win, L=w.n)
        dt = time.perf_counter() - t0
        spent += dt
        for p in rows:
            p = int(p)
            if w.win <= 0:
                cnt = p + 1
            else:
                lo = max(0, p - w.win + 1)
                cnt = (p - lo + 1) + min(w.sink, lo)
            flops += 4.0 * w.head_dim * w.n_q_heads * cnt
        nrows += rows_n
        if spent < budget_s / 4:
            rows_n *= 2
    return flops / spent / 1e12, oracle.num_threads(), \
        f"{nrows} random query rows x {w.n_q_heads} heads of {w.name}, {spent:.1f} s"


# ------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fa", choices=["fa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="run only this workload (name from workloads.py) for an ncu capture")
    ap.add_argument("--profile-slots", type=int, default=0,
                    help="with --profile: decode slots instead of the workload's")
    ap.add_argument("--profile-n", type=int, default=0,
                    help="with --profile: prefill tokens (or decode context) instead of the "
                         "workload's")
    ap.add_argument("--profile-window", default=None,
                    help="with --profile: 'sink,win' attended set instead of the workload's")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from workloads import BY_NAME
    headline = BY_NAME["prefill_f32_n8192_h16x2_d256"]
    flops_step = 4.0 * headline.head_dim * headline.n_q_heads * visible_pairs(
        headline.n, headline.sink, headline.win)

    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import build as ob
        ob.build()
        from workloads import prefill_inputs
        q, k, v = prefill_inputs(headline.n, headline.n_q_heads, headline.n_kv_heads,
                                 headline.head_dim, headline.seed)
        oracle_prefill_sample(q, k, v, headline, budget_s=0.5)   # warm-up, untimed
        vals = []
        for _ in range(args.steps):
            val, threads, desc = oracle_prefill_sample(q, k, v, headline,
                                                       budget_s=max(1.0, 90.0 / args.steps))
            vals.append(val)
        val = statistics.median(vals)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": headline.name},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    B = GpuBench(dev)
    peaks = load_peaks()

    if args.profile:
        import dataclasses
        w = BY_NAME[args.profile]
        w = dataclasses.replace(w, nslots=args.profile_slots or w.nslots,
                                n=args.profile_n or w.n)
        if args.profile_window:
            sk, wn = (int(x) for x in args.profile_window.split(","))
            w = dataclasses.replace(w, sink=sk, win=wn)
        S = B.decode_setup(w) if w.kind == "decode" else B.prefill_setup(w)
        fn = (lambda: B.decode_step(S)) if w.kind == "decode" else (lambda: B.prefill_step(S))
        sm, km = B.timed_steps(fn, args.warmup, args.steps)
        print(json.dumps({"profile": w.name, "ms_per_step": statistics.mean(sm),
                          "kernel_ms": statistics.mean(km)}))
        return

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    def max_over_ranks(x):
        return reduce_max_over_ranks(x, torch.distributed if world > 1 else None, dev)

    # ---------------- headline: prefill n=8192 fp32 KV, full causal
    S = B.prefill_setup(headline)
    barrier()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clk:
        step_ms, kern_ms = B.timed_steps(lambda: B.prefill_step(S), args.warmup, args.steps,
                                         graph=True)
    barrier()
    wall = time.perf_counter() - t_wall
    ms = max_over_ranks(statistics.mean(step_ms))
    value = job_throughput(flops_step, ms, world) / 1e12
    kms = statistics.mean(kern_ms)
    achieved = flops_step / (kms * 1e-3) / 1e12
    traffic = profiled_traffic("prefill_tc_kernel<256>", src_hash("prefill_tc.cu", "fa_device.cuh"))
    roofline = {"kernel": "prefill_tc_kernel<256>", "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 dense (fp16 has the same nominal rate), "
                               "burst", "kernel_ms": kms}
    e2e_ms, h2d, d2h = B.prefill_e2e(S, args.warmup, max(3, args.steps // 2))
    e2e_serial = job_throughput(flops_step, max_over_ranks(statistics.mean(e2e_ms)), world) / 1e12
    e2e_pipe_ms = max_over_ranks(B.prefill_e2e_pipelined(S, args.warmup, args.steps))
    e2e_val = job_throughput(flops_step, e2e_pipe_ms, world) / 1e12
    launches_per_step = 3  # append, stage Q, K and V, tensor-core kernel

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        val, threads, desc = oracle_prefill_sample(S["q_host"], S["k_host"], S["v_host"],
                                                   headline)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc}
    del S
    torch.cuda.empty_cache()

    # ---------------- other workloads
    extra = {}
    for name in ("prefill_f32_n8192_h16x2_d256_sink4_win1024",
                 "prefill_q4_n8192_h16x2_d256_shadow4_256",
                 "prefill_q4_n8192_h16x2_d256_shadow4_256_sink4_win1024",
                 "prefill_f16_n8192_h16x2_d256", "prefill_fp8_n8192_h16x2_d256"):
        w = BY_NAME[name]
        S = B.prefill_setup(w)
        f = 4.0 * w.head_dim * w.n_q_heads * visible_pairs(w.n, w.sink, w.win)
        sm, km = B.timed_steps(lambda: B.prefill_step(S), args.warmup, args.steps, graph=True)
        a = f / (statistics.mean(km) * 1e-3) / 1e12
        extra[name] = {"value": f / (statistics.mean(sm) * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "ms_per_step": statistics.mean(sm), "flop_per_step": f,
                       "launch": "graph replay" if B.graph_steps else "plain calls",
                       "roofline": {"kernel": "prefill_tc_kernel<256>", "bound": "tensor",
                                    "achieved": a, "peak": peaks["bf16_tflops"],
                                    "unit": "TFLOP/s", "frac": a / peaks["bf16_tflops"],
                                    "kernel_ms": statistics.mean(km)}}
        del S
        torch.cuda.empty_cache()
    # chunked prefill: the second half of the 8192-token sequence (queries at
    # positions 4096..8191) over the cache rows 0..8191; a step appends the
    # chunk's rows and runs fa_prefill_chunk
    w = BY_NAME["prefill_f32_n8192_h16x2_d256"]
    pos0 = w.n // 2
    nq = w.n - pos0
    S = B.prefill_setup(w)
    B.prefill_step(S)  # the context rows 0..pos0-1 (and the chunk's, rewritten each step)
    qc = S["q"][pos0:].contiguous()
    kc, vc = S["k"][:, pos0:].contiguous(), S["v"][:, pos0:].contiguous()
    p0c = torch.full((1,), pos0, dtype=torch.int32, device=dev)
    outc = torch.empty((nq, w.n_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    wsc = torch.empty(B.fa.prefill_chunk_workspace_bytes(pos0, nq, w.n_q_heads, w.n_kv_heads,
                                                         w.head_dim),
                      dtype=torch.uint8, device=dev)

    def chunk_step():
        B.fa.kv_append(kc, vc, S["kp"], S["vp"], p0c, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_seq=w.n, kv_fmt=S["code"])
        B.fa.prefill_chunk(qc, S["kp"], S["vp"], outc, pos0, nq, w.n_q_heads, w.n_kv_heads,
                           w.head_dim, w.sink, w.win, S["code"], max_seq=w.n, workspace=wsc)
    f = 4.0 * w.head_dim * w.n_q_heads * (visible_pairs(w.n, w.sink, w.win)
                                          - visible_pairs(pos0, w.sink, w.win))
    sm, km = B.timed_steps(chunk_step, args.warmup, args.steps, graph=True)
    a = f / (statistics.mean(km) * 1e-3) / 1e12
    extra["prefill_chunk_f32_pos4096_n4096_h16x2_d256"] = {
        "value": f / (statistics.mean(sm) * 1e-3) / 1e12, "unit": "TFLOP/s",
        "ms_per_step": statistics.mean(sm), "flop_per_step": f,
        "step": "kv_append of the chunk + fa_prefill_chunk",
        "launch": "graph replay" if B.graph_steps else "plain calls",
        "roofline": {"kernel": "prefill_tc_kernel<256>", "bound": "tensor", "achieved": a,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": a / peaks["bf16_tflops"], "kernel_ms": statistics.mean(km)}}
    del S, qc, kc, vc, outc, wsc
    torch.cuda.empty_cache()

    decode_names = () if args.no_decode else (
        "decode_q4_32slots_L32768_h16x2_d256_sink4", "decode_f16_32slots_L32768_h16x2_d256_sink4",
        "decode_fp8_32slots_L32768_h16x2_d256_sink4")
    for name in decode_names:
        w = BY_NAME[name]
        kname = {"q4_0": "decode_q4_kernel<256>", "f16": "decode_dense_kernel<256,f16>",
                 "fp8_e4m3": "decode_dense_kernel<256,fp8>"}[w.kv_fmt]
        srcs = (("decode.cu", "decode_common.cuh") if w.kv_fmt == "q4_0"
                else ("decode_dense.cu",)) + ("fa_device.cuh",)
        S = B.decode_setup(w)
        kvb = decode_kv_bytes(w)
        sm, km = B.timed_steps(lambda: B.decode_step(S), args.warmup, args.steps)
        a = kvb / (statistics.mean(km) * 1e-3) / 1e9
        extra[w.name] = {"value": kvb / (statistics.mean(sm) * 1e-3) / 1e9, "unit": "GB/s",
                         "ms_per_step": statistics.mean(sm), "kv_bytes_per_step": kvb,
                         "step": "append 1 row/slot + split decode + combine",
                         "launch": "plain calls",
                         "roofline": {"kernel": kname, "bound": "hbm",
                                      "achieved": a, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": a / peaks["hbm_gbs"], "frac_of_8tbs": a / 8000.0,
                                      "traffic": profiled_traffic(
                                          kname, src_hash(*srcs)),
                                      "kernel_ms": statistics.mean(km)}}
        del S
        torch.cuda.empty_cache()

    # Q4_0 append alone: 8192 new rows x 2 kv heads x head_dim 256 of K and V
    # quantised into Q4_0 blocks, with the fp16 mirrors of the 4 sink rows and
    # of the 256 newest rows (the Q4_0 prefill workload's cache)
    w = BY_NAME["prefill_q4_n8192_h16x2_d256_shadow4_256"]
    S = B.prefill_setup(w)
    abytes = append_q4_bytes(w)

    def append_step():
        B.fa.kv_append(S["k"], S["v"], S["kp"], S["vp"], S["pos0"], n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_seq=w.n, kv_fmt=S["code"],
                       shadow_sink=w.shadow_sink, shadow_win=w.shadow_win)
    sm, _ = B.timed_steps(append_step, args.warmup, args.steps, kernel_events=False)
    a = abytes / (statistics.mean(sm) * 1e-3) / 1e9
    extra["append_q4_n8192_h2_d256_shadow4_256"] = {
        "value": a, "unit": "GB/s", "ms_per_step": statistics.mean(sm),
        "bytes_per_step": abytes, "step": "fa_kv_append (one launch)",
        "roofline": {"kernel": "kv_append_q4_kernel<256>", "bound": "hbm", "achieved": a,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": a / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("kv_append_q4_kernel<256>",
                                                 src_hash("kv_append.cu", "fa_device.cuh")),
                     "kernel_ms": statistics.mean(sm)}}
    del S
    torch.cuda.empty_cache()

    if not args.no_decode:
        # merge of two attention states (fp32 outputs [T][H][D], lses [H][T]):
        # the context-chunk + new-tokens combination of chunked prefill
        T, H, D = 8192, 16, 256
        g = torch.Generator(device=dev).manual_seed(20261202)
        po = torch.randn(T, H, D, device=dev, generator=g)
        so = torch.randn(T, H, D, device=dev, generator=g)
        pl = torch.randn(H, T, device=dev, generator=g) * 4
        sl = torch.randn(H, T, device=dev, generator=g) * 4
        mo = torch.empty_like(po)
        ml = torch.empty_like(pl)
        mbytes = 3 * T * H * D * 4 + 3 * H * T * 4
        sm, _ = B.timed_steps(lambda: B.fa.merge_attn_states(mo, ml, po, pl, so, sl),
                              args.warmup, args.steps, kernel_events=False)
        a = mbytes / (statistics.mean(sm) * 1e-3) / 1e9
        extra["merge_attn_states_t8192_h16_d256"] = {
            "value": a, "unit": "GB/s", "ms_per_step": statistics.mean(sm),
            "bytes_per_step": mbytes, "step": "fa_merge_attn_states",
            "roofline": {"kernel": "merge_attn_states_kernel", "bound": "hbm", "achieved": a,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": a / peaks["hbm_gbs"],
                         "kernel_ms": statistics.mean(sm)}}
        del po, so, pl, sl, mo, ml
        torch.cuda.empty_cache()

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": headline.name, "n": headline.n,
                       "n_q_heads": headline.n_q_heads, "n_kv_heads": headline.n_kv_heads,
                       "head_dim": headline.head_dim, "sink": headline.sink, "win": headline.win,
                       "kv_fmt": headline.kv_fmt, "flop_per_step": flops_step,
                       "step": "kv_append + prefill", "l2": "flushed between steps: 256 MB written, then another 256 MB read "
                             "(the flush's dirty lines are written back before the step)",
                       "launch": ("the step captured once in a CUDA graph, each timed step one "
                                  "replay" if B.graph_steps else
                                  f"plain calls (graph capture failed: {B.graph_error})"),
                       "parallelism": "replicas" if world > 1 else "1 GPU"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_pipe_ms,
                    "mode": "pipelined: copies in, kernels and copy out of consecutive steps "
                            "on three streams, two device buffer sets; no L2 flush (a step "
                            f"moves {(h2d + d2h) / 1e6:.0f} MB, more than the 129 MB L2)",
                    "serial_value": e2e_serial,
                    "serial_ms_per_step": max_over_ranks(statistics.mean(e2e_ms))},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "wall_s_timed": wall,
            "workloads": extra,
            "workload_fracs": {k: {"value": round(v["value"], 1), "unit": v["unit"],
                                   "kernel": v["roofline"]["kernel"],
                                   "frac": round(v["roofline"]["frac"], 3)}
                               for k, v in extra.items()},
        }))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
