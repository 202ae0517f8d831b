"""Benchmark of the attention hot path on GB300: one JSON line on rank 0.

Headline workload (the decode configuration): 12 query heads over 2 KV heads,
head_dim 128, a 4096-row cache, no window.  One step = append of the new
K/V row at position total_seq-1 and decode over all 4096 rows
(attn_decode_append: the decode kernel with the append fused, and its
combine kernel).
Metric value = algorithmic K+V bytes (2 * kv_heads * total_seq * head_dim * 4)
per step x steps / device time, in GB/s.  The caches rotate over enough
replicas that every step reads them cold from HBM (the replicas together
exceed twice the 129 MB L2).  Steps run as CUDA-graph replays so that host
launch overhead does not bound a 5-microsecond step.

The same line ends with one compact object per named workload, cfg1 ... cfg5
(the 64-token exact prefill, this decode call alone, the 2048-token
tensor-core prefill, the windowed 32768-row decode after an append, the
16384-token tensor-core prefill): value, unit, time per call, fraction of the
roofline peak, max abs error against the fp64 oracle, and for the prefills
the end-to-end figure.  Before them: the roofline of the dominant decode
kernel, an end-to-end number through the Python API with host buffers, the
fp64 CPU oracle timed on the host cores, the SM clocks sampled during the
timed region, the full-cache decode and the 28-layer prefill stack.

--impl reference times the oracle (the plain CPU definition) on the host
cores instead, on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "decode KV GB/s and causal prefill TFLOP/s vs GB300 roofline (1 GPU)"
L2_BYTES = 129 * 1024 * 1024
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "attention_attn_prefill_causal_gb300", "csrc")


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def aggregate(per_rank_seconds: float, per_rank_units: float, ws: int):
    """Whole-job throughput: units of all ranks / max seconds over ranks."""
    if ws > 1:
        t = torch.tensor([per_rank_seconds], dtype=torch.float64)
        u = torch.tensor([per_rank_units], dtype=torch.float64)
        if torch.distributed.get_backend() == "nccl":
            t, u = t.cuda(), u.cuda()
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
        return float(t.item()), float(u.item())
    return per_rank_seconds, per_rank_units


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def code_text(src: str) -> str:
    """CUDA/C++ source without comments and blank space, so that an edit of
    comments alone keeps the hash of the code."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, files):
    """DRAM bytes per launch from a committed ncu capture, only while the
    kernel's sources are unchanged since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not t or t.get("source_sha") != source_sha(files):
        return None
    return t.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling (200 ms) in a background process; keeps the
    samples whose timestamps fall inside [t0, t1] (host clock)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def pump():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=pump, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 - 0.25 <= ts <= t1 + 0.25]
        if not inside and rows:  # timed region shorter than one sample period
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))[1]]
        if not inside:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[6:10]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": num(inside[0][3]),
                "reasons": sorted(reasons), "samples": len(inside)}


def lead_in():
    """Keep the GPU busy for about half a millisecond on the current stream
    before a device-timed region starts.  Without it the start event runs
    on an idle GPU at once and the region then waits for the host to submit
    its first graph launch, a fixed cost that short runs spread over few
    steps (about 35 us at 20 steps).  The spin runs before the start event,
    so the region still holds exactly the timed steps."""
    torch.cuda._sleep(1_000_000)  # clock cycles: about 0.5 ms at 2 GHz


def make_graph(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # make sure lazily created state exists before capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


# ---------------------------------------------------------------- decode (headline)

class DecodeBench:
    def __init__(self, attn, shape, device):
        self.attn, self.c, self.dev = attn, shape, device
        q, kc, vc, kn, vn = workloads.decode_inputs(shape.num_heads, shape.kv_heads,
                                                    shape.head_dim, shape.max_seq, shape.seed,
                                                    append=True)
        self.host = (q, kc, vc, kn, vn)
        # replicas so that the live K/V bytes of R consecutive steps exceed 2x L2
        self.R = max(2, math.ceil(2 * L2_BYTES / shape.kv_bytes_algorithmic()))
        self.kc = [kc.to(device) for _ in range(self.R)]
        self.vc = [vc.to(device) for _ in range(self.R)]
        # The per-step inputs q, k_new, v_new live in one device buffer (three
        # 16-byte aligned views), so a step's host-to-device input is one copy.
        nq, nk = q.numel(), kn.numel()
        self.io = torch.cat([q.reshape(-1), kn.reshape(-1), vn.reshape(-1)]).to(device)
        self.q = self.io[:nq].view_as(q)
        self.kn = self.io[nq:nq + nk].view_as(kn)
        self.vn = self.io[nq + nk:].view_as(vn)
        self.out = torch.empty(shape.num_heads, shape.head_dim, device=device)
        ws = attn.attn_decode_workspace_size(shape.num_heads, shape.kv_heads, shape.head_dim,
                                             shape.total_seq, shape.window)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.ws_bytes = ws
        self.pos = shape.total_seq - 1
        self.launches_per_step = 2  # fused append + decode kernel, PDL combine kernel

    def step(self, i, stream, append=True, bufs=None):
        """One step on replica i % R.  ``bufs`` = (q, k_new, v_new, out) to
        use instead of the device buffers (e.g. page-locked host buffers)."""
        c, a = self.c, self.attn
        r = i % self.R
        q, kn, vn, out = bufs if bufs is not None else (self.q, self.kn, self.vn, self.out)
        if append:
            a.attn_decode_append(q, kn, vn, self.kc[r], self.vc[r], out,
                                 c.num_heads, c.kv_heads, c.head_dim, c.max_seq, c.total_seq,
                                 self.pos, window=c.window, workspace=self.ws,
                                 workspace_bytes=self.ws_bytes, stream=stream)
        else:
            a.attn_decode(q, self.kc[r], self.vc[r], out, c.num_heads, c.kv_heads,
                          c.head_dim, c.max_seq, c.total_seq, window=c.window,
                          workspace=self.ws, workspace_bytes=self.ws_bytes, stream=stream)

    def graphs(self, stream, append=True):
        def chunk():
            for i in range(self.R):
                self.step(i, stream, append)
        return make_graph(chunk, stream)

    def check(self):
        """Untimed parity check of what the bench times (replica 0)."""
        import oracle
        c = self.c
        q, kc, vc, kn, vn = self.host
        kh, vh = kc.numpy().copy(), vc.numpy().copy()
        oracle.kv_append(kn.numpy(), vn.numpy(), kh, vh, c.kv_heads, c.head_dim, c.max_seq,
                         self.pos)
        ref = oracle.decode(q.numpy(), kh, vh, c.num_heads, c.kv_heads, c.head_dim, c.max_seq,
                            c.total_seq, c.window)
        s = torch.cuda.current_stream()
        self.step(0, s)
        torch.cuda.synchronize()
        return float(np.abs(self.out.cpu().numpy() - ref).max())


def run_graph_steps(graph, steps_per_graph, rem_graph, steps):
    """Replay graphs to execute exactly `steps` steps."""
    full, rem = divmod(steps, steps_per_graph)
    for _ in range(full):
        graph.replay()
    if rem:
        rem_graph[rem].replay()


def time_steps(graph, R, rem_graphs, steps, stream):
    # A graph of the last steps % R steps is captured on first use: capture
    # it (and run it once) before the timed region starts.
    if steps % R:
        rem_graphs[steps % R]
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        lead_in()
        start.record(stream)
        run_graph_steps(graph, R, rem_graphs, steps)
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


class RemainderGraphs(dict):
    """Graphs of n < R steps, captured on first use."""

    def __init__(self, bench, stream, append=True):
        super().__init__()
        self.bench, self.stream, self.append = bench, stream, append

    def __missing__(self, n):
        def f():
            for i in range(n):
                self.bench.step(i, self.stream, self.append)
        g = make_graph(f, self.stream)
        self[n] = g
        return g


def remainder_graphs(bench, stream, append=True):
    return RemainderGraphs(bench, stream, append)


# ---------------------------------------------------------------- prefill (companion)

# Dense tensor peaks relative to the 16-bit one (nominal GB300 figures:
# 2.25 PFLOP/s fp16/bf16, 1.1 PFLOP/s tf32); the measured bf16 peak is
# scaled by this ratio for the TF32 mode.
TF32_PEAK_RATIO = 1.1 / 2.25


def prefill_uses_pairs(m, num_q_heads, sms, tf32=False):
    """The library's kernel choice: 16-bit calls whose query-tile pairs fill
    the SMs twice over run the pair kernel (a work item is two 128-row query
    tiles), the others and every TF32 call the single-tile kernel."""
    return not tf32 and -(-m // 256) * num_q_heads >= 2 * sms


def prefill_kernel(m, num_q_heads, sms, tf32=False):
    """(name, source files) of the main kernel of a tensor-core prefill call."""
    if prefill_uses_pairs(m, num_q_heads, sms, tf32):
        return "prefill_pair_kernel", ["prefill_tc_pair.cu", "prefill_tc_common.cuh", "sm103_ptx.cuh"]
    return "prefill_tc_kernel", ["prefill_tc.cu", "prefill_tc_common.cuh", "sm103_ptx.cuh"]


def prefill_launches(m, num_q_heads, sms, tf32=False):
    """Kernels one tensor-core prefill call launches: the rounding pre-pass
    and the main kernel, plus the combine kernel when the call splits its key
    walk.  Mirrors the library's plan: the key walk is split only when work
    items x heads leave SMs idle, with the smallest chunk whose items fit in
    one wave."""
    n_qt = -(-m // 128)
    tiles_per_item = 2 if prefill_uses_pairs(m, num_q_heads, sms, tf32) else 1
    n_units = -(-m // (128 * tiles_per_item))

    def nk(u):
        return min(tiles_per_item * u + tiles_per_item, n_qt)
    if n_units == 0 or n_units * num_q_heads >= sms:
        return 2
    nk_last = nk(n_units - 1)
    for c in range(2, nk_last):
        if sum(-(-nk(u) // c) for u in range(n_units)) * num_q_heads <= sms:
            return 3
    return 2
    nk_last = nk(n_units - 1)
    for c in range(2, nk_last):
        if sum(-(-nk(u) // c) for u in range(n_units)) * num_q_heads <= sms:
            return 3
    return 2


class PrefillBench:
    def __init__(self, attn, shape, device, precision=None):
        self.attn, self.c, self.dev = attn, shape, device
        self.prec = attn.ATTN_PREC_FP16 if precision is None else precision
        q, k, v = workloads.shape_inputs(shape)
        self.host = (q, k, v)
        in_bytes = (q.numel() + k.numel() + v.numel() + q.numel()) * 4
        self.R = 1 if in_bytes > 2 * L2_BYTES else max(2, math.ceil(2 * L2_BYTES / in_bytes))
        self.q = [q.to(device) for _ in range(self.R)]
        self.k = [k.to(device) for _ in range(self.R)]
        self.v = [v.to(device) for _ in range(self.R)]
        self.o = [torch.empty_like(self.q[0]) for _ in range(self.R)]
        ws = attn.attn_prefill_workspace_size(shape.m, shape.num_q_heads, shape.num_kv_heads,
                                              shape.head_dim, self.prec)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        # The workspace holds the rounded K and V (two 256-byte aligned
        # matrices of 2 bytes per element, 4 in the TF32 mode) and, when the
        # call splits its key walk, the partials that a third kernel merges.
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.launches_per_call = prefill_launches(
            shape.m, shape.num_q_heads, sms, self.prec == attn.ATTN_PREC_TF32)

    def call(self, i, stream):
        c, a, r = self.c, self.attn, i % self.R
        a.attn_prefill_causal(self.q[r], self.k[r], self.v[r], self.o[r], c.m, c.num_q_heads,
                              c.num_kv_heads, c.head_dim, c.q_stride, c.kv_stride,
                              precision=self.prec, workspace=self.ws, stream=stream)

    def check(self):
        import oracle
        c = self.c
        q, k, v = self.host
        # every row of a short prompt; a seeded sample of rows of a long one
        # (the full comparison of the long prompt is a GPU test of its own)
        rows = None if c.m <= 4096 else workloads.sample_rows(c.m, c.seed, 16, 16, 32)
        t0 = time.perf_counter()
        ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), c.m, c.num_q_heads,
                                    c.num_kv_heads, c.head_dim, c.q_stride, c.kv_stride, rows=rows)
        secs = time.perf_counter() - t0
        # the oracle's own rate on the host cores: row i attends i + 1 keys,
        # 4 * head_dim FLOP per key and query head (scores and P.V)
        keys = c.m * (c.m + 1) // 2 if rows is None else int(sum(int(r) + 1 for r in rows))
        self.oracle_tflops = 4.0 * c.head_dim * c.num_q_heads * keys / secs / 1e12
        self.oracle_rows = c.m if rows is None else len(rows)
        self.oracle_cores = oracle.max_threads()
        self.call(0, torch.cuda.current_stream())
        torch.cuda.synchronize()
        got = self.o[0].view(c.m, c.q_stride)[:, : c.num_q_heads * c.head_dim]
        got = got.cpu().numpy().reshape(c.m, c.num_q_heads, c.head_dim)
        if rows is not None:
            got = got[rows]
        return float(np.abs(got - ref).max())


def time_prefill_calls(pb, stream, calls):
    """Device seconds per call of a prefill workload: CUDA-graph replays of
    one call per input replica (after two warm-up replays), CUDA events on
    the launching stream.  Returns (seconds per call, calls, total seconds)."""
    def chunk():
        for i in range(pb.R):
            pb.call(i, stream)
    g = make_graph(chunk, stream)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(calls / pb.R))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        lead_in()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    end.synchronize()
    secs = start.elapsed_time(end) / 1e3
    n = reps * pb.R
    return secs / n, n, secs


def bench_prefill_tf32(attn, shape, device, stream, calls, peaks, peak_src):
    """The TF32 mode on a prefill workload: device time per call and its
    fraction of the TF32 dense peak (no end-to-end leg)."""
    pb = PrefillBench(attn, shape, device, attn.ATTN_PREC_TF32)
    err = pb.check()
    per_call, _, secs = time_prefill_calls(pb, stream, calls)
    tflops = shape.flops() / per_call / 1e12
    peak_key = "bf16_tflops_sustained" if secs > 1.0 else "bf16_tflops"
    peak = float(peaks[peak_key]) * TF32_PEAK_RATIO
    return {"value": round(tflops, 2), "unit": "TFLOP/s", "us": round(per_call * 1e6, 2),
            "frac": round(tflops / peak, 4), "peak": round(peak, 1), "err": float(f"{err:.3g}"),
            "launches": pb.launches_per_call}


def bench_prefill(attn, shape, device, stream, calls, peaks, peak_src):
    pb = PrefillBench(attn, shape, device)
    err = pb.check()
    per_call, n, secs = time_prefill_calls(pb, stream, calls)
    flops = shape.flops()
    tflops = flops / per_call / 1e12
    peak_key = "bf16_tflops_sustained" if secs > 1.0 else "bf16_tflops"
    peak = float(peaks[peak_key])
    kname, kfiles = prefill_kernel(shape.m, shape.num_q_heads,
                                   torch.cuda.get_device_properties(device).multi_processor_count)
    traffic = traffic_for(f"{kname}:{shape.name}", kfiles)

    # End to end through the Python API with page-locked host buffers: every
    # call's Q, K, V come from host memory (H2D copies) and its O goes back
    # (D2H copy).  Two schedules of the same calls:
    #  * pipelined (`value`): a stream of independent prompts, double-buffered
    #    device buffers; call n+1's H2D, call n's kernels and call n-1's D2H
    #    run on three streams;
    #  * serial: H2D, call and D2H one after another on one stream.
    q, k, v = pb.host
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = [torch.empty_like(hq).pin_memory() for _ in range(2)]
    c = shape
    sets = [(pb.q[0], pb.k[0], pb.v[0], pb.o[0])]
    if pb.R > 1:
        sets.append((pb.q[1], pb.k[1], pb.v[1], pb.o[1]))
    else:
        sets.append((torch.empty_like(pb.q[0]), torch.empty_like(pb.k[0]),
                     torch.empty_like(pb.v[0]), torch.empty_like(pb.o[0])))

    def call_on(b):
        dq, dk, dv, do = sets[b]
        attn.attn_prefill_causal(dq, dk, dv, do, c.m, c.num_q_heads, c.num_kv_heads,
                                 c.head_dim, c.q_stride, c.kv_stride,
                                 precision=attn.ATTN_PREC_FP16, workspace=pb.ws, stream=stream)

    def serial(n):
        with torch.cuda.stream(stream):
            for _ in range(n):
                dq, dk, dv, do = sets[0]
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                call_on(0)
                ho[0].copy_(do, non_blocking=True)

    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        for i in range(n):
            b = i % 2
            dq, dk, dv, do = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[b])  # call i-2 no longer reads set b
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # call i-2's output has left set b
            call_on(b)
            ev_cmp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                ho[b].copy_(do, non_blocking=True)
                ev_out[b].record(s_out)

    def timed(fn, n, first, last):
        fn(2)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(first)
        fn(n)
        t1.record(last)
        t1.synchronize()
        return t0.elapsed_time(t1) / 1e3 / n

    # enough calls that filling and draining the three-stage pipeline (both
    # included in the timed region) is a small part of the total
    e_calls = 24 if c.m > 4096 else 120
    serial_per_call = timed(serial, e_calls, stream, stream)
    # s_in waits on the compute stream once before the first copy, so the
    # start event on the compute stream precedes every copy of the run
    s_in.wait_stream(stream)
    pipe_per_call = timed(pipelined, e_calls, s_in, s_out)
    torch.cuda.synchronize()
    got = ho[(e_calls - 1) % 2].view(c.m, c.q_stride)[:, : c.num_q_heads * c.head_dim]
    ref = pb.o[0].view(c.m, c.q_stride)[:, : c.num_q_heads * c.head_dim].cpu()
    if not torch.equal(got, ref):
        raise SystemExit("pipelined prefill output differs from the device-buffer one")
    e2e_per_call = pipe_per_call
    h2d = (q.numel() + k.numel() + v.numel()) * 4
    d2h = q.numel() * 4
    compact = {"value": round(tflops, 2), "unit": "TFLOP/s", "us": round(per_call * 1e6, 2),
               "frac": round(tflops / peak, 4), "err": float(f"{err:.3g}"),
               "e2e": round(flops / e2e_per_call / 1e12, 2),
               "cpu": float(f"{pb.oracle_tflops:.3g}"), "traffic": traffic,
               "launches": pb.launches_per_call}
    detail = {"workload": shape.name, "calls": n, "flops_per_call": flops,
              "peak": peak, "peak_source": f"{peak_key} ({peak_src})", "kernel": kname,
              "traffic": traffic,
              "l2": (f"inputs {pb.R} rotating replicas" if pb.R > 1 else "inputs larger than 2x L2"),
              "e2e_pipelined_ms": round(e2e_per_call * 1e3, 4),
              "e2e_serial_ms": round(serial_per_call * 1e3, 4),
              "e2e_calls": e_calls, "h2d_bytes_per_call": h2d, "d2h_bytes_per_call": d2h,
              "cpu_oracle": {"tflops": pb.oracle_tflops, "rows": pb.oracle_rows,
                             "cores": pb.oracle_cores}}
    return compact, detail


# ---------------------------------------------------------------- copy floor (context)

def copy_floor_us(replicas, traffic_bytes, stream, reps=50):
    """Device time of a torch copy that moves the same number of DRAM bytes
    as one decode call reads (half read, half written), rotating over the
    cache replicas so that every copy reads cold, as CUDA-graph replays.
    The measured HBM peak is this same copy at 1 Gi elements; at a decode's
    size the copy shows what launch latency and ramp-up leave of it."""
    n = traffic_bytes // 8  # floats read (= floats written)
    srcs = [r.reshape(-1)[:n] for r in replicas]
    dst = torch.empty(n, dtype=torch.float32, device=srcs[0].device)

    def run():
        for s in srcs:
            dst.copy_(s)
    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    g = make_graph(run, stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        lead_in()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(srcs))


# ---------------------------------------------------------------- companion workloads

def bench_decode_companion(attn, shape, device, stream, steps, peaks, peak_src):
    """A decode after an append (32 query heads over 8 KV heads, a
    32768-row cache, window 4096 or none): one step = attn_decode_append at
    total_seq-1.  L2-cold through cache replicas sized by the live bytes."""
    db = DecodeBench(attn, shape, device)
    err = db.check()
    g = db.graphs(stream)
    rem = remainder_graphs(db, stream)
    time_steps(g, db.R, rem, 3 * db.R, stream)
    n = max(steps, 8 * db.R)
    secs = time_steps(g, db.R, rem, n, stream)
    per = secs / n
    live = shape.kv_bytes_algorithmic()
    hbm = float(peaks["hbm_gbs"])
    gbs = live / per / 1e9
    traffic = traffic_for(f"attn_decode:{shape.name}", ["decode.cu"])
    compact = {"value": round(gbs, 2), "unit": "GB/s", "us": round(per * 1e6, 3),
               "frac": round(gbs / hbm, 4), "err": float(f"{err:.3g}"), "traffic": traffic}
    if shape.window:
        compact["copy_floor_us"] = round(copy_floor_us(db.kc, live, stream), 3)
        # the same time over the formula's byte count (all total_seq rows,
        # which the kernel does not read: rows below the window are skipped)
        compact["gbs_all_rows_formula"] = round(shape.kv_bytes_all_rows() / per / 1e9, 2)
    detail = {"workload": shape.name, "steps": n, "bytes_per_step": live,
              "bytes_all_rows": shape.kv_bytes_all_rows(),
              "gbs_all_rows_formula": round(shape.kv_bytes_all_rows() / per / 1e9, 2),
              "l2": f"{db.R} rotating cache replicas (live bytes {db.R * live // 2**20} MiB)",
              "traffic": traffic,
              "peak_source": f"hbm_gbs ({peak_src})", "launches_per_step": db.launches_per_step}
    return compact, detail


def fp32_peak_tflops(sm_count, clock_mhz):
    """FP32 CUDA-core peak: SMs x 128 FMA lanes x 2 FLOP x clock."""
    return sm_count * 128 * 2 * clock_mhz * 1e6 / 1e12


def bench_prefill_fp32_small(attn, shape, device, stream, calls, peaks):
    """The small exact-mode prefill (64 tokens, 4 query heads over 2 KV heads,
    head_dim 32) on the fp32 CUDA-core kernel.  Latency-bound: the inputs are
    98 KB and stay in L2; timed as CUDA-graph replays of back-to-back calls."""
    import oracle
    q, k, v = workloads.shape_inputs(shape)
    dq, dk, dv = q.to(device), k.to(device), v.to(device)
    o = torch.empty_like(dq)
    c = shape

    def call():
        attn.attn_prefill_causal(dq, dk, dv, o, c.m, c.num_q_heads, c.num_kv_heads, c.head_dim,
                                 c.q_stride, c.kv_stride, precision=attn.ATTN_PREC_FP32,
                                 stream=stream)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    ref = oracle.prefill_causal(q.numpy(), k.numpy(), v.numpy(), c.m, c.num_q_heads,
                                c.num_kv_heads, c.head_dim, c.q_stride, c.kv_stride)
    got = o.view(c.m, c.q_stride)[:, : c.num_q_heads * c.head_dim].cpu().numpy()
    err = float(np.abs(got.reshape(c.m, c.num_q_heads, c.head_dim) - ref).max())

    def batch():
        for _ in range(32):
            call()
    g = make_graph(batch, stream)
    reps = max(1, calls // 32)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        lead_in()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    per = e0.elapsed_time(e1) / 1e3 / (reps * 32)
    tf = shape.flops() / per / 1e12
    props = torch.cuda.get_device_properties(device)
    peak = fp32_peak_tflops(props.multi_processor_count, float(peaks.get("sm_max_mhz", 2070.0)))
    rel = err / float(np.abs(ref).max())
    return {"value": round(tf, 4), "unit": "TFLOP/s", "us": round(per * 1e6, 3),
            "frac": round(tf / peak, 5), "err": float(f"{err:.3g}"), "rel": float(f"{rel:.3g}")}


# ---------------------------------------------------------------- layer stack (launch cost)

def bench_layer_stack(attn, shape, device, stream, layers=28, reps=5):
    """A prefill pass over an L-layer stack (the pages' 28-layer model
    context): every layer runs attn_prefill_causal on its own Q/K/V.
    Timed as eager launches from Python and as one CUDA-graph replay; the
    difference is the host launch cost a graph removes."""
    q, k, v = workloads.shape_inputs(shape)
    qs = [q.to(device) for _ in range(layers)]
    ks = [k.to(device) for _ in range(layers)]
    vs = [v.to(device) for _ in range(layers)]
    os_ = [torch.empty_like(qs[0]) for _ in range(layers)]
    ws = torch.empty(attn.attn_prefill_workspace_size(shape.m, shape.num_q_heads,
                                                      shape.num_kv_heads, shape.head_dim),
                     dtype=torch.uint8, device=device)
    c = shape

    def one_pass():
        for i in range(layers):
            attn.attn_prefill_causal(qs[i], ks[i], vs[i], os_[i], c.m, c.num_q_heads,
                                     c.num_kv_heads, c.head_dim, c.q_stride, c.kv_stride,
                                     workspace=ws, stream=stream)

    def timed(fn):
        """(device ms per pass, host ms to issue one pass)."""
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            lead_in()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        t1 = time.perf_counter()
        e1.synchronize()
        return e0.elapsed_time(e1) / reps, (t1 - t0) * 1e3 / reps
    eager_ms, eager_issue_ms = timed(one_pass)
    g = make_graph(one_pass, stream)
    graph_ms, _ = timed(g.replay)
    return {"eager_ms": round(eager_ms, 4), "graph_ms": round(graph_ms, 4),
            "eager_issue_ms": round(eager_issue_ms, 4)}


# ---------------------------------------------------------------- CPU oracle timing

def cpu_baseline_decode(shape, budget_s=10.0, max_steps=2000):
    import oracle
    q, kc, vc, kn, vn = workloads.decode_inputs(shape.num_heads, shape.kv_heads, shape.head_dim,
                                                shape.max_seq, shape.seed, append=True)
    q, kh, vh, kn, vn = q.numpy(), kc.numpy().copy(), vc.numpy().copy(), kn.numpy(), vn.numpy()
    cores = oracle.max_threads()
    pos = shape.total_seq - 1
    steps, t0 = 0, time.perf_counter()
    while steps < max_steps and time.perf_counter() - t0 < budget_s:
        oracle.kv_append(kn, vn, kh, vh, shape.kv_heads, shape.head_dim, shape.max_seq, pos)
        oracle.decode(q, kh, vh, shape.num_heads, shape.kv_heads, shape.head_dim, shape.max_seq,
                      shape.total_seq, shape.window)
        steps += 1
    secs = time.perf_counter() - t0
    return steps, secs, cores


# ---------------------------------------------------------------- arms

def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    shape = workloads.DECODE_4K
    import oracle
    q, kc, vc, kn, vn = workloads.decode_inputs(shape.num_heads, shape.kv_heads, shape.head_dim,
                                                shape.max_seq, shape.seed, append=True)
    q, kh, vh, kn, vn = q.numpy(), kc.numpy().copy(), vc.numpy().copy(), kn.numpy(), vn.numpy()
    pos = shape.total_seq - 1

    def step():
        oracle.kv_append(kn, vn, kh, vh, shape.kv_heads, shape.head_dim, shape.max_seq, pos)
        oracle.decode(q, kh, vh, shape.num_heads, shape.kv_heads, shape.head_dim, shape.max_seq,
                      shape.total_seq, shape.window)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    bytes_step = shape.kv_bytes_algorithmic()
    value = bytes_step * args.steps / secs / 1e9
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "num_heads": shape.num_heads,
                   "kv_heads": shape.kv_heads, "head_dim": shape.head_dim,
                   "total_seq": shape.total_seq, "window": shape.window,
                   "step": "kv_append + decode, fp64 CPU oracle"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{args.steps} full decode steps (all 12 heads, 4096 rows)"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def our_arm(args):
    ws, rank, local = dist_env()
    init_dist(ws, "nccl")
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import attention_attn_prefill_causal_gb300 as attn

    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)
    if args.only in ("prefill_2k_tf32", "prefill_16k_tf32"):
        # Profiling aid: the TF32 mode on one prefill workload alone.
        ps = workloads.PREFILL_2K if args.only == "prefill_2k_tf32" else workloads.PREFILL_16K
        res = bench_prefill_tf32(attn, ps, device, stream, 200 if ps.m <= 4096 else 10, peaks,
                                 peak_src)
        if rank == 0:
            print(json.dumps({"only": args.only, "result": res}), flush=True)
        return 0
    if args.only in ("prefill_2k", "prefill_16k"):
        # Profiling aid: one prefill workload alone (no headline line).
        ps = workloads.PREFILL_2K if args.only == "prefill_2k" else workloads.PREFILL_16K
        res, det = bench_prefill(attn, ps, device, stream, 200 if ps.m <= 4096 else 20, peaks,
                                 peak_src)
        if rank == 0:
            print(json.dumps({"only": args.only, "result": res, "detail": det}), flush=True)
        return 0
    if args.only in ("decode_32k_window", "decode_32k_stream"):
        # Profiling aid: one 32768-row decode workload alone (no headline line).
        cs = (workloads.DECODE_32K_WINDOW if args.only == "decode_32k_window"
              else workloads.DECODE_32K_STREAM)
        res, det = bench_decode_companion(attn, cs, device, stream,
                                          2000 if cs.window else 200, peaks, peak_src)
        if rank == 0:
            print(json.dumps({"only": args.only, "result": res, "detail": det}), flush=True)
        return 0
    shape = workloads.DECODE_4K
    db = DecodeBench(attn, shape, device)
    err = db.check()
    if err > 1e-4:
        raise SystemExit(f"decode parity check failed before timing: max abs error {err}")

    g = db.graphs(stream)
    rem = remainder_graphs(db, stream)
    time_steps(g, db.R, rem, args.warmup, stream)  # warm-up: W untimed steps
    if args.steps % db.R:
        rem[args.steps % db.R]  # the graph of the last K % R steps, captured before the barrier

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t_host0 = time.time()
    secs = time_steps(g, db.R, rem, args.steps, stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(ws)
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)

    bytes_step = shape.kv_bytes_algorithmic()
    max_secs, total_bytes = aggregate(secs, bytes_step * args.steps, ws)
    value = total_bytes / max_secs / 1e9

    # Dominant kernel (the decode call: split + combine) timed alone in the
    # same way: graphs of decode calls over the rotating replicas.
    gd = db.graphs(stream, append=False)
    remd = remainder_graphs(db, stream, append=False)
    time_steps(gd, db.R, remd, db.R * 4, stream)
    n_dec = max(args.steps, db.R * 8)
    dsecs = time_steps(gd, db.R, remd, n_dec, stream)
    per_decode = dsecs / n_dec
    achieved = bytes_step / per_decode / 1e9
    hbm = float(peaks["hbm_gbs"])
    traffic = traffic_for(f"attn_decode:{shape.name}", ["decode.cu"])

    # Context for the small workload: a torch copy moving the same number of
    # DRAM bytes (the measurement that defines the HBM peak, at this size).
    floor_us = copy_floor_us(db.kc, bytes_step, stream)

    # End to end through the Python API.  Every step takes its q, k_new and
    # v_new from page-locked host memory and leaves its output in page-locked
    # host memory.  Two transports, each timed as eager Python calls and as
    # CUDA-graph replays of R steps:
    #  * host-resident: the call gets the host buffers; a one-CTA kernel of
    #    the call copies the inputs into the workspace over the CPU-GPU link
    #    and the combine writes the output there (no memcpy);
    #  * memcpy: one H2D copy of the packed inputs, the call on device
    #    buffers, one D2H copy of the output.
    # `value` is the eager host-resident step (max over ranks): one Python
    # API call per step, as a user writes it.
    q, kc, vc, kn, vn = db.host
    nq, nk = q.numel(), kn.numel()
    hio = torch.cat([q.reshape(-1), kn.reshape(-1), vn.reshape(-1)]).pin_memory()
    hbufs = (hio[:nq].view_as(q), hio[nq:nq + nk].view_as(kn), hio[nq + nk:].view_as(vn),
             torch.empty(shape.num_heads, shape.head_dim).pin_memory())
    hout = hbufs[3]

    def step_host(i):
        db.step(i, stream, bufs=hbufs)

    def step_copy(i):
        db.io.copy_(hio, non_blocking=True)
        db.step(i, stream)
        hout.copy_(db.out, non_blocking=True)

    e_steps = min(args.steps, 2000)

    def eager_secs(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(e_steps):
                fn(i)
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3, e_steps

    def graph_secs(fn):
        def chunk():
            for i in range(db.R):
                fn(i)
        g = make_graph(chunk, stream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, e_steps // db.R)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3, reps * db.R

    with torch.cuda.stream(stream):
        step_copy(0)
    torch.cuda.synchronize()
    ref_out = hout.clone()
    e_var = {}
    for name, fn, timer in (("graph_host_resident", step_host, graph_secs),
                            ("graph_memcpy", step_copy, graph_secs),
                            ("eager_host_resident", step_host, eager_secs),
                            ("eager_memcpy", step_copy, eager_secs)):
        secs_v, n_v = timer(fn)
        e_var[name] = (secs_v, n_v)
        if name.endswith("host_resident"):
            torch.cuda.synchronize()
            if not torch.equal(hout, ref_out):
                raise SystemExit("host-resident decode output differs from the device-buffer one")
    e_secs, e_n = e_var["eager_host_resident"]
    e_max, e_bytes = aggregate(e_secs, bytes_step * e_n, ws)
    e_variants = {k: {"gbs": round(bytes_step * n / sec / 1e9, 3),
                      "us_per_step": round(sec / n * 1e6, 3), "steps": n}
                  for k, (sec, n) in e_var.items()}

    # The other workloads, each as one compact object (cfg1 ... cfg5 in the
    # order of the five named workloads); details go to stderr with --detail.
    cfgs, details = {}, {}
    if not args.no_prefill and args.only == "all":
        cfgs["cfg1"] = bench_prefill_fp32_small(attn, workloads.PREFILL_SMALL, device, stream,
                                                3200, peaks)
    cfgs["cfg2"] = {"value": round(achieved, 2), "unit": "GB/s", "us": round(per_decode * 1e6, 3),
                    "frac": round(achieved / hbm, 4), "err": float(f"{err:.3g}"),
                    "copy_floor_us": round(floor_us, 3)}
    if not args.no_prefill and args.only == "all":
        cfgs["cfg3"], details["cfg3"] = bench_prefill(attn, workloads.PREFILL_2K, device, stream,
                                                      200, peaks, peak_src)
        cfgs["cfg4"], details["cfg4"] = bench_decode_companion(
            attn, workloads.DECODE_32K_WINDOW, device, stream, 2000, peaks, peak_src)
        cfgs["cfg5"], details["cfg5"] = bench_prefill(attn, workloads.PREFILL_16K, device, stream,
                                                      20, peaks, peak_src)
        cfgs["cfg3_tf32"] = bench_prefill_tf32(attn, workloads.PREFILL_2K, device, stream, 200,
                                               peaks, peak_src)
        cfgs["cfg5_tf32"] = bench_prefill_tf32(attn, workloads.PREFILL_16K, device, stream, 10,
                                               peaks, peak_src)
        stream32k, details["stream32k"] = bench_decode_companion(
            attn, workloads.DECODE_32K_STREAM, device, stream, 200, peaks, peak_src)
        cfgs_extra = {"stream32k": {"value": stream32k["value"], "frac": stream32k["frac"]},
                      "layers28": bench_layer_stack(attn, workloads.PREFILL_2K, device, stream)}
    else:
        cfgs_extra = {}

    status = attn.attn_get_device_status()
    if status != attn.ATTN_OK:
        raise SystemExit(f"device status after the run: {attn.attn_status_string(status)}")

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        steps_c, secs_c, cores = cpu_baseline_decode(shape)
        cpu = {"value": round(bytes_step * steps_c / secs_c / 1e9, 3), "unit": "GB/s",
               "cores": cores, "kind": "oracle",
               "sample": f"{steps_c} decode steps (append + all heads) in {secs_c:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(max_secs / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": shape.name, "num_heads": shape.num_heads,
                       "kv_heads": shape.kv_heads, "head_dim": shape.head_dim,
                       "total_seq": shape.total_seq, "window": shape.window,
                       "step": "attn_decode_append, CUDA-graph replays",
                       "l2": f"inputs larger than L2: {db.R} cache replicas",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                         "peak_source": f"hbm_gbs ({peak_src})", "kernel": "attn_decode call"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e_bytes / e_max / 1e9, 3), "unit": "GB/s",
                    "h2d_bytes_per_step": (q.numel() + kn.numel() + vn.numel()) * 4,
                    "d2h_bytes_per_step": shape.num_heads * shape.head_dim * 4},
            "gpu_launches": args.steps * db.launches_per_step,
            "clocks": clocks,
        }
        line.update(cfgs_extra)
        line.update(cfgs)
        print(json.dumps(line), flush=True)
        if args.detail:
            details["e2e_variants"] = e_variants
            print(json.dumps(details), file=sys.stderr, flush=True)
    barrier(ws)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--detail", action="store_true",
                    help="also print the per-workload details as JSON on stderr")
    ap.add_argument("--only", choices=["all", "decode", "prefill_2k", "prefill_16k",
                                       "prefill_2k_tf32", "prefill_16k_tf32",
                                       "decode_32k_window", "decode_32k_stream"],
                    default="all", help="profiling aid: run one workload only")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
