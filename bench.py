#!/usr/bin/env python
"""Benchmark of one grouped-query decode step on B300.

A step is one pass of the whole decode path over one batch: the new
token's K/V appended to the cache, then split-KV attention over the grown
cache with its log-sum-exp merge -- one ``gqa_decode_step`` call of the C ABI
of ``libgqa.so`` (one launch; a second, merge launch only for many-head
groups whose sequences the split cuts).  Inputs are seeded synthetic N(0, 1)
tensors resident in HBM.  Every step gets its own copy of the lengths
``seq_lens = L - 1``, so that each step appends at row L-1 and attends over
exactly the workload's L_b positions; the caches rotate through enough
copies that the bytes read between two uses of one copy exceed three L2
sizes.

Default workload: MHA decode, B=8, H=G=32, d=128, N=4096, bf16.  ``value`` is
the algorithmic HBM bytes of all steps on all ranks (K/V rows read once, q
read, out written, new K/V rows read and written) over the slowest rank's
time, in GB/s.  The line also carries the roofline of the attention call,
the end-to-end figure through host buffers, a CPU baseline (the fp64
oracle on a bounded sample) and a per-workload table (µs per call, GB/s)
covering the other decode workloads and the group-count sweep.

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-table]
  torchrun --nproc-per-node N bench.py --gpus N ...   (N > 1: one replica per GPU)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402
from grouped_query_decode_kv_b300 import cost  # noqa: E402

METRIC = "GQA decode attention µs/step and achieved HBM GB/s (fraction of B300 peak) vs G"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
TABLE_WORKLOADS = ["tiny", "mha", "gqa8", "mqa", "long"] + workloads.sweep_names()
FP8_TABLE = ("mha", "gqa8", "mqa", "sweep_g8")  # decode workloads also timed over an FP8 cache
CSRC = os.path.join(ROOT, "grouped_query_decode_kv_b300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------- helpers
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def hbm_peak():
    pk = measured_peaks()
    if "hbm_gbs" in pk:
        return float(pk["hbm_gbs"]), "measured (copy, MEASURED_PEAKS.json)"
    return FALLBACK_HBM_GBS, "fallback 6.4 TB/s"


# Device sources of the decode-attention kernels (split kernels, merge,
# append): an ncu traffic figure is only reported while it was taken on
# these exact sources.
STEP_KERNEL_SOURCES = ("gqa_device.cuh", "gqa_params.cuh", "gqa_schedule.cuh", "gqa_pipeline.cuh", "gqa_merge.cuh",
                       "gqa_tcgen05.cuh", "gqa_split_simt.cuh", "gqa_split_mma.cuh", "gqa_split_tc.cuh",
                       "gqa_small_kernels.cuh")


def code_of(text: str) -> str:
    """A C++ source without its comments, trailing blanks and empty lines:
    what the compiler sees (the sources hold no string that contains a
    comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the decode-attention kernels' device code (comments left out,
    so that editing a comment does not part a profile from its kernel)."""
    h = hashlib.sha256()
    for fn in STEP_KERNEL_SOURCES:
        with open(os.path.join(CSRC, fn)) as f:
            h.update(fn.encode() + code_of(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch of the split kernel from the committed ncu
    summary of this workload, if it was taken on the current sources."""
    path = os.path.join(PROFILES, f"gqa_split_{workload_name}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip().strip("`- ")
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(float(vals["traffic_bytes_per_call"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of this GPU's SM clock and throttle
    reasons while the benchmark runs; read-only."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        """Median SM clock and the active throttle reasons of the samples
        taken within [t0 - 0.25 s, t1 + 0.25 s] (wall clock)."""
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except (ValueError, IndexError):
                    continue
        try:
            os.unlink(self.path)
        except OSError:
            pass
        sel = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        if not sel and rows:
            sel = [min(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel)}


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a host scalar over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(per_rank_bytes: int, seconds_max: float, world: int) -> float:
    """Whole-job GB/s: the bytes every replica processed over the slowest
    replica's time (weak scaling: each rank runs the full workload)."""
    return per_rank_bytes * world / seconds_max / 1e9


# ----------------------------------------------------------------- GPU state
class DecodeState:
    """Device tensors of one workload: `copies` rotating cache sets, one
    lengths row per step, and the step's q / k_new / v_new / out."""

    def __init__(self, w: workloads.Workload, steps_total: int, device, copies: int, seed: int = 0):
        dt = w.torch_dtype
        self.w = w
        self.lens = workloads.make_seq_lens(w).to(torch.int64)
        g = torch.Generator(device=device).manual_seed(1000 + w.index + seed)
        self.k = [torch.randn(w.B, w.G, w.Nmax, w.d, generator=g, device=device).to(dt) for _ in range(copies)]
        self.v = [torch.randn(w.B, w.G, w.Nmax, w.d, generator=g, device=device).to(dt) for _ in range(copies)]
        # a step's inputs q, k_new, v_new are views of one buffer per copy, so
        # that the end-to-end leg moves them from the host in one copy
        nq, nkv = w.B * w.H * w.d, w.B * w.G * w.d
        self.inp = [torch.randn(nq + 2 * nkv, generator=g, device=device).to(dt) for _ in range(copies)]
        self.q = [t[:nq].view(w.B, w.H, w.d) for t in self.inp]
        self.kn = [t[nq:nq + nkv].view(w.B, w.G, w.d) for t in self.inp]
        self.vn = [t[nq + nkv:].view(w.B, w.G, w.d) for t in self.inp]
        self.out = [torch.empty(w.B, w.H, w.d, dtype=dt, device=device) for _ in range(copies)]
        pre = torch.clamp(self.lens - 1, min=0).to(torch.int32)
        self.sl = pre.unsqueeze(0).repeat(steps_total, 1).to(device).contiguous()
        self.copies = copies
        self.lens_after = torch.clamp(self.lens - 1, min=0) + 1
        from grouped_query_decode_kv_b300 import gqa_decode_workspace_bytes
        self.ws_bytes = gqa_decode_workspace_bytes(w.B, w.H, w.G, w.d, w.Nmax, dt)
        # the step's workspace: zero-filled once, each call leaves it ready
        self.ws = torch.zeros(max(self.ws_bytes, 1), dtype=torch.uint8, device=device)

    def reset_lengths(self):
        pre = torch.clamp(self.lens - 1, min=0).to(torch.int32)
        self.sl.copy_(pre.unsqueeze(0).expand_as(self.sl))

    @property
    def attention_bytes(self) -> int:
        return cost.decode_attention_bytes(self.lens_after.tolist(), self.w.H, self.w.G, self.w.d, self.w.elt)

    @property
    def append_bytes(self) -> int:
        return cost.kv_append_bytes(self.w.B, self.w.G, self.w.d, self.w.elt)


def copies_for(w: workloads.Workload, l2_bytes: int, mem_budget: int) -> int:
    cache = cost.kv_cache_bytes(w.B, w.G, w.Nmax, w.d, w.elt)
    c = max(2, math.ceil(3 * l2_bytes / max(cache, 1)))
    return max(1, min(c, mem_budget // max(cache, 1), 64))


def run_steps(st: DecodeState, first: int, count: int, ev=None):
    """`count` decode steps (gqa_decode_step_ws: append + attention in one call);
    step i uses cache copy i % copies and lengths row i.  With `ev` (a list of
    event pairs) every step call is bracketed by CUDA events on the current
    stream."""
    import grouped_query_decode_kv_b300 as gqa
    w = st.w
    for i in range(first, first + count):
        c = i % st.copies
        sl = st.sl[i]
        if ev is not None:
            ev[i - first][0].record()
        gqa.gqa_decode_step_ws(st.q[c], st.kn[c], st.vn[c], st.k[c], st.v[c], sl, w.scale, st.out[c], st.ws)
        if ev is not None:
            ev[i - first][1].record()


def _graph_stats(fn_seq, reset=None, reps: int = 21) -> dict:
    """Device time per call (µs) of a sequence of library calls captured into
    one CUDA graph (back to back, so the host's per-call cost is out): the
    graph is replayed `reps` times after one untimed replay, each replay
    bracketed by CUDA events; every replay gives the mean time of its calls,
    and the median with the 10th and 90th percentiles of those replay means
    is returned ({"us", "p10", "p90", "calls"}).  `reset` (outside the timed
    replays) restores state between replays."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    if reset:
        reset()  # the warm-up calls start from the same state as every replay
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn_seq()  # warm the calls once outside capture (module load, attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    if reset:
        reset()
    with torch.cuda.graph(g):
        n = fn_seq()
    per_call = []
    for i in range(reps + 1):
        if reset:
            reset()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        if i > 0:
            per_call.append(a.elapsed_time(b) * 1e3 / n)
    del g
    per_call.sort()
    q = lambda f: per_call[min(len(per_call) - 1, int(f * len(per_call)))]
    return {"us": statistics.median(per_call), "p10": q(0.1), "p90": q(0.9), "calls": n * reps}


def _graph_time(fn_seq, reset=None) -> float:
    return _graph_stats(fn_seq, reset)["us"]


def time_attention_only(w: workloads.Workload, device, iters: int, warm: int, l2_bytes: int, mem_budget: int):
    """Per-workload table row: device time per attention call and per
    kv_append call, from CUDA-graph replays of `iters` back-to-back calls
    (the caches rotate over enough copies to defeat L2; lengths fixed at L_b)."""
    import grouped_query_decode_kv_b300 as gqa
    copies = copies_for(w, l2_bytes, mem_budget)
    st = DecodeState(w, iters, device, copies, seed=17)
    full = st.lens.to(torch.int32).to(device)
    ws = torch.zeros(max(st.ws_bytes, 1), dtype=torch.uint8, device=device)

    def attn_seq():
        for i in range(iters):
            c = i % copies
            gqa.gqa_decode_attention_ws(st.q[c], st.k[c], st.v[c], full, w.scale, st.out[c], ws)
        return iters

    def append_seq():
        for i in range(iters):
            c = i % copies
            gqa.kv_append(st.kn[c], st.vn[c], st.k[c], st.v[c], st.sl[i])
        return iters

    def step_seq():
        for i in range(iters):
            c = i % copies
            gqa.gqa_decode_step_ws(st.q[c], st.kn[c], st.vn[c], st.k[c], st.v[c], st.sl[i], w.scale, st.out[c], ws)
        return iters

    for i in range(warm):
        c = i % copies
        gqa.gqa_decode_attention_ws(st.q[c], st.k[c], st.v[c], full, w.scale, st.out[c], ws)
    stats = _graph_stats(attn_seq)
    us = stats["us"]
    us_append = _graph_time(append_seq, reset=st.reset_lengths)
    us_step = _graph_time(step_seq, reset=st.reset_lengths)
    err = gqa.gqa_get_device_error()
    lens_full = st.lens.tolist()
    abytes = cost.decode_attention_bytes(lens_full, w.H, w.G, w.d, w.elt)
    peak, _ = hbm_peak()
    row = {
        "B": w.B, "H": w.H, "G": w.G, "d": w.d, "Nmax": w.Nmax, "dtype": w.dtype, "sum_L": int(sum(lens_full)),
        "us": round(us, 2), "us_p10": round(stats["p10"], 2), "us_p90": round(stats["p90"], 2),
        "calls_timed": stats["calls"], "bytes": abytes, "gbs": round(abytes / us / 1e3, 1),
        "frac_measured": round(abytes / us / 1e3 / peak, 3),
        "frac_8tbs": round(abytes / us / 1e3 / NOMINAL_HBM_GBS, 3),
        "tflops": round(cost.decode_attention_flops(lens_full, w.H, w.d) / us / 1e6, 1),
        "kv_append_us": round(us_append, 2), "step_us": round(us_step, 2), "copies": copies,
        "device_error": err,
    }
    del st, ws
    torch.cuda.empty_cache()
    return row


def time_multi(w: workloads.Workload, device, iters: int, warm: int, l2_bytes: int, mem_budget: int):
    """Table row of a several-token workload (w.tokens query tokens per
    sequence, one gqa_decode_attention_multi_ex call): device time per call
    from CUDA-graph replays over rotating cache copies, the algorithmic bytes
    (cache once, q and out of every token) and query tokens per second."""
    import grouped_query_decode_kv_b300 as gqa
    T = w.tokens
    copies = copies_for(w, l2_bytes, mem_budget)
    dt = w.torch_dtype
    lens = workloads.make_seq_lens(w)
    g = torch.Generator(device=device).manual_seed(1000 + w.index + 17)
    k = [torch.randn(w.B, w.G, w.Nmax, w.d, generator=g, device=device).to(dt) for _ in range(copies)]
    v = [torch.randn(w.B, w.G, w.Nmax, w.d, generator=g, device=device).to(dt) for _ in range(copies)]
    q = [torch.randn(w.B, T, w.H, w.d, generator=g, device=device).to(dt) for _ in range(copies)]
    out = [torch.empty(w.B, T, w.H, w.d, dtype=dt, device=device) for _ in range(copies)]
    sl = lens.to(device)
    need = gqa.gqa_decode_workspace_bytes_ex(w.B, T * w.H, w.G, w.d, w.Nmax, dt, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

    def seq():
        for i in range(iters):
            c = i % copies
            gqa.gqa_decode_attention_multi_ex(q[c], k[c], v[c], sl, w.scale, out[c], 0, ws)
        return iters

    for i in range(warm):
        c = i % copies
        gqa.gqa_decode_attention_multi_ex(q[c], k[c], v[c], sl, w.scale, out[c], 0, ws)
    us = _graph_time(seq)
    err = gqa.gqa_get_device_error()
    lens_l = lens.tolist()
    abytes = cost.decode_attention_bytes(lens_l, w.H, w.G, w.d, w.elt, tokens=T)
    peak, _ = hbm_peak()
    row = {
        "B": w.B, "T": T, "H": w.H, "G": w.G, "d": w.d, "Nmax": w.Nmax, "dtype": w.dtype, "sum_L": int(sum(lens_l)),
        "us": round(us, 2), "bytes": abytes, "gbs": round(abytes / us / 1e3, 1),
        "frac_measured": round(abytes / us / 1e3 / peak, 3),
        "tflops": round(cost.decode_attention_flops(lens_l, w.H, w.d, tokens=T) / us / 1e6, 1),
        "query_tokens_per_s": round(w.B * T / us * 1e6, 1), "copies": copies, "device_error": err,
    }
    del k, v, q, out, ws
    torch.cuda.empty_cache()
    return row


def time_fp8(w: workloads.Workload, device, iters: int, l2_bytes: int, mem_budget: int):
    """Table row of a decode workload over an FP8 E4M3 cache: device time per
    gqa_decode_attention_fp8_ws call and per kv_append_fp8 call (CUDA-graph
    replays over rotating cache copies, together >= 3 x L2), GB/s of the
    algorithmic bytes (one byte per cached K/V element, bf16 q and out)."""
    import grouped_query_decode_kv_b300 as gqa
    cache = cost.kv_cache_bytes(w.B, w.G, w.Nmax, w.d, 1)
    copies = max(2, min(64, math.ceil(3 * l2_bytes / max(cache, 1)), max(1, mem_budget // max(cache, 1))))
    g = torch.Generator(device=device).manual_seed(3000 + w.index)
    k = [torch.randint(0, 0x7E, (w.B, w.G, w.Nmax, w.d), generator=g, device=device, dtype=torch.uint8)
         for _ in range(copies)]
    v = [torch.randint(0, 0x7E, (w.B, w.G, w.Nmax, w.d), generator=g, device=device, dtype=torch.uint8)
         for _ in range(copies)]
    q = torch.randn(w.B, w.H, w.d, generator=g, device=device).bfloat16()
    out = torch.empty_like(q)
    ks = torch.full((w.G,), 1 / 64, device=device)
    vs = torch.full((w.G,), 1 / 64, device=device)
    kn = torch.randn(w.B, w.G, w.d, generator=g, device=device).bfloat16()
    vn = torch.randn(w.B, w.G, w.d, generator=g, device=device).bfloat16()
    lens = workloads.make_seq_lens(w)
    full = lens.to(device)
    pre = torch.clamp(lens.to(torch.int64) - 1, min=0).to(torch.int32)
    rows = pre.unsqueeze(0).repeat(iters, 1).to(device).contiguous()
    need = gqa.gqa_decode_workspace_bytes_fp8(w.B, w.H, w.G, w.d, w.Nmax)
    ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=device)

    def attn():
        for i in range(iters):
            c = i % copies
            gqa.gqa_decode_attention_fp8_ws(q, k[c], v[c], ks, vs, full, w.scale, out, ws)
        return iters

    def app():
        for i in range(iters):
            c = i % copies
            gqa.kv_append_fp8(kn, vn, k[c], v[c], ks, vs, rows[i])
        return iters

    def reset():
        rows.copy_(pre.unsqueeze(0).expand_as(rows))

    us = _graph_time(attn)
    us_app = _graph_time(app, reset=reset)
    err = gqa.gqa_get_device_error()
    nbytes = 2 * w.G * int(lens.sum()) * w.d + 2 * w.B * w.H * w.d * 2
    peak, _ = hbm_peak()
    row = {"B": w.B, "H": w.H, "G": w.G, "d": w.d, "Nmax": w.Nmax, "cache": "fp8 e4m3", "us": round(us, 2),
           "bytes": nbytes, "gbs": round(nbytes / us / 1e3, 1), "frac_measured": round(nbytes / us / 1e3 / peak, 3),
           "kv_append_fp8_us": round(us_app, 2), "copies": copies, "device_error": err}
    del k, v, ws
    torch.cuda.empty_cache()
    return row


def time_projection(name: str, device, iters: int, l2_bytes: int, mem_budget: int):
    """Table row of a Q/K/V projection layer: device time per
    gqa_qkv_project_ws call from CUDA-graph replays over rotating weight
    copies (together >= 3 x L2), GB/s of the weight, x and q/k/v bytes."""
    import grouped_query_decode_kv_b300 as gqa
    c = workloads.PROJECTIONS[name]
    B, A, H, G, d = c["B"], c["A"], c["H"], c["G"], c["d"]
    wbytes = (H + 2 * G) * A * d * 2
    copies = max(2, min(64, math.ceil(3 * l2_bytes / wbytes), max(1, mem_budget // wbytes)))
    g = torch.Generator(device=device).manual_seed(c["seed"])
    s = A ** -0.5
    x = torch.randn(B, A, generator=g, device=device).bfloat16()
    ws_ = [(torch.randn(H, A, d, generator=g, device=device) * s).bfloat16() for _ in range(copies)]
    wk_ = [(torch.randn(G, A, d, generator=g, device=device) * s).bfloat16() for _ in range(copies)]
    wv_ = [(torch.randn(G, A, d, generator=g, device=device) * s).bfloat16() for _ in range(copies)]
    q = torch.empty(B, H, d, dtype=torch.bfloat16, device=device)
    kn = torch.empty(B, G, d, dtype=torch.bfloat16, device=device)
    vn = torch.empty(B, G, d, dtype=torch.bfloat16, device=device)
    need = gqa.gqa_qkv_project_workspace_bytes(B, A, H, G, d)
    wsp = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

    def seq():
        for i in range(iters):
            j = i % copies
            gqa.gqa_qkv_project_ws(x, ws_[j], wk_[j], wv_[j], q, kn, vn, wsp)
        return iters

    us = _graph_time(seq)
    err = gqa.gqa_get_device_error()
    nbytes = cost.qkv_project_bytes(B, A, H, G, d)
    peak, _ = hbm_peak()
    row = {"B": B, "A": A, "H": H, "G": G, "d": d, "us": round(us, 2), "bytes": nbytes,
           "gbs": round(nbytes / us / 1e3, 1), "frac_measured": round(nbytes / us / 1e3 / peak, 3),
           "tflops": round(cost.qkv_project_flops(B, A, H, G, d) / us / 1e6, 1), "copies": copies,
           "device_error": err}
    del ws_, wk_, wv_, wsp
    torch.cuda.empty_cache()
    return row


def read_ceiling(device) -> dict:
    """Read-only streaming ceiling of this GPU: the library's probe reads a
    4 GiB buffer once (16-byte loads, and bulk copies into shared memory as
    the K/V pipeline does), best of 10 timed passes each after 3 warm-up
    passes, in GB/s; `gbs` is the larger of the two."""
    import grouped_query_decode_kv_b300 as gqa
    nbytes = 1 << 32
    x = torch.ones(nbytes // 2, dtype=torch.bfloat16, device=device)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    out = {}
    for mode, name in ((0, "loads"), (1, "bulk_copies")):
        for _ in range(3):
            gqa.gqa_stream_read(x, mode, sink)
        ts = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gqa.gqa_stream_read(x, mode, sink)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e-3)
        out[name] = round(nbytes / min(ts) / 1e9, 1)
    del x
    torch.cuda.empty_cache()
    out["gbs"] = max(out["loads"], out["bulk_copies"])
    return out


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(w: workloads.Workload, budget_s: float, max_units: int = 1 << 30, _cache={}, threads: int = 0):
    """Times the fp64 CPU oracle on a bounded sample of the workload: whole
    (batch, KV group) units, batch rows in order, as many as fit in about
    `budget_s` seconds (at least one), on `threads` host threads (0: every
    core in this process's affinity mask).  Returns (GB/s of algorithmic
    bytes, units done, seconds, threads)."""
    import oracle
    threads = threads or len(os.sched_getaffinity(0))
    lens = workloads.make_seq_lens(w).tolist()
    key = w.name
    if key not in _cache:
        # one batch row of inputs, reused for every sampled row (timing only)
        small = w.replace(B=1, Nmax=max(lens))
        _cache[key] = workloads.make_inputs(small, seq_lens=torch.tensor([max(lens)], dtype=torch.int32),
                                            poison=False)
    x = _cache[key]
    done_bytes, done_units, spent = 0, 0, 0.0
    b = 0
    per_row = None
    while (done_units == 0 or spent < budget_s) and done_units < max_units:
        L = int(lens[b % w.B])
        groups = w.G
        if per_row is not None and spent + per_row > budget_s * 1.2:
            # a whole row would overrun the budget: take a slice of its groups
            groups = max(1, int(w.G * (budget_s - spent) / per_row))
        groups = min(groups, max_units - done_units)
        q = x["q"][:, : groups * w.n_rep].contiguous()
        k = x["k_cache"][:, :groups, :L].contiguous()
        v = x["v_cache"][:, :groups, :L].contiguous()
        sl = torch.tensor([L], dtype=torch.int32)
        t0 = time.perf_counter()
        oracle.decode_attention(q, k, v, sl, w.scale, nthreads=threads)
        dt = time.perf_counter() - t0
        spent += dt
        if groups == w.G:
            per_row = dt
        done_units += groups
        done_bytes += cost.decode_attention_bytes([L], groups * w.n_rep, groups, w.d, w.elt)
        b += 1
    return done_bytes / spent / 1e9, done_units, spent, threads


ORACLE_TABLE = ["tiny", "mha", "gqa8", "mqa", "long", "sweep_g1", "sweep_g8", "sweep_g64"]
ORACLE_ONE_THREAD = ["tiny", "mha", "gqa8"]


def oracle_table(budget_s: float) -> dict:
    """The fp64 oracle per decode workload on a bounded sample of each (about
    `budget_s` seconds), on every host core and, for the three smaller
    workloads, on one thread: GB/s of algorithmic bytes and the µs one whole
    call would take at that rate."""
    out = {}
    for name in ORACLE_TABLE:
        w = workloads.workload(name)
        lens = workloads.make_seq_lens(w).tolist()
        call_bytes = cost.decode_attention_bytes(lens, w.H, w.G, w.d, w.elt)
        row = {}
        for label, thr in (("all_cores", 0), ("one_thread", 1)):
            if label == "one_thread" and name not in ORACLE_ONE_THREAD:
                continue
            gbs, units, spent, used = oracle_sample(w, budget_s, threads=thr)
            row[label] = {"gbs": round(gbs, 4), "us_per_call": round(call_bytes / gbs / 1e3, 1), "threads": used,
                          "units_sampled": units, "seconds": round(spent, 2)}
        out[name] = row
    return out


# ----------------------------------------------------------------- arms
def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, timed on this
    host's cores over a bounded sample of the workload per step."""
    if rank != 0:
        return 0
    w = workloads.workload(args.workload)
    steps, warm = args.steps, args.warmup
    # size each step so that the whole run stays within about two minutes
    _, units1, t1, threads = oracle_sample(w, 0.0, max_units=1)
    per_unit = max(t1, 1e-6)
    per_step_budget = min(5.0, 120.0 / max(steps + warm, 1))
    units = max(1, min(w.B * w.G, int(per_step_budget / per_unit)))
    for _ in range(warm):
        oracle_sample(w, 0.0, max_units=units)
    tot_bytes, tot_s = 0.0, 0.0
    for _ in range(steps):
        gbs, u, s, _ = oracle_sample(w, 1e9, max_units=units)
        tot_bytes += gbs * s * 1e9
        tot_s += s
    value = tot_bytes / tot_s / 1e9
    sample = f"{units} of {w.B * w.G} (batch, KV-group) units of the {w.name} workload per step, fp64 oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": round(tot_s / steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.description, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import grouped_query_decode_kv_b300 as gqa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    gqa.load_library()
    gqa.gqa_get_device_error()

    w = workloads.workload(args.workload)
    props = torch.cuda.get_device_properties(device)
    l2 = props.L2_cache_size
    mem_budget = int(props.total_memory * 0.5)
    copies = copies_for(w, l2, mem_budget)
    steps, warm = args.steps, args.warmup
    st = DecodeState(w, warm + steps, device, copies)
    stream = torch.cuda.current_stream(device)

    # ---- pre-warm: about a second of the same step so that clocks settle
    # before the W warm-up steps (untimed; lengths are reset afterwards).
    # The clock sampler starts first, and nothing idles the GPU between the
    # pre-warm and the timed region.
    sampler = ClockSampler(device.index)
    pre = 0
    t_pre = time.time()
    while time.time() - t_pre < args.prewarm:
        run_steps(st, 0, min(warm + steps, 200))
        torch.cuda.synchronize()
        st.reset_lengths()
        pre += 1

    # ---- device-resident timed region: K steps, nothing else in the stream
    run_steps(st, 0, warm)
    torch.cuda.synchronize()
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_begin.record(stream)
    run_steps(st, warm, steps)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world, device)
    wall1 = time.time()

    # ---- the same K steps again with CUDA events around every attention
    # call, for the per-call duration of the roofline (events between the
    # kernels cost a few µs of overlap, so they stay out of the region above)
    st.reset_lengths()
    run_steps(st, 0, warm)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    run_steps(st, warm, steps, ev)
    torch.cuda.synchronize()
    wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(wall0, wall2)
    secs = t_begin.elapsed_time(t_end) * 1e-3
    secs_max = reduce_max(secs, world, device)
    attn_us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    dev_err = gqa.gqa_get_device_error()

    # kernels per step, counted from a graph of one step (the lengths are
    # restored afterwards); the static rule if the count is unavailable
    per_step = counted_launches(lambda: gqa.gqa_decode_step_ws(st.q[0], st.kn[0], st.vn[0], st.k[0], st.v[0],
                                                                st.sl[0], w.scale, st.out[0], st.ws))
    st.reset_lengths()
    if per_step is None:
        per_step = launches_per_step(w)
    step_bytes = st.attention_bytes + st.append_bytes
    value = aggregate(step_bytes * steps, secs_max, world)
    peak, peak_src = hbm_peak()
    attn_mean = statistics.mean(attn_us)
    # The roofline's launch duration: the timed region's device time over its
    # launches (the step is one kernel; with the merge kernel too, the pair).
    # Events around every call, the second pass above, add a gap between the
    # kernels; that distribution is reported beside it.
    launch_us = secs * 1e6 / steps
    achieved = step_bytes / launch_us / 1e3

    # ---- end to end through host buffers: q, k_new, v_new in, out back
    hin = [t.cpu().pin_memory() for t in st.inp]  # q | k_new | v_new of each copy
    ho = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.out]
    st.reset_lengths()
    e_steps = steps

    # Copies run on their own stream, pipelined with the steps: step i's
    # inputs are copied while step i-1 computes and step i's result is read
    # back while step i+1 computes (every step still moves its own bytes;
    # events order each copy against the step that uses its buffers, and the
    # caches rotate over `copies` >= 2 sets).
    cstream = torch.cuda.Stream(device)
    h_ev = [torch.cuda.Event() for _ in range(copies)]
    s_ev = [torch.cuda.Event() for _ in range(copies)]

    def h2d(i):
        c = i % copies
        with torch.cuda.stream(cstream):
            if i >= copies:
                cstream.wait_event(s_ev[c])  # step i - copies has stopped reading buffer c
            st.inp[c].copy_(hin[c], non_blocking=True)
            h_ev[c].record(cstream)

    def e2e_run(first, count):
        h2d(first)
        for i in range(first, first + count):
            c = i % copies
            stream.wait_event(h_ev[c])
            gqa.gqa_decode_step_ws(st.q[c], st.kn[c], st.vn[c], st.k[c], st.v[c], st.sl[i], w.scale, st.out[c],
                                   st.ws, stream=stream)
            s_ev[c].record(stream)
            if i + 1 < first + count:
                h2d(i + 1)
            with torch.cuda.stream(cstream):
                cstream.wait_event(s_ev[c])
                ho[c].copy_(st.out[c], non_blocking=True)
        stream.wait_stream(cstream)

    # Untimed pre-warm of this loop too (about as long as the device leg's):
    # after even half a second of idling (the clock sampler's shutdown, the
    # pinned buffers) the host issues the loop up to twice as slowly until it
    # has been busy for a while, and this leg is bound by the host side.
    t_pre = time.time()
    while time.time() - t_pre < args.prewarm:
        e2e_run(0, min(warm + steps, 200))
        torch.cuda.synchronize()
        st.reset_lengths()
    e2e_run(0, warm)
    torch.cuda.synchronize()
    st.reset_lengths()
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cstream.wait_event(e0)
    h0 = time.perf_counter()
    e2e_run(0, e_steps)
    host_issue_us = (time.perf_counter() - h0) * 1e6 / e_steps
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world, device)
    e_secs = reduce_max(e0.elapsed_time(e1) * 1e-3, world, device)
    e2e_value = aggregate(step_bytes * e_steps, e_secs, world)
    h2d = hin[0].numel() * hin[0].element_size()
    d2h = ho[0].numel() * ho[0].element_size()
    dev_err |= gqa.gqa_get_device_error()

    # ---- per-workload table and the read-only ceiling (rank 0 only)
    table = None
    table_multi = None
    table_proj = None
    table_fp8 = None
    ceiling = None
    del st
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_table:
        ceiling = read_ceiling(device)
        table = {}
        for name in TABLE_WORKLOADS:
            table[name] = time_attention_only(workloads.workload(name), device, args.table_iters, 5, l2, mem_budget)
            table[name]["frac_read_ceiling"] = round(table[name]["gbs"] / ceiling["gbs"], 3)
        table_multi = {}
        for name in workloads.multi_names():
            table_multi[name] = time_multi(workloads.workload(name), device, args.table_iters, 5, l2, mem_budget)
        table_fp8 = {}
        for name in FP8_TABLE:
            table_fp8[name] = time_fp8(workloads.workload(name), device, args.table_iters, l2, mem_budget)
        table_proj = {}
        for name in sorted(workloads.PROJECTIONS):
            table_proj[name] = time_projection(name, device, args.table_iters, l2, mem_budget)

    cpu = None
    cpu_table = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu_table = oracle_table(args.cpu_table_seconds)
        gbs, units, spent, threads = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{units} (batch, KV-group) units of the {w.name} workload, taken in batch-row order "
                         f"over its {w.B * w.G} units ({units / (w.B * w.G):.1f} passes; {spent:.1f} s of fp64 "
                         f"CPU work)"}

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return 0

    traffic = profiled_traffic(w.name)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": round(secs_max / steps * 1e3, 5),
        "us_per_step": round(secs_max / steps * 1e6, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {
            "workload": w.description, "B": w.B, "H": w.H, "G": w.G, "d": w.d, "Nmax": w.Nmax,
            "seq_lens": "fixed" if w.lens[0] == "fixed" else f"uniform[{w.lens[1]},{w.lens[2]}]",
            "parallelism": f"replicas x{world}",
            "l2": f"rotating {copies} cache copies ({copies * cost.kv_cache_bytes(w.B, w.G, w.Nmax, w.d, w.elt) / 2**20:.0f} MiB"
                  f" >= 3 x L2 {l2 / 2**20:.0f} MiB)",
            "step": "gqa_decode_step: kv_append + split-KV attention + LSE merge, one launch",
            "timing": f"{args.prewarm:.1f} s untimed pre-warm, W warm-up steps, then K steps bracketed by "
                      "CUDA events with nothing else in the stream; the roofline's launch duration is that "
                      "region's device time over its K launches (a second pass with events around each step "
                      "call is reported beside it); the end-to-end leg has its own untimed pre-warm of the "
                      "same length and W warm-up steps; table rows are CUDA-graph replays of 200 calls, "
                      "median and p10/p90 of 21 replay means",
            "l2_table": "every table row rotates cache copies totalling >= 3 x L2",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "gqa_decode_step call (split-KV kernel with the append fused; in-kernel merge)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": peak_src,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "frac_read_ceiling": round(achieved / ceiling["gbs"], 4) if ceiling else None,
            "bytes_per_call": step_bytes,
            "us_per_call": round(launch_us, 2),
            "us_per_call_evented": {"mean": round(attn_mean, 2),
                                    "median": round(statistics.median(attn_us), 2),
                                    "p10": round(sorted(attn_us)[len(attn_us) // 10], 2),
                                    "p90": round(sorted(attn_us)[(9 * len(attn_us)) // 10], 2),
                                    "calls": len(attn_us)},
            "traffic": traffic,
        },
        "cpu_baseline": cpu,
        "cpu_baseline_table": cpu_table,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e_secs / e_steps * 1e6, 2), "host_issue_us_per_step": round(host_issue_us, 2)},
        "gpu_launches": per_step * steps,
        "clocks": clocks,
        "device_error": dev_err,
        "read_ceiling_gbs": ceiling["gbs"] if ceiling else None,
        "read_ceiling": ceiling,
        "table": table,
        "table_multi_token": table_multi,
        "table_qkv_projection": table_proj,
        "table_fp8_cache": table_fp8,
    }
    print(json.dumps(line), flush=True)
    return 0


def counted_launches(fn) -> int:
    """Kernels one call of `fn` launches, counted from a CUDA graph of it:
    the kernel nodes of the captured graph (None when the count fails)."""
    try:
        from cuda.bindings import runtime as cudart
        g = torch.cuda.CUDAGraph(keep_graph=True)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize()
        graph = cudart.cudaGraph_t(init_value=g.raw_cuda_graph())
        err, nodes, n = cudart.cudaGraphGetNodes(graph, 0)
        err, nodes, n = cudart.cudaGraphGetNodes(graph, n)
        kinds = [cudart.cudaGraphNodeGetType(x)[1] for x in nodes]
        count = sum(1 for k in kinds if k == cudart.cudaGraphNodeType.cudaGraphNodeTypeKernel)
        g.reset()
        return count
    except Exception:
        return None


def launches_per_step(w: workloads.Workload) -> int:
    """Kernels one gqa_decode_step launches: the split kernel, plus the merge
    kernel for groups of three or more heads (bf16) whose sequences a split
    may cut (the merge of one- and two-head groups runs inside the split
    kernel)."""
    import grouped_query_decode_kv_b300 as gqa
    ws = gqa.gqa_decode_workspace_bytes(w.B, w.H, w.G, w.d, w.Nmax, w.torch_dtype)
    many_heads = w.dtype == "bf16" and w.n_rep >= 3
    return 1 + (1 if (ws > 0 and many_heads) else 0)


def st_bytes(w: workloads.Workload) -> int:
    lens = workloads.make_seq_lens(w).tolist()
    return cost.decode_attention_bytes(lens, w.H, w.G, w.d, w.elt)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="mha", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-table", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--table-iters", type=int, default=200)
    ap.add_argument("--table-only", choices=["proj", "fp8", "multi"], default=None,
                    help="time only one group of table rows (projection layers, FP8 cache, several "
                         "tokens) and print them as one JSON line; for profiling those kernels")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-table-seconds", type=float, default=2.0,
                    help="seconds of oracle work per workload (and thread count) in cpu_baseline_table")
    ap.add_argument("--prewarm", type=float, default=1.0, help="seconds of untimed steps before the warm-up")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.table_only:
        return run_table_only(args, local)
    return run_ours(args, world, rank, local)


def run_table_only(args, local):
    """One group of table rows on this GPU, printed as one JSON line (no
    step timing, no baselines): the command the ncu summaries of the
    projection and FP8 kernels are taken with."""
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    mem_budget = int(torch.cuda.mem_get_info(device)[0] * 0.5)
    rows = {}
    if args.table_only == "proj":
        for name in sorted(workloads.PROJECTIONS):
            rows[name] = time_projection(name, device, args.table_iters, l2, mem_budget)
    elif args.table_only == "fp8":
        for name in FP8_TABLE:
            rows[name] = time_fp8(workloads.workload(name), device, args.table_iters, l2, mem_budget)
    else:
        for name in workloads.multi_names():
            rows[name] = time_multi(workloads.workload(name), device, args.table_iters, 5, l2, mem_budget)
    print(json.dumps({"table_only": args.table_only, "rows": rows}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
