#!/usr/bin/env python
"""Throughput of the ClusterKV decode path on one GB300 (or N, one process each).

One bench step is one whole ClusterKV job of the 32k decode workload: 32 layers
x 8 KV heads (256 units), head dim 128, GQA 4, bf16, a 32768-token prompt:
  * prefill clustering of every unit (C = 409, 10 Lloyd iterations);
  * 1024 decode steps, each: centroid scoring, cluster selection (B = 1024),
    sparse attention over sinks + pending + selected tokens; incremental
    clustering of the 320 newest tokens into 4 clusters before steps 320, 640
    and 960.
Inputs (keys, values, the 1024 queries of every unit) are generated on the
device before the timed region.  value = decode tokens of the job / job time
(clustering included); the per-phase numbers are extra keys.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from recallable_kv_cache_gb300 import synth  # noqa: E402

METRIC = "sparse-decode tokens/s at 32k ctx, B=1024; K-means ms/layer; % of HBM roofline"

# DRAM bytes (read + write) of one decode step (the kernels of one step) per
# algorithmic byte, from one ncu capture of the current kernels on a 64-unit
# case; the traffic of a full-size step is this ratio times its algorithmic
# bytes.  None whenever a kernel changes until it is captured again.
STEP_TRAFFIC_PER_ALG_BYTE = 45.19e6 / 42.46e6
STEP_TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the four kernels of one decode step, "
                       "64-unit case (caches flushed between kernels), scaled by algorithmic bytes "
                       "(profiles/decode_step_traffic_decode_32k.md)")
WORKLOAD = "decode_32k"
K_UPLOAD_STREAMS = 1  # the prompt's keys go up in this many concurrent copies


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-workloads", action="store_true", help="skip the other workloads' measurements")
    p.add_argument("--no-comparators", action="store_true", help="skip the Quest / reuse / channel / full-KV side "
                                                                  "measurements")
    p.add_argument("--units", type=int, default=0, help="override the unit count (small profiling cases)")
    p.add_argument("--decode-steps", type=int, default=0, help="override the decode steps (profiling)")
    p.add_argument("--sync-incremental", action="store_true",
                   help="cluster the new tokens inline instead of on a side stream overlapping the next step")
    p.add_argument("--e2e-out-copies", action="store_true",
                   help="end-to-end run with mapped host memory: each step's output into a device buffer read "
                        "back while the next step runs, instead of written by the attention straight into pinned "
                        "host memory (measured slower: with a copy node per step the graph's prompt upload slows "
                        "down too)")
    p.add_argument("--e2e-copy-nodes", action="store_true",
                   help="end-to-end run: copy each step's inputs and outputs instead of mapping host memory")
    p.add_argument("--upload-streams", type=int, default=K_UPLOAD_STREAMS,
                   help="concurrent copies for the prompt keys' upload in the end-to-end run")
    p.add_argument("--no-l2-persist", action="store_true",
                   help="leave the centroid scoring copy and perm out of a persisting L2 set-aside")
    p.add_argument("--path", choices=["separate", "step"], default="separate",
                   help="decode step as ckv_select + ckv_sparse_decode_attn, or one "
                        "ckv_decode_step call")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), "measured", d
    return 6800.0, "fallback", {}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.index is not None:
            cmd += ["-i", str(self.index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- events in graphs
class ExternalEvents:
    """cudaEventRecordWithFlags(..., cudaEventRecordExternal) so that event
    records captured into a CUDA graph become timing nodes of the graph."""

    def __init__(self):
        path = None
        for line in open("/proc/self/maps"):
            if "libcudart" in line:
                path = line.split()[-1]
                break
        self.rt = ctypes.CDLL(path or "libcudart.so")
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventRecordWithFlags.restype = ctypes.c_int
        self.rt.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        self.rt.cudaMemcpy2DAsync.restype = ctypes.c_int

    def record(self, ev: torch.cuda.Event, stream: torch.cuda.Stream):
        r = self.rt.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event), ctypes.c_void_p(stream.cuda_stream), 1)
        if r != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed: {r}")

    def host_mapped(self, t: torch.Tensor) -> bool:
        """True when kernels can address the pinned host tensor t at its host
        address (unified addressing), checked with cudaHostGetDevicePointer."""
        self.rt.cudaHostGetDevicePointer.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p,
                                                     ctypes.c_uint]
        self.rt.cudaHostGetDevicePointer.restype = ctypes.c_int
        dptr = ctypes.c_void_p()
        r = self.rt.cudaHostGetDevicePointer(ctypes.byref(dptr), ctypes.c_void_p(t.data_ptr()), 0)
        return r == 0 and dptr.value == t.data_ptr()

    def copy_prefix_h2d(self, dst: torch.Tensor, src: torch.Tensor, rows: int, stream: torch.cuda.Stream):
        """Rows [0, rows) of every unit of src [units, max_len, d] (pinned host)
        into dst (same shape, device): one cudaMemcpy2DAsync (a little faster
        than one copy per unit; the host link runs at ~211 GB/s either way)."""
        pitch = src.stride(0) * src.element_size()
        r = self.rt.cudaMemcpy2DAsync(ctypes.c_void_p(dst.data_ptr()), ctypes.c_size_t(dst.stride(0) * dst.element_size()),
                                      ctypes.c_void_p(src.data_ptr()), ctypes.c_size_t(pitch),
                                      ctypes.c_size_t(rows * src.stride(1) * src.element_size()),
                                      ctypes.c_size_t(src.shape[0]), 1, ctypes.c_void_p(stream.cuda_stream))
        if r != 0:
            raise RuntimeError(f"cudaMemcpy2DAsync failed: {r}")

    def copy_prefix_h2d_split(self, dst: torch.Tensor, src: torch.Tensor, rows: int, stream: torch.cuda.Stream,
                              streams, forks, joins):
        """copy_prefix_h2d with the units cut into len(streams) groups, each
        copied on its own stream (forked from and joined back into `stream`),
        so that several copy engines share the host link."""
        n, U = len(streams), src.shape[0]
        forks[0].record(stream)
        for i, st in enumerate(streams):
            u0, u1 = U * i // n, U * (i + 1) // n
            if u0 == u1:
                continue
            st.wait_event(forks[0])
            self.copy_prefix_h2d(dst[u0:u1], src[u0:u1], rows, st)
            joins[i].record(st)
            stream.wait_event(joins[i])

    def copy_rows_h2d(self, dst: torch.Tensor, src: torch.Tensor, stream: torch.cuda.Stream):
        """src [n, w] contiguous pinned host -> dst [n, w] device view with a row
        stride: one cudaMemcpy2DAsync (rows land where the caller's layout wants
        them, no staging copy)."""
        width = src.shape[1] * src.element_size()
        r = self.rt.cudaMemcpy2DAsync(ctypes.c_void_p(dst.data_ptr()), ctypes.c_size_t(dst.stride(0) * dst.element_size()),
                                      ctypes.c_void_p(src.data_ptr()), ctypes.c_size_t(width), ctypes.c_size_t(width),
                                      ctypes.c_size_t(src.shape[0]), 1, ctypes.c_void_p(stream.cuda_stream))
        if r != 0:
            raise RuntimeError(f"cudaMemcpy2DAsync failed: {r}")


# ----------------------------------------------------------------------------- algorithmic bytes
def decode_bytes(w, step: int, C: int, async_incr: bool = False, pend: int | None = None):
    """Algorithmic HBM bytes of decode step `step` for all units: (attention, whole step).
    Attention reads every attended K and V row once (256 B each in bf16, 512
    in fp32) for all g heads, the indices, q, and writes out (fp32).  Scoring
    reads the centroid scoring copy and q; selection reads sizes, offsets and
    the selected perm entries, writes idx and count.  Above 1024 clusters the
    scores also go through memory (written by the scoring kernel, read by the
    selection); up to that the selection CTA scores its own unit and they do
    not.  `pend` overrides the pending tokens of the step."""
    U, g, d, B = w.units, w.g, w.d, w.B
    e = 4 if w.dtype == "f32" else 2
    if pend is None:
        pend = step % w.m + 1
        if async_incr and step >= w.m and step % w.m == 0:
            pend += w.m  # the block being clustered on the side stream is still pending
    rows = w.sinks + pend + B
    attn = U * (rows * 2 * d * e + B * 4 + 4 + g * d * e + g * d * 4)
    scores_through_memory = 2 * C * 4 if C > 1024 else 0
    score = U * (C * d * e + g * d * e)
    select = U * (scores_through_memory + C * 4 + (C + 1) * 4 + B * 4 + B * 4 + 4)
    return attn, attn + score + select


def kmeans_flops_bytes(w):
    """Per prefill clustering of all units: assignment FLOPs (2 n C d per
    iteration) and the two key passes per iteration (assign + update)."""
    n = w.L - w.sinks
    flops = w.iters * w.units * 2.0 * n * w.C * w.d
    byts = w.iters * w.units * (2 * n * w.d * 2 + n * 4 * 4)
    return flops, byts


# ----------------------------------------------------------------------------- our path
class DecodeStep:
    """Issues one decode step of every unit through the public calls on
    stream `s`: the step's new K/V row into the caches, then either
    ckv_decode_step (after the append) or ckv_select + ckv_sparse_decode_attn
    with the append forked onto a side stream: the row is read only by the
    attention, so the append overlaps the scoring and selection and is joined
    before the attention (as a serving loop writes the new token's K/V while
    the query is scored)."""

    def __init__(self, ctx, K, V, B, idx, cnt, out, one_call, s):
        self.ctx, self.K, self.V, self.B = ctx, K, V, B
        self.idx, self.cnt, self.out = idx, cnt, out
        self.one_call, self.s = one_call, s
        self.side = torch.cuda.Stream()
        self.fork, self.join = torch.cuda.Event(), torch.cuda.Event()

    def __call__(self, q, k_row, v_row, pos, cur_len, before_decode=None):
        from recallable_kv_cache_gb300 import ckv
        s = self.s
        if self.one_call:
            ckv.append_kv(k_row, v_row, self.K, self.V, pos, stream=s)
            if before_decode:
                before_decode()
            self.ctx.decode_step(q, self.K, self.V, self.B, cur_len, self.idx, self.cnt, self.out, stream=s)
            return
        self.fork.record(s)
        self.side.wait_event(self.fork)
        ckv.append_kv(k_row, v_row, self.K, self.V, pos, stream=self.side)
        self.join.record(self.side)
        if before_decode:
            before_decode()
        self.ctx.select(q, self.B, self.idx, self.cnt, stream=s)
        s.wait_event(self.join)
        self.ctx.sparse_decode_attn(q, self.K, self.V, self.idx, self.cnt, self.B, cur_len, self.out, stream=s)


def rank_workload(w, rank: int, world: int):
    """Weak scaling: every rank runs the whole workload on its own units (its
    own sequences: a seed of its own); units never cross ranks, so the path
    needs no collective."""
    return synth.scaled(w, seed=w.seed + 1000 * rank) if world > 1 else w


def max_over_ranks(values, world: int, device="cuda"):
    """Element-wise maximum of a list of floats over all ranks (the job ends
    when the slowest rank ends)."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_value(world: int, decode_steps: int, step_ms: float, batch: int = 1) -> float:
    """Whole-job throughput: decode tokens of all ranks (every step decodes one
    token for each of the `batch` sequences) / job time (the max over ranks)."""
    return world * batch * decode_steps / (step_ms / 1000.0)


def run_ours(args, w, rank, world, device):
    from recallable_kv_cache_gb300 import ckv
    torch.cuda.set_device(device)
    w = rank_workload(w, rank, world)
    U, L, B, T = w.units, w.L, w.B, w.decode_steps
    K, V = synth.make_kv(w, device="cuda")
    Q = synth.make_queries(w, T, device="cuda")
    # the K/V row each decode step appends (rows L .. L + T - 1 of the cache,
    # kept apart so that every step really copies its row into the cache)
    Knew, Vnew = K[:, L:L + T].clone(), V[:, L:L + T].clone()
    torch.cuda.synchronize()
    ctx = ckv.Context(units=U, g=w.g, max_len=w.max_len, max_clusters=w.max_clusters, max_budget=B,
                      iters=w.iters, m=w.m, c_plus=w.c_plus)
    if not args.no_l2_persist:
        ctx.set_l2_persistence(-1)  # the tables every step re-reads stay in L2
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    out = torch.empty(U, w.g, w.d, dtype=torch.float32, device="cuda")
    one_call = args.path == "step"

    # eager pass first (validates every call), then capture
    ctx.cluster_prefill(K, L, w.C)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()

    issue_step = DecodeStep(ctx, K, V, B, idx, cnt, out, one_call, s)

    def decode_loop(sync_incremental):
        """Every decode step of the job: append the step's K/V row, cluster the
        last m tokens every m steps (on a side stream overlapping the step,
        committed before the next one; or inline), then the decode step."""
        state = {"commit_at": -1}

        def incremental(t):
            if t > 0 and t % w.m == 0:
                if sync_incremental:
                    ctx.cluster_incremental(K, L + t - w.m, stream=s)
                else:
                    fork.record(s)
                    side.wait_event(fork)
                    ctx.cluster_incremental_begin(K, L + t - w.m, stream=side)
                    state["commit_at"] = t + 1
            if t == state["commit_at"]:
                ctx.cluster_incremental_commit(stream=s)

        for t in range(T):
            issue_step(Q[t], Knew[:, t:t + 1], Vnew[:, t:t + 1], L + t, L + t + 1, lambda: incremental(t))

    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    # per step: append, selection (which scores up to 1024 clusters itself;
    # above that a scoring kernel first), attention, combine (either path);
    # plus one incremental kernel per block
    C_max = w.C + w.c_plus * w.n_incremental
    per_step = 4 if C_max <= 1024 else 5
    launches = {"prefill": 1 + w.iters * 6, "decode": per_step * T + w.n_incremental}
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_pre, stream=s):
            ctx.cluster_prefill(K, L, w.C, stream=s)
        with torch.cuda.graph(g_dec, stream=s):
            decode_loop(args.sync_incremental)
    # clusters visible at step t (an asynchronous clustering begun at step t is
    # committed before step t + 1)
    C_at = [w.C + w.c_plus * ((t // w.m) if args.sync_incremental else max(0, (t - 1) // w.m)) for t in range(T)]
    p0, p1, p2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))

    def one_step(sample):
        with torch.cuda.stream(s):
            p0.record(s)
            g_pre.replay()
            p1.record(s)
            g_dec.replay()
            p2.record(s)
        torch.cuda.synchronize()
        if sample is not None:
            sample["prefill"].append(p0.elapsed_time(p1))
            sample["decode"].append(p1.elapsed_time(p2))

    for _ in range(args.warmup):
        one_step(None)
    assert ctx.device_error() == 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    smi_index = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[device] if os.environ.get(
        "CUDA_VISIBLE_DEVICES") else device
    clk = ClockSampler(smi_index)
    clk.start()
    time.sleep(0.3)
    sample = {"prefill": [], "decode": []}
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        one_step(sample)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    err = ctx.device_error()
    if err:
        raise RuntimeError(f"device error {err} during the timed region")

    step_ms = [a + b for a, b in zip(sample["prefill"], sample["decode"])]
    res = dict(step_ms=sum(step_ms) / len(step_ms), prefill_ms=statistics.mean(sample["prefill"]),
               decode_ms=statistics.mean(sample["decode"]), wall_s=wall, clocks=clocks,
               launches=(launches["prefill"] + launches["decode"]) * args.steps)
    ai = not args.sync_incremental
    res["one_call"] = one_call
    res["decode_bytes_per_step"] = sum(decode_bytes(w, t, C_at[t], ai)[1] for t in range(T)) / T
    res["step_timing"] = time_decode_steps(ctx, w, K, V, Q, Knew, Vnew, one_call)
    if w.n_incremental > 0 and not args.sync_incremental:
        res["async_clustering"] = hidden_clustering(ctx, w, K, g_pre, g_dec, decode_loop, s,
                                                    statistics.mean(sample["decode"]))
    res["assign_ms"] = time_assign(ctx, w, K)
    res["recall"] = selection_recall(lambda q, i, c: ctx.select(q, w.B, i, c), w, K, Q)
    if not args.no_comparators:
        res["reuse"] = selection_reuse(ctx, w)
        res["quest"] = quest_comparator(w, K, V, Q)
        res["channel_prescore"] = channel_prescore_comparator(w, K, Q)
        res["full_kv"] = full_kv_attention(w, K, V, Q)
    res["w"] = w
    res["ctx"] = ctx
    res["tensors"] = (K, V, Q)
    if not args.no_e2e:
        res["e2e"] = run_e2e(ctx, w, K, V, Q, one_call, args.sync_incremental, args.upload_streams,
                             args.e2e_copy_nodes, not args.e2e_out_copies)
    return res


def time_decode_steps(ctx, w, K, V, Q, Knew, Vnew, one_call, n=64, p_first=129, reps=5):
    """The decode step timed on its own: `n` consecutive steps (append, then
    the decode step) with p_first .. p_first + n - 1 pending tokens (around the
    job's mean of ~160) over the prompt clusters, captured in one CUDA graph
    with no event inside; CUDA events around `reps` whole replays give the
    time per step.  For the per-kernel path the attention (+ combine) launch
    is also timed alone the same way (a graph of n attention launches)."""
    from recallable_kv_cache_gb300 import ckv
    U, L, B = w.units, w.L, w.B
    ctx.cluster_prefill(K, L, w.C)  # back to the prompt clusters
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    out = torch.empty(U, w.g, w.d, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    T = w.decode_steps
    n = max(1, min(n, T))
    p_first = max(1, min(p_first, T - n + 1))  # short jobs: the steps that exist
    steps = [(p_first + i - 1, L + p_first + i) for i in range(n)]  # (row appended, cur_len)

    issue = DecodeStep(ctx, K, V, B, idx, cnt, out, one_call, s)

    def step(t, row, cur):
        issue(Q[t], Knew[:, row:row + 1], Vnew[:, row:row + 1], L + row, cur)

    def timed(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            body()  # eager once: validates the calls
            with torch.cuda.graph(g, stream=s):
                body()
            for _ in range(3):
                g.replay()
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return 1000.0 * e0.elapsed_time(e1) / (reps * n)

    step_us = timed(lambda: [step(i, row, cur) for i, (row, cur) in enumerate(steps)])
    byts = statistics.mean(decode_bytes(w, row, w.C)[1] for row, _ in steps)
    append_b = U * 2 * w.d * 2 * 2  # the new K and V rows: read and written
    res = {"step_us": step_us, "bytes_per_step": byts + append_b, "pending": [steps[0][0] + 1, steps[-1][0] + 1],
           "what": f"{n} decode steps (append + " + ("ckv_decode_step" if one_call else
                                                        "ckv_select + ckv_sparse_decode_attn") +
                   f") with {steps[0][0] + 1}..{steps[-1][0] + 1} pending tokens in one graph, "
                   f"{reps} replays between two CUDA events"}
    if not one_call:
        ctx.select(Q[0], B, idx, cnt, stream=s)
        cur = L + p_first + n // 2
        res["attn_us"] = timed(lambda: [ctx.sparse_decode_attn(Q[i], K, V, idx, cnt, B, cur, out, stream=s)
                                        for i in range(n)])
        res["attn_bytes"] = decode_bytes(w, cur - L - 1, w.C)[0]
    return res


def hidden_clustering(ctx, w, K, g_pre, g_dec, decode_loop, s, async_ms, reps=2):
    """What the side stream saves: the same decode loop with the clustering
    inline (a graph of its own) against the asynchronous one, beside the
    clustering kernel's own time (one incremental clustering of every unit,
    warm, timed alone).  saved_ms = inline - async; saved_per_clustering_ms =
    saved / blocks, to compare with clustering_ms (it can exceed it: inline,
    the clustering also breaks the decode kernels' dependent-launch chain)."""
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(3):
        ctx.cluster_prefill(K, w.L, w.C, stream=s)
        with torch.cuda.stream(s):
            e0.record(s)
            ctx.cluster_incremental(K, w.L, stream=s)
            e1.record(s)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    incr_ms = min(ts[1:])
    ctx.cluster_prefill(K, w.L, w.C)
    g_sync = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_sync, stream=s):
            decode_loop(True)
        g_pre.replay()
        g_sync.replay()
        ts = []
        for _ in range(reps):
            g_pre.replay()
            e0.record(s)
            g_sync.replay()
            e1.record(s)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
    sync_ms = statistics.mean(ts)
    blocks = w.n_incremental
    return {"decode_ms_async": async_ms, "decode_ms_inline": sync_ms, "clustering_ms": incr_ms,
            "blocks": blocks, "saved_ms": sync_ms - async_ms, "saved_per_clustering_ms": (sync_ms - async_ms) / blocks,
            "what": "decode loop with the incremental clustering inline vs on a side stream; clustering_ms = one "
                    "incremental clustering of every unit timed alone (warm)"}


def time_assign(ctx, w, K, reps=5):
    """The tensor-core assignment kernel timed alone (outside the timed job):
    one K-means assignment pass over every unit's prompt keys against the
    prefill centroids, CUDA events on the launching stream."""
    ctx.cluster_prefill(K, w.L, w.C)  # back to the prefill clusters (C of the prompt)
    lab = torch.empty(w.units, w.L - w.sinks, dtype=torch.int32, device="cuda")
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        ctx.kmeans_assign(K, w.L, lab)
    torch.cuda.synchronize()
    a0.record()
    for _ in range(reps):
        ctx.kmeans_assign(K, w.L, lab)
    a1.record()
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / reps


def selection_recall(select, w, K, Q, units=(0, 97, 201), queries=(0, 1, 2), what="prefill clusters"):
    """Recall of a selection against the exact top-B tokens by sum_h q_h . k
    (a measurement, not part of the path): token recall |S n TopB| / B and
    attention-mass recall sum_S a / sum_TopB a, a = the full softmax over the
    clustered prompt tokens averaged over the g heads.  `select(q, idx, cnt)`
    runs the library's selection for every unit."""
    units = [u for u in units if u < w.units] or [0]
    idx = torch.empty(w.units, w.B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    tok, mass = [], []
    for qi in queries:
        q = Q[qi]
        select(q, idx, cnt)
        torch.cuda.synchronize()
        for u in units:
            keys = K[u, w.sinks:w.L].float()
            qu = q[u].float()                                        # [g, d]
            logits = qu @ keys.T / (w.d ** 0.5)                      # [g, n]
            a = torch.softmax(logits, dim=1).mean(0)                 # [n]
            top = torch.topk((qu.sum(0) @ keys.T), w.B).indices
            sel = idx[u, :int(cnt[u])].long() - w.sinks
            inter = torch.isin(sel, top).sum().item()
            tok.append(inter / w.B)
            mass.append((a[sel].sum() / a[top].sum()).item())
    return {"token": statistics.mean(tok), "attention_mass": statistics.mean(mass),
            "sample": f"{len(units)} units x {len(queries)} queries, {what}, B={w.B}"}


def selection_reuse(ctx, w, steps=64):
    """Hit rate of a cache of the last R steps' selections (the ClusterKV
    page's cluster-granular cache of selected KV; a measurement, not part of
    the path): tokens of a step's selection already selected in one of the R
    previous steps, over all tokens selected, for R = 1 and 2, on two query
    streams of the same units: a new topic every step (the bench's stream)
    and one topic held for the whole sample (fresh noise every step)."""
    from recallable_kv_cache_gb300 import ckv
    U, B = w.units, w.B
    res = {}
    for name, run in (("new_topic_every_step", 1), ("topic_held", steps)):
        Qr = synth.make_queries(w, steps, device="cuda", topic_run=run)
        hi = [torch.empty(U, B, dtype=torch.int32, device="cuda") for _ in range(steps)]
        hc = [torch.empty(U, dtype=torch.int32, device="cuda") for _ in range(steps)]
        for t in range(steps):
            ctx.select(Qr[t], B, hi[t], hc[t])
        hits = torch.empty(U, dtype=torch.int32, device="cuda")
        rates = {}
        for R in (1, 2):
            hs, ns = 0, 0
            for t in range(R, steps):
                ckv.selection_overlap([(hi[t - r], hc[t - r]) for r in range(1, R + 1)], hi[t], hc[t], hits,
                                      w.max_len)
                hs += int(hits.sum())
                ns += int(hc[t].sum())
            rates[f"R{R}"] = hs / max(ns, 1)
        res[name] = rates
    sel_bytes = U * B * 2 * w.d * 2
    res["offload_h2d_bytes_saved_per_step"] = {k: v["R1"] * sel_bytes for k, v in res.items()}
    res["sample"] = f"{steps} decode steps x {U} units, clusters of the current state, B={B}"
    res["on_gpu"] = ("no HBM bytes saved: every K/V row is resident and each selected row is read once either "
                     "way; the hit rate prices the host-to-device bytes an offloaded cache would skip")
    return res


def quest_comparator(w, K, V, Q, steps=64):
    """The page-granular comparator (Quest) on the same units, budget and
    queries: page bounds of the prompt (pages of 16 tokens), then per step the
    page weights, the selection of whole pages and the same attention kernel,
    captured in a graph of `steps` steps (one pending token) and timed; and
    its recall, measured like the cluster selection's."""
    from recallable_kv_cache_gb300 import ckv
    U, L, B, sinks = w.units, w.L, w.B, w.sinks
    n = L - sinks
    P = (n + 15) // 16
    pmax = torch.empty(U, P, w.d, dtype=K.dtype, device="cuda")
    pmin = torch.empty_like(pmax)
    scores = torch.empty(U, P, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ckv.quest_pages(K, L, pmax, pmin)
    e0.record()
    ckv.quest_pages(K, L, pmax, pmin)
    e1.record()
    torch.cuda.synchronize()
    build_ms = e0.elapsed_time(e1)
    pctx = ckv.Context(units=U, g=w.g, max_len=w.max_len, max_clusters=P, max_budget=B, iters=1, m=w.m,
                       c_plus=w.c_plus)
    sizes = torch.full((U, P), 16, dtype=torch.int32, device="cuda")
    sizes[:, -1] = n - 16 * (P - 1)
    offs = torch.zeros(U, P + 1, dtype=torch.int32, device="cuda")
    offs[:, 1:] = torch.cumsum(sizes, dim=1)
    perm = torch.arange(sinks, L, dtype=torch.int32, device="cuda").expand(U, n).contiguous()
    pctx.import_clusters(P, L, torch.zeros(U, P, w.d, device="cuda"), sizes, offs, perm)

    def select(q, idx, cnt):
        ckv.quest_score(q, pmax, pmin, scores)
        pctx.select_scored(scores, B, idx, cnt)

    recall = selection_recall(select, w, K, Q, what="pages of 16 tokens")
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    out = torch.empty(U, w.g, w.d, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for t in range(2):
            select(Q[t], idx, cnt)
            pctx.sparse_decode_attn(Q[t], K, V, idx, cnt, B, L + 1, out)
        with torch.cuda.graph(g, stream=s):
            for t in range(steps):
                select(Q[t], idx, cnt)
                pctx.sparse_decode_attn(Q[t], K, V, idx, cnt, B, L + 1, out)
        g.replay()
        e0.record(s)
        for _ in range(3):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    step_us = 1000.0 * e0.elapsed_time(e1) / (3 * steps)
    pctx.close()
    return {"step_us": step_us, "page_bounds_ms": build_ms, "recall": recall,
            "metadata_bytes_per_step": U * P * 2 * w.d * K.element_size(),
            "what": "Quest-style pages of 16 tokens: per-channel max / min keys, weight = upper bound of q.k "
                    "summed over the heads; whole pages up to B; same attention kernel; one pending token"}


def channel_prescore_comparator(w, K, Q, steps=64, rs=(8, 16)):
    """TailorKV-style channel pre-score as the centroid scorer (an alternative
    cheap scorer, a comparator): the same prefill clusters, per step the r
    critical channels of |sum_h q_h| * max_c |mu_c| and the scores over them,
    then the same cluster selection.  Reports the selection time per step
    (scoring + selection, a graph of `steps` steps) beside the exact scorer's,
    and the recall of each, measured like the main recall."""
    from recallable_kv_cache_gb300 import ckv
    U, L, B = w.units, w.L, w.B
    tctx = ckv.Context(units=U, g=w.g, max_len=w.max_len, max_clusters=w.max_clusters, max_budget=B,
                       iters=w.iters, m=w.m, c_plus=w.c_plus)
    tctx.cluster_prefill(K, L, w.C)
    muT = torch.empty(U, w.d, w.max_clusters, dtype=K.dtype, device="cuda")
    chmax = torch.empty(U, w.d, dtype=torch.float32, device="cuda")
    tctx.centroid_channels(muT, chmax)
    scores = torch.empty(U, w.C, dtype=torch.float32, device="cuda")
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(select):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            for t in range(2):
                select(Q[t], idx, cnt)
            with torch.cuda.graph(g, stream=s):
                for t in range(steps):
                    select(Q[t], idx, cnt)
            g.replay()
            e0.record(s)
            for _ in range(3):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return 1000.0 * e0.elapsed_time(e1) / (3 * steps)

    exact = lambda q, i, c: tctx.select(q, B, i, c)
    res = {"exact": {"select_us": timed(exact),
                     "recall": selection_recall(exact, w, K, Q, what="exact centroid scores")}}
    for r in rs:
        def pre(q, i, c, r=r):
            tctx.channel_prescore(q, muT, chmax, r, scores)
            tctx.select_scored(scores, B, i, c)
        res[f"r{r}"] = {"select_us": timed(pre),
                        "recall": selection_recall(pre, w, K, Q, what=f"{r} critical channels"),
                        "centroid_bytes_per_step": U * r * w.C * K.element_size()}
    e0.record()
    tctx.centroid_channels(muT, chmax)
    e1.record()
    torch.cuda.synchronize()
    res["channel_copy_ms"] = e0.elapsed_time(e1)
    res["what"] = ("scores over the r channels of largest |sum_h q_h,i| * max_c |mu_c,i| from a channel-major "
                   "centroid copy (rebuilt when the clusters change), then the same selection")
    tctx.close()
    return res


def full_kv_attention(w, K, V, Q, reps=5):
    """Comparator: the same attention kernel over every token (B = L - sinks,
    all prompt tokens selected) for all units, timed alone with CUDA events."""
    from recallable_kv_cache_gb300 import ckv
    n = w.L - w.sinks
    fctx = ckv.Context(units=w.units, g=w.g, max_len=w.L, max_clusters=1, max_budget=n, iters=1,
                       m=w.m, c_plus=w.c_plus)
    idx = torch.arange(w.sinks, w.L, dtype=torch.int32, device="cuda").expand(w.units, n).contiguous()
    cnt = torch.full((w.units,), n, dtype=torch.int32, device="cuda")
    out = torch.empty(w.units, w.g, w.d, dtype=torch.float32, device="cuda")
    # one cluster holding the whole prompt, so that every prompt token counts as
    # clustered and none as pending
    mu = torch.zeros(w.units, 1, w.d, dtype=torch.float32, device="cuda")
    sizes = torch.full((w.units, 1), n, dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, n], dtype=torch.int32, device="cuda").expand(w.units, 2).contiguous()
    fctx.import_clusters(1, w.L, mu, sizes, offs, idx)
    Kp, Vp = K[:, :w.L].contiguous(), V[:, :w.L].contiguous()
    for _ in range(3):
        fctx.sparse_decode_attn(Q[0], Kp, Vp, idx, cnt, n, w.L, out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for r in range(reps):
        fctx.sparse_decode_attn(Q[r + 1], Kp, Vp, idx, cnt, n, w.L, out)
    e1.record()
    torch.cuda.synchronize()
    fctx.close()
    us = 1000.0 * e0.elapsed_time(e1) / reps
    byts = w.units * (w.L * 2 * w.d * 2 + n * 4)
    return {"attention_us": us, "gbs": byts / (us / 1e6) / 1e9,
            "what": "attention over all L tokens of every unit with the same kernel (idx = every prompt token)"}


def run_e2e(ctx, w, K, V, Q, one_call=False, sync_incremental=False, upload_streams=K_UPLOAD_STREAMS,
            copy_nodes=False, out_direct=True):
    """The same job through the public API from pinned host buffers: upload the
    prompt K/V, prefill clustering, then per decode step upload q and the new
    K/V row of every unit, select, attend, and read the output back.  The calls
    are recorded once into a CUDA graph, as a serving loop would, and the timed
    region replays it: every copy and kernel of the job runs inside it.
    Dependencies are those of a real decode loop: the V upload overlaps the
    clustering (which reads K only) after K's.  Where the device maps pinned
    host memory (unified addressing) the step's kernels read q and the new K/V
    rows from it (ckv_append_kv puts the rows into the caches); otherwise a
    step's q and new K and V rows are copied in parallel when the step starts
    (the rows straight into the caches by strided copies).  The output is read
    back on a side stream while the next step runs (two device buffers), or
    with out_direct written by the attention straight into pinned host memory."""
    from recallable_kv_cache_gb300 import ckv
    U, L, B, T, d, g = w.units, w.L, w.B, w.decode_steps, w.d, w.g
    Kh = torch.empty(U, w.max_len, d, dtype=K.dtype, pin_memory=True)
    Vh = torch.empty_like(Kh, pin_memory=True)
    Kh.copy_(K)
    Vh.copy_(V)
    # per step, one packed host record: q [U, g, d] | new K row [U, d] | new V row [U, d]
    nq, nr = U * g * d, U * d
    inp_h = torch.empty(T, nq + 2 * nr, dtype=K.dtype, pin_memory=True)
    inp_h[:, :nq].copy_(Q[:T].reshape(T, nq))
    inp_h[:, nq:nq + nr].copy_(K[:, L:L + T].transpose(0, 1).reshape(T, nr))
    inp_h[:, nq + nr:].copy_(V[:, L:L + T].transpose(0, 1).reshape(T, nr))
    outh = torch.empty(T, U, g, d, dtype=torch.float32, pin_memory=True)
    Kd = torch.empty_like(K)
    Vd = torch.empty_like(V)
    qd = torch.empty(U, g, d, dtype=Q.dtype, device="cuda")
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    outs = [torch.empty(U, g, d, dtype=torch.float32, device="cuda") for _ in range(2)]
    s, side, up, dn, sk, sv = (torch.cuda.Stream() for _ in range(6))
    e_fork, e_v = torch.cuda.Event(), torch.cuda.Event()
    k_streams = [torch.cuda.Stream() for _ in range(max(1, upload_streams))]
    k_forks, k_joins = [torch.cuda.Event()], [torch.cuda.Event() for _ in k_streams]
    e_step = [torch.cuda.Event() for _ in range(T)]
    e_k = [torch.cuda.Event() for _ in range(T)]
    e_vr = [torch.cuda.Event() for _ in range(T)]
    e_out = [torch.cuda.Event() for _ in range(T)]
    e_read = [torch.cuda.Event() for _ in range(T)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:  # torch creates the CUDA event on first record
        e.record(s)
    ext = ExternalEvents()  # captured records become timing nodes
    # on unified-addressing systems (Grace: the C2C link) the kernels can read
    # and write pinned host memory directly, which saves the per-step copy nodes
    zero_copy = not copy_nodes and ext.host_mapped(inp_h) and ext.host_mapped(outh)
    torch.cuda.synchronize()
    # the host link as this machine gives it: one 1 GiB copy from pinned memory
    n_probe = min(Kh.numel(), (1 << 30) // Kh.element_size())
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(2):
            p0.record(s)
            Kd.view(-1)[:n_probe].copy_(Kh.view(-1)[:n_probe], non_blocking=True)
            p1.record(s)
    torch.cuda.synchronize()
    link_gbs = n_probe * Kh.element_size() / (p0.elapsed_time(p1) / 1e3) / 1e9

    def job():
        ext.record(ev[0], s)
        ext.copy_prefix_h2d_split(Kd, Kh, L, s, k_streams, k_forks, k_joins)
        ext.record(ev[1], s)
        # V is not read before the first decode step: its upload follows K's
        # (the two would share the link) and overlaps the clustering
        e_fork.record(s)
        up.wait_event(e_fork)
        ext.copy_prefix_h2d(Vd, Vh, L, up)
        e_v.record(up)
        ctx.cluster_prefill(Kd, L, w.C)
        ext.record(ev[2], s)
        s.wait_event(e_v)
        state = {"commit_at": -1}

        def incremental(t):
            if t > 0 and t % w.m == 0:
                if sync_incremental:
                    ctx.cluster_incremental(Kd, L + t - w.m)
                else:
                    e_fork.record(s)
                    side.wait_event(e_fork)
                    ctx.cluster_incremental_begin(Kd, L + t - w.m, stream=side)
                    state["commit_at"] = t + 1
            if t == state["commit_at"]:
                ctx.cluster_incremental_commit(stream=s)

        def decode(t, q, out):
            if one_call:
                ctx.decode_step(q, Kd, Vd, B, L + t + 1, idx, cnt, out)
            else:
                ctx.select(q, B, idx, cnt)
                ctx.sparse_decode_attn(q, Kd, Vd, idx, cnt, B, L + t + 1, out)

        def out_buffer(t):
            """Where step t's attention writes: the host record itself, or a
            device buffer (two in turn) read back on a side stream while the
            next step runs."""
            if zero_copy and out_direct:
                return outh[t]
            if t >= 2:
                s.wait_event(e_read[t - 2])  # that buffer's read-back is done
            return outs[t % 2]

        def read_back(t, out):
            if zero_copy and out_direct:
                return
            e_out[t].record(s)
            dn.wait_event(e_out[t])
            with torch.cuda.stream(dn):
                outh[t].copy_(out, non_blocking=True)
                e_read[t].record(dn)

        for t in range(T):
            if zero_copy:
                # the kernels read this step's q and new K/V rows from pinned host
                # memory.  The rows are read only by the attention: with separate
                # calls they are appended on a side stream while the scoring and
                # selection run
                q, kh, vh = inp_h[t, :nq].view(U, g, d), inp_h[t, nq:nq + nr].view(U, d), inp_h[t, nq + nr:].view(U, d)
                out = out_buffer(t)
                if one_call:
                    ckv.append_kv(kh, vh, Kd, Vd, L + t, stream=s)
                    incremental(t)
                    decode(t, q, out)
                    read_back(t, out)
                    continue
                e_step[t].record(s)
                sk.wait_event(e_step[t])
                ckv.append_kv(kh, vh, Kd, Vd, L + t, stream=sk)
                e_k[t].record(sk)
                incremental(t)
                ctx.select(q, B, idx, cnt)
                s.wait_event(e_k[t])
                ctx.sparse_decode_attn(q, Kd, Vd, idx, cnt, B, L + t + 1, out)
                read_back(t, out)
                continue
            # the step's three inputs in parallel: q, and the new K and V rows
            # straight into their place in the caches (one strided copy each)
            e_step[t].record(s)
            sk.wait_event(e_step[t])
            ext.copy_rows_h2d(Kd[:, L + t], inp_h[t, nq:nq + nr].view(U, d), sk)
            e_k[t].record(sk)
            sv.wait_event(e_step[t])
            ext.copy_rows_h2d(Vd[:, L + t], inp_h[t, nq + nr:].view(U, d), sv)
            e_vr[t].record(sv)
            qd.view(-1).copy_(inp_h[t, :nq], non_blocking=True)
            s.wait_event(e_k[t])
            s.wait_event(e_vr[t])
            incremental(t)
            out = out_buffer(t)
            decode(t, qd, out)
            read_back(t, out)
        if not (zero_copy and out_direct):
            s.wait_event(e_read[T - 1])
        ext.record(ev[3], s)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            job()
        graph.replay()  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    phases = {"upload_k_ms": ev[0].elapsed_time(ev[1]), "prefill_ms": ev[1].elapsed_time(ev[2]),
              "decode_ms": ev[2].elapsed_time(ev[3])}
    h2d = 2 * U * L * d * 2 + T * (nq + 2 * nr) * 2
    d2h = T * U * g * d * 4
    return {"value": w.batch * T / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "job_s": dt, "phases_ms": {k: round(v, 3) for k, v in phases.items()},
            "host_link_h2d_gbs": round(link_gbs, 1), "upload_streams": len(k_streams),
            "how": "public API calls recorded once into a CUDA graph and replayed; the prompt K/V, every "
                   "step's q and new K/V rows come from pinned host memory and every step's output goes "
                   "back to it inside the timed replay (V upload overlapping the clustering; " +
                   ("the step's kernels read q and the new rows from pinned host memory" if zero_copy else
                    "the step's three input copies in parallel") +
                   ("; the attention writes the output there" if zero_copy and out_direct else
                    "; outputs read back while the next step runs") + ")",
            "step_io": ("zero-copy inputs (kernels read pinned host memory)" if zero_copy else "copy nodes") +
                       (", zero-copy outputs" if zero_copy and out_direct else ", output copies")}


# ----------------------------------------------------------------------------- the other workloads
OTHER_WORKLOADS = ("tiny_2k", "layer_32k", "batch16_32k", "long_128k")


def measure_workload(name, hbm, reps=2, l2_persist=True):
    """One of the other workloads on this GPU, beside the main line:
    prefill clustering of every unit (CUDA events, after a warm-up run) and
    K-means ms per layer; for the decode loops (batch16_32k, long_128k) the
    whole decode loop of the job as one CUDA graph (append the step's K/V row,
    selection, attention) and its roofline; for the single-step workloads
    (tiny_2k: 8 independent queries of one fp32 head; layer_32k: one step of a
    layer) the latency of a decode step.  Inputs generated on the device."""
    from recallable_kv_cache_gb300 import ckv
    w = synth.WORKLOADS[name]
    U, L, B = w.units, w.L, w.B
    T = max(w.decode_steps, 1)
    K, V = synth.make_kv(w, device="cuda")
    Q = synth.make_queries(w, w.n_queries if w.decode_steps == 0 else T, device="cuda")
    ctx = ckv.Context(units=U, g=w.g, max_len=w.max_len, max_clusters=w.max_clusters, max_budget=B,
                      kv_dtype=w.dtype, iters=w.iters, m=w.m, c_plus=w.c_plus)
    if l2_persist:
        ctx.set_l2_persistence(-1)
    s = torch.cuda.Stream()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    res = {"units": U, "L": L, "B": B, "C": w.C, "dtype": w.dtype}
    with torch.cuda.stream(s):
        ctx.cluster_prefill(K, L, w.C, stream=s)
        ts = []
        for _ in range(reps):
            e0.record(s)
            ctx.cluster_prefill(K, L, w.C, stream=s)
            e1.record(s)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
    prefill_ms = statistics.mean(ts)
    res["prefill_ms"] = prefill_ms
    res["kmeans_ms_per_layer"] = prefill_ms * w.kv_heads * w.batch / U
    kflops, _ = kmeans_flops_bytes(w)
    res["kmeans_tflops"] = kflops / (prefill_ms / 1000.0) / 1e12
    idx = torch.empty(U, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(U, dtype=torch.int32, device="cuda")
    out = torch.empty(U, w.g, w.d, dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    if w.decode_steps > 0:
        Knew, Vnew = K[:, L:L + T].clone(), V[:, L:L + T].clone()

        def body():
            for t in range(T):
                ckv.append_kv(Knew[:, t:t + 1], Vnew[:, t:t + 1], K, V, L + t, stream=s)
                ctx.decode_step(Q[t], K, V, B, L + t + 1, idx, cnt, out, stream=s)
        steps = T
    else:
        n_q = Q.shape[0]

        def body():
            for i in range(64):
                ctx.decode_step(Q[i % n_q], K, V, B, L, idx, cnt, out, stream=s)
        steps = 64
    with torch.cuda.stream(s):
        body()
        with torch.cuda.graph(g, stream=s):
            body()
        g.replay()
        ts = []
        for _ in range(reps):
            e1.record(s)
            g.replay()
            e2.record(s)
            torch.cuda.synchronize()
            ts.append(e1.elapsed_time(e2))
    assert ctx.device_error() == 0
    step_us = 1000.0 * statistics.mean(ts) / steps
    byts = (statistics.mean(decode_bytes(w, t, w.C)[1] for t in range(T)) if w.decode_steps > 0
            else decode_bytes(w, 0, w.C, pend=0)[1])
    if w.decode_steps > 0:
        byts += U * 2 * w.d * (4 if w.dtype == "f32" else 2) * 2  # the appended row, read and written
        job_ms = prefill_ms + statistics.mean(ts)
        res["tokens_per_s"] = w.batch * T / (job_ms / 1000.0)
        res["decode_tokens_per_s"] = w.batch * T / (statistics.mean(ts) / 1000.0)
        res["job_ms"] = job_ms
        res["what"] = (f"whole job: prefill clustering + {T} decode steps (append + ckv_decode_step) as one graph; "
                       "no incremental clustering in this workload")
    else:
        res["what"] = (f"one decode step (ckv_decode_step: scoring, selection, attention) over the prompt, "
                       f"{w.n_queries} different queries cycled, 64 steps per graph replay")
    gbs = byts / (step_us / 1e6) / 1e9
    res["decode_step_us"] = step_us
    res["decode_roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                              "bytes_per_step": byts}
    ctx.close()
    del K, V, Q
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- the oracle on the CPU
def oracle_jobs(w, n_units=None, device_tensors=None):
    """The C++ oracle (float64, oracle/clusterkv_ref.cpp) on whole jobs of the
    first n_units units (default: one per host core), all at once on a pool of
    std::threads (one unit per thread): prefill clustering, then every decode
    step (incremental clustering every m steps, score, select, sparse
    attention).  Units are independent, so the workload's job time is the
    measured wall time times units / n_units (an extrapolation, stated)."""
    import oracle.cpp as cc
    threads = os.cpu_count() or 1
    n_units = min(w.units, n_units or threads)
    units = list(range(n_units))
    T = w.decode_steps
    if device_tensors is not None:
        K, V, Q = device_tensors
        Ks = [K[u].double().cpu().numpy() for u in units]
        Vs = [V[u].double().cpu().numpy() for u in units]
        Qs = [Q[:T, u].double().cpu().numpy() for u in units]
    else:
        Kt, Vt = synth.make_kv(w, units=units)
        Qt = synth.make_queries(w, T, units=units)
        Ks = [Kt[i].double().numpy() for i in range(n_units)]
        Vs = [Vt[i].double().numpy() for i in range(n_units)]
        Qs = [Qt[:, i].double().numpy() for i in range(n_units)]
    operand = "bf16" if w.dtype == "bf16" else "f64"

    def run():
        t0 = time.perf_counter()
        _, times = cc.unit_jobs(Ks, Vs, Qs, w.L, w.C, w.B, iters=w.iters, m=w.m, c_plus=w.c_plus, sinks=w.sinks,
                                operand=operand, threads=threads)
        wall = time.perf_counter() - t0
        job_s = wall * w.units / n_units
        return {"wall_s": wall, "job_s": job_s, "tokens_per_s": w.batch * T / job_s,
                "prefill_s_per_unit": float(times[:, 0].mean()), "decode_s_per_unit": float(times[:, 1].mean())}

    return run, n_units, min(threads, n_units)


def cpu_threads():
    """Threads of the BLAS pool numpy would use (reported beside the core count)."""
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.WORKLOADS[args.workload]
    if args.units:
        w = synth.scaled(w, units=args.units)
    if args.decode_steps:
        w = synth.scaled(w, decode_steps=args.decode_steps)
    cfg = {"workload": f"{w.name}: {w.layers} layers x {w.kv_heads} KV heads x batch {w.batch} "
                       f"({w.units} units), d={w.d}, GQA {w.g}, prompt L={w.L}, {w.decode_steps} decode "
                       f"steps, B={w.B}, C={w.C} + {w.c_plus} every {w.m} steps, {w.iters} Lloyd iterations",
           "units": w.units, "L": w.L, "decode_steps": w.decode_steps, "B": w.B, "C": w.C,
           "path": ("ckv_append_kv, then ckv_decode_step" if args.path == "step" else
                    "ckv_append_kv on a side stream (joined before the attention) beside ckv_select, "
                    "then ckv_sparse_decode_attn"),
           "incremental": "inline before the step" if args.sync_incremental else
                          "side stream: begun at the step, overlapping it; committed before the next step",
           "l2": (f"inputs larger than L2: {2 * w.units * w.max_len * w.d * 2 / 1e9:.1f} GB of K/V and "
                  f"{w.decode_steps * w.units * w.g * w.d * 2 / 1e6:.0f} MB of queries resident; a decode step "
                  f"gathers ~{decode_bytes(w, w.decode_steps // 2, w.C, True)[0] / 1e6:.0f} MB of scattered rows "
                  f"(L2 is 129 MB); no flush" +
                  ("" if args.no_l2_persist else
                   "; the centroid scoring copy and perm, which every step re-reads, in a persisting L2 "
                   "set-aside (ckv_set_l2_persistence)"))}

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: the C++ oracle on the whole jobs of one unit per host core,
        # run at once and timed as they run; the workload's job time is that
        # wall time times units / sampled units (reported as an extrapolation)
        run, n_units, threads = oracle_jobs(w)
        runs = [run() for _ in range(args.warmup + args.steps)][args.warmup:]
        sample_desc = (f"{n_units} units' whole jobs per step (prefill clustering of {w.L - w.sinks} keys + "
                       f"{w.decode_steps} decode steps each), one unit per thread, extrapolated "
                       f"x{w.units}/{n_units} units")
        v = statistics.mean(r["tokens_per_s"] for r in runs)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000 * statistics.mean(r["wall_s"] for r in runs),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "extrapolated_job_s": statistics.mean(r["job_s"] for r in runs),
                "kmeans_ms_per_layer": 1000 * statistics.mean(r["prefill_s_per_unit"] for r in runs) * w.kv_heads
                                       * w.batch,
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "host_cores": os.cpu_count(),
                                 "kind": "oracle (C++, float64, std::thread pool)", "sample": sample_desc},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    r = run_ours(args, w, rank, world, local)
    w = r["w"]
    hbm, peak_kind, meas = peaks()
    step_ms, prefill_ms, decode_ms = r["step_ms"], r["prefill_ms"], r["decode_ms"]
    step_ms, prefill_ms, decode_ms = max_over_ranks([step_ms, prefill_ms, decode_ms], world)
    T = w.decode_steps
    value = job_value(world, T, step_ms, w.batch)
    # the decode step over the timed region: the job's algorithmic bytes per
    # step (scoring, selection, gather + attention, the appended row) over the
    # mean step time (CUDA events on the decode stream around the replay of
    # the whole decode loop, which holds no event of its own)
    append_b = w.units * 2 * w.d * 2 * 2
    step_bytes = r["decode_bytes_per_step"] + append_b
    step_us = 1000.0 * decode_ms / T
    decode_gbs = step_bytes / (step_us / 1e6) / 1e9
    kernels = ("append_kv_kernel + sel_kernel (scoring and selection) + attn_mma_kernel + attn_mma_combine_kernel "
               "(ckv_append_kv + " + ("ckv_decode_step)" if r["one_call"] else
                                      "ckv_select + ckv_sparse_decode_attn)"))
    traffic_ratio = STEP_TRAFFIC_PER_ALG_BYTE
    roofline = {"bound": "hbm", "kernel": kernels, "achieved": decode_gbs, "peak": hbm, "unit": "GB/s",
                "frac": decode_gbs / hbm, "traffic": traffic_ratio * step_bytes if traffic_ratio else None,
                "traffic_source": STEP_TRAFFIC_SOURCE,
                "bytes_per_launch": step_bytes, "launch_us": step_us, "peak_kind": peak_kind,
                "timing": "mean decode step of the timed region: CUDA events around each replay of the "
                          f"{T}-step decode graph (incremental clustering included), on the decode stream"}
    st = r["step_timing"]
    iso_gbs = st["bytes_per_step"] / (st["step_us"] / 1e6) / 1e9
    isolated = {"achieved": iso_gbs, "peak": hbm, "unit": "GB/s", "frac": iso_gbs / hbm,
                "bytes_per_step": st["bytes_per_step"], "step_us": st["step_us"], "pending": st["pending"],
                "timing": st["what"]}
    if "attn_us" in st:
        a_gbs = st["attn_bytes"] / (st["attn_us"] / 1e6) / 1e9
        isolated["attention_alone"] = {"kernel": "attn_mma_kernel + attn_mma_combine_kernel", "us": st["attn_us"],
                                       "bytes": st["attn_bytes"], "achieved": a_gbs, "frac": a_gbs / hbm}
    kflops, kbytes = kmeans_flops_bytes(w)
    assign_flops = kflops / w.iters
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": roofline,
        "decode_tokens_per_s": world * w.batch * T / (decode_ms / 1000.0),
        "kmeans_ms_per_layer": prefill_ms * w.kv_heads / w.units,
        "decode_step_us": step_us,
        "decode_step_isolated": isolated,
        "kmeans_roofline": {"tflops": kflops / (prefill_ms / 1000.0) / 1e12,
                            "peak_tflops": meas.get("bf16_tflops_sustained", 1700.0),
                            "bytes_gbs": kbytes / (prefill_ms / 1000.0) / 1e9},
        "assign_roofline": {"bound": "tensor", "kernel": "assign_tc_kernel",
                            "achieved": assign_flops / (r["assign_ms"] / 1000.0) / 1e12,
                            "peak": meas.get("bf16_tflops", 1900.0), "unit": "TFLOP/s",
                            "frac": assign_flops / (r["assign_ms"] / 1000.0) / 1e12 / meas.get("bf16_tflops", 1900.0),
                            "launch_us": 1000.0 * r["assign_ms"], "peak_kind": peak_kind + " (burst: timed alone)"},
        "recall": r["recall"],
        "phase_ms": {"prefill_clustering": prefill_ms, "decode_loop": decode_ms},
        "gpu_launches": r["launches"], "clocks": r["clocks"],
    }
    for k in ("reuse", "channel_prescore", "quest", "async_clustering"):
        if k in r:
            line[k] = r[k]
    if "full_kv" in r:
        line["full_kv"] = dict(r["full_kv"], decode_speedup=r["full_kv"]["attention_us"] / step_us)
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        run, n_units, threads = oracle_jobs(w, device_tensors=r["tensors"])
        cb = run()
        line["cpu_baseline"] = {"value": cb["tokens_per_s"], "unit": "tokens/s", "cores": threads,
                                "host_cores": os.cpu_count(), "kind": "oracle (C++, float64, std::thread pool)",
                                "sample": f"{n_units} units' whole jobs (prefill clustering + {T} decode steps each) "
                                          f"on {threads} threads in {cb['wall_s']:.1f} s, extrapolated "
                                          f"x{w.units}/{n_units} units"}
    if rank == 0 and world == 1 and not args.no_workloads and args.workload == WORKLOAD:
        # the main workload's tensors go first: the batch-16 and 128k jobs hold ~69 GB each
        r.clear()
        torch.cuda.empty_cache()
        line["workloads"] = {n: measure_workload(n, hbm, l2_persist=not args.no_l2_persist) for n in OTHER_WORKLOADS}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
