"""Benchmark of the lightning-indexer top-k on GB300.

One step = one call of the whole path (scoring + streaming top-k, and the
merge of the key splits) over one batch of synthetic input. By default the
five workloads of the method are measured in turn and ONE JSON line is
printed (rank 0), headlined by the largest single-GPU one (the long prefill:
2048 queries x 131072 keys), with every workload under "workloads":

  tiny      4 queries x 2048 keys, H=8, D=64, f16 integers (exactness case)
  decode    1 query x 131072 keys, H=64, D=128, bf16
  prefill   512 queries x 16384 keys, causal
  long      2048 queries x 131072 keys, causal   (headline)
  multiseq  4 sequences x 262144 of 1048576 shared keys
  attn_decode, attn_prefill: the consumer, sparse attention over the
            decode and prefill selections (lid_sparse_attn)

Inputs are resident in HBM before the timed region; enough input sets that
their total is over twice the L2 are rotated, so no step reads its keys from
L2 (or one set larger than twice the L2). The workspace is caller-owned
(lid_topk_ws), so a step is its kernels only. Steps are replayed from a CUDA
graph and timed with CUDA events on the launching stream, bracketed by a
barrier and a synchronize. A step that is one kernel is timed back to back
(its launch duration = timed region / steps); a step of two kernels carries
events around its scoring kernel inside the timed region. Decode is also
timed with eager launches.

`--workload NAME` measures one workload only (it is then the headline).
`--impl reference` times the CPU oracle on the host cores instead (the
reference arm: there is no other implementation of this path to run).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import lid_inputs as li  # noqa: E402

METRIC = "indexer query-key pairs/s & top-512 rows/s; % of tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOAD_TEXT = {
    "tiny": "tiny exactness: n_q=4 at pos 2044..2047, n_kv=2048, H=8, D=64, f16 ints, causal, top_k=64",
    "decode": "single-token decode: n_q=1, n_kv=131072, H=64, D=128, bf16 N(0,1), w N(0,1/H), mask 0, top_k=512",
    "prefill": "prefill ubatch: n_q=512 at pos 15872..16383, n_kv=16384, H=64, D=128, bf16, causal, top_k=512",
    "long": "long prefill: n_q=2048 at pos 129024..131071, n_kv=131072, H=64, D=128, bf16, causal, top_k=512",
    "multiseq": "multi-sequence decode: 4 rows, n_kv=1048576 shared keys, disjoint 262144 ranges, top_k=512",
    "decode_e4m3": "single-token decode, E4M3 q and k with per-row scales: n_q=1, n_kv=131072, H=64, D=128, "
                   "quantised N(0,1), w N(0,1/H), mask 0, top_k=512",
    "multiseq_ranges": "multi-sequence decode through lid_topk_ranges: 4 rows, n_kv=1048576 shared keys, each row's "
                       "visible range [262144 j, 262144 (j+1)) passed instead of the dense mask, top_k=512",
    "multiseq_e4m3": "multi-sequence decode, E4M3 q and k with per-row scales: 4 rows, n_kv=1048576 shared keys, "
                     "disjoint 262144 ranges, top_k=512",
    "attn_decode": "sparse attention of the decode selection: n_q=1, 512 of n_kv=131072 latent rows (Dc=512), "
                   "Ha=64 heads, bf16 N(0,1), scale 1/sqrt(512), the top-k's scores passed through",
    "attn_prefill": "sparse attention of the prefill selections: n_q=512 at pos 15872..16383, 512 causal rows of "
                    "n_kv=16384 each (Dc=512), Ha=64 heads, bf16 N(0,1)",
}
ATTN_WORKLOADS = ("attn_decode", "attn_prefill")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# the sources of each kernel family: a recorded ncu figure holds for the code it was measured on
SOURCE_GROUPS = {
    "indexer": ("lid_api.cu", "lid_kernels.cuh", "lid_ptx.cuh", "lid_select.cuh", "lid_stream.cuh"),
    "attention": ("lid_attn.cu", "lid_attn.cuh", "lid_attn_tc.cuh", "lid_ptx.cuh"),
}


def source_hash(group="indexer"):
    """Hash of one kernel family's sources (comments and layout removed), so that
    a recorded ncu traffic figure is used only for the code it was measured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_lightning_lid_gb300", "csrc")
    for name in sorted(SOURCE_GROUPS[group]):
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the workload's dominant kernel from a committed
    ncu summary, if it was taken on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    group = "attention" if workload.startswith("attn_") else "indexer"
    if not e or e.get("source_sha") != source_hash(group):
        return None
    return e.get("dram_bytes_per_launch")


def k_row_bytes(inp):
    """Bytes of one key row: D 16-bit values, or D E4M3 codes and an f32 scale."""
    return inp.D * inp.k_bits.itemsize + (4 if inp.k_scale is not None else 0)


def q_bytes(inp):
    return inp.q_bits.nbytes + (0 if inp.q_scale is None else inp.q_scale.nbytes)


def algorithmic_work(inp, ranges=None):
    """(bytes, flops, visible pairs) one call must move / compute at least. With
    per-row visible key ranges instead of a mask, no mask bytes are read."""
    if ranges is not None:
        lo = np.clip(ranges[0].astype(np.int64), 0, inp.n_kv)
        hi = np.clip(ranges[1].astype(np.int64), lo, inp.n_kv)
        visible = int((hi - lo).sum())
        covered = np.zeros(inp.n_kv + 1, np.int64)
        np.add.at(covered, lo, 1)
        np.add.at(covered, hi, -1)
        k_rows = int(np.count_nonzero(np.cumsum(covered)[:-1]))
        nbytes = k_rows * k_row_bytes(inp) + 8 * inp.n_q + q_bytes(inp) + inp.w.nbytes + inp.n_q * inp.top_k * 8
        return nbytes, 2.0 * inp.H * inp.D * visible, visible
    m = inp.mask
    visible = inp.n_q * inp.n_kv if m is None else int(np.count_nonzero(m != li.F16_NEG_INF))
    if m is None:
        k_rows = inp.n_kv
    else:
        k_rows = int(np.count_nonzero((m != li.F16_NEG_INF).any(axis=0)))
    nbytes = (k_rows * k_row_bytes(inp) + (0 if m is None else m.nbytes) + q_bytes(inp) + inp.w.nbytes
              + inp.n_q * inp.top_k * 8)
    flops = 2.0 * inp.H * inp.D * visible
    return nbytes, flops, visible


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms for the
    whole run; window(t0, t1) summarises the samples of one timed region
    (host perf_counter times; the nearest sample when none falls inside)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.samples = []  # (perf_counter, sm, max, power, reasons)
        self.t = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.NAMES, parts[5:9]) if v.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)

    def window(self, t0, t1):
        sel = [x for x in self.samples if t0 <= x[0] <= t1]
        note = "samples inside the timed region"
        if not sel and self.samples:
            mid = 0.5 * (t0 + t1)
            sel = [min(self.samples, key=lambda x: abs(x[0] - mid))]
            note = "nearest sample (timed region shorter than the 200 ms sampling period)"
        if not sel:
            return None
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "reasons": sorted(set().union(*(x[4] for x in sel))), "samples": len(sel),
                "power_w_max": max(x[3] for x in sel), "note": note}


def gpu_uuid(torch):
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[0] if vis else None


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity
    without an initialised process group). `device` holds the reduction
    tensor: a CUDA device for NCCL, None (CPU) for gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_step_per_rank, steps, world, max_ms):
    """Units per second of the whole job: every rank processes its own
    units_per_step_per_rank each step (weak scaling); the slowest rank's time
    counts."""
    return world * units_per_step_per_rank * steps / (max_ms * 1e-3)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------- ours

HEADLINE = "long"
# timed steps of the workloads beside the headline: at least this much timed work
MIN_TIMED_S = 0.25


def roofline(inp, kern_us, ranges=None, workload=None, traffic_ok=True):
    nbytes, flops, _ = algorithmic_work(inp, ranges)
    peaks, peak_kind = load_peaks()
    hbm_bound = flops / nbytes < (peaks["bf16_tflops"] * 1e12) / (peaks["hbm_gbs"] * 1e9)
    kern_s = kern_us * 1e-6
    if hbm_bound:
        achieved = nbytes / kern_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_kind": peak_kind + " (copy bandwidth)",
                "algorithmic_bytes_per_launch": nbytes}
    else:
        achieved = flops / kern_s / 1e12
        pk = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        kind = peak_kind + " (cuBLAS bf16 burst)"
        if inp.dtype == "e4m3":  # 8-bit operands: the bf16 figure times the nominal fp8 / bf16 ratio (2)
            pk, kind = 2 * pk, kind + " x 2, nominal fp8 / bf16 ratio"
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                "peak_kind": kind, "algorithmic_flops_per_launch": flops}
    roof["traffic"] = recorded_traffic(workload) if (traffic_ok and workload) else None
    roof["kernel"] = "score_select_kernel"
    roof["kernel_avg_us"] = kern_us
    return roof


def measure(args, name, inp, dev, stream, sampler, world, steps, ranges_np=None, eager=False, e2e=False):
    """Time `steps` steps of workload `name` (inputs `inp`) on `stream`."""
    import torch

    import sparse_attention_lightning_lid_gb300 as lid

    def to_dev(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt)

    tdt = torch.float16 if inp.dtype == "f16" else torch.bfloat16
    e4m3 = inp.dtype == "e4m3"
    ranges = None
    if ranges_np is not None:
        ranges = (torch.from_numpy(ranges_np[0]).to(dev), torch.from_numpy(ranges_np[1]).to(dev))
        inp = dataclasses.replace(inp, mask=None)  # the dense mask is neither copied nor read
    set_bytes = inp.nbytes
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(2 * l2 / set_bytes) + (1 if set_bytes < 2 * l2 else 0))
    if set_bytes * n_sets > 60 << 30:
        n_sets = 1
    if e4m3:  # codes as uint8, with the per-row scales
        base = (torch.from_numpy(inp.q_bits).to(dev), torch.from_numpy(inp.k_bits).to(dev),
                torch.from_numpy(inp.w).to(dev), None if inp.mask is None else to_dev(inp.mask, torch.float16),
                torch.from_numpy(inp.q_scale).to(dev), torch.from_numpy(inp.k_scale).to(dev))
    else:
        base = (to_dev(inp.q_bits, tdt), to_dev(inp.k_bits, tdt), torch.from_numpy(inp.w).to(dev),
                None if inp.mask is None else to_dev(inp.mask, torch.float16), None, None)
    sets = [base] + [tuple(None if t is None else t.clone() for t in base) for _ in range(n_sets - 1)]
    outs = [(torch.empty((inp.n_q, inp.top_k), dtype=torch.int32, device=dev),
             torch.empty((inp.n_q, inp.top_k), dtype=torch.float32, device=dev)) for _ in range(n_sets)]
    # (the per-row range form has a plan of its own: plan_ranges)
    popt = lid.Options(force_splits=args.splits, early_tiles=args.early_tiles, force_kstages=args.kstages,
                       plan_ranges=1 if ranges is not None else 0)
    plan = lid.plan(inp.n_q, inp.n_kv, inp.H, inp.D, inp.top_k, popt)
    ws = lid.workspace(inp.n_q, inp.n_kv, inp.H, inp.D, inp.top_k, popt, device=dev)
    two_kernels = plan["splits"] > 1 and not plan["fused"]
    launches_per_step = 2 if two_kernels else 1

    G = max(1, min(args.graph_steps, steps))
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(G)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(G)]
    with torch.cuda.stream(stream):
        for e in ev_b + ev_e:
            e.record(stream)
    base_opt = lid.Options(force_splits=args.splits, early_tiles=args.early_tiles, force_kstages=args.kstages)
    # a two-kernel step carries events around its scoring kernel (inside the timed region)
    opts = [lid.Options(force_splits=args.splits, early_tiles=args.early_tiles, force_kstages=args.kstages,
                        ev_score_begin=ev_b[i].cuda_event, ev_score_end=ev_e[i].cuda_event) if two_kernels else base_opt
            for i in range(G)]

    def step(i, opt=None):
        q, k, w, m, qs, ks = sets[i % n_sets]
        oi, os_ = outs[i % n_sets]
        lid.topk_ws(q, k, w, inp.top_k, ws, mask=m, row_lo=None if ranges is None else ranges[0],
                    row_hi=None if ranges is None else ranges[1], q_scale=qs, k_scale=ks, out_idx=oi,
                    out_score=os_, stream=stream, options=base_opt if opt is None else opt)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize()

    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(G):
                    step(i, opts[i])
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
        except Exception as exc:  # capture refused: time eager launches instead
            print(f"bench: graph capture failed ({exc}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()

    reps = max(1, steps // G) if graph is not None else 0
    steps_done = reps * G if graph is not None else steps

    def timed(fn):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        t0.record(stream)
        fn()
        t1.record(stream)
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        if world > 1:
            torch.distributed.barrier()
        return t0.elapsed_time(t1), h0, h1

    def run_graph():
        with torch.cuda.stream(stream):  # replay on the stream the timing events are on
            for _ in range(reps):
                graph.replay()

    def run_eager():
        with torch.cuda.stream(stream):
            for i in range(steps_done):
                step(i, opts[i % G])

    ms, h0, h1 = timed(run_graph if graph is not None else run_eager)
    clocks = sampler.window(h0, h1) if sampler else None
    if two_kernels:
        kern_ms = sum(ev_b[i].elapsed_time(ev_e[i]) for i in range(G)) / G
        kern_src = "CUDA events around the scoring kernel of each step, inside the timed region"
    else:
        kern_ms = ms / steps_done
        kern_src = "timed region / launches: one kernel per step, launched back to back"
    ms, kern_ms = max_over_ranks([ms, kern_ms], dev)
    res = {"ms": ms, "steps": steps_done, "kern_ms": kern_ms, "kern_src": kern_src, "clocks": clocks,
           "plan": plan, "launches": steps_done * launches_per_step, "n_sets": n_sets, "graph": graph is not None,
           "G": G, "ranges": ranges_np is not None}
    if eager:
        def run_eager_plain():
            with torch.cuda.stream(stream):
                for i in range(steps_done):
                    step(i)
        ems, _, _ = timed(run_eager_plain)
        res["eager_ms_per_step"] = max_over_ranks([ems / steps_done], dev)[0]

    if e2e and not e4m3 and ranges is None:
        # end to end through the host-buffer entry point: pinned inputs in, results out
        hq = torch.from_numpy(np.ascontiguousarray(inp.q_bits).view(np.int16)).pin_memory()
        hk = torch.from_numpy(np.ascontiguousarray(inp.k_bits).view(np.int16)).pin_memory()
        hw = torch.from_numpy(np.ascontiguousarray(inp.w)).pin_memory()
        hm = None if inp.mask is None else torch.from_numpy(np.ascontiguousarray(inp.mask).view(np.int16)).pin_memory()
        ho_i = torch.empty((inp.n_q, inp.top_k), dtype=torch.int32).pin_memory()
        ho_s = torch.empty((inp.n_q, inp.top_k), dtype=torch.float32).pin_memory()
        for _ in range(3):
            lid.topk_host(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, inp.dtype, ho_i, ho_s, stream)
        n_e2e = max(3, min(args.e2e_steps, steps))
        # one call at a time, the stream drained after each (lid_topk_host)
        if world > 1:
            torch.distributed.barrier()
        tt = time.perf_counter()
        for _ in range(n_e2e):
            lid.topk_host(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, inp.dtype, ho_i, ho_s, stream)
        sync_s = max_over_ranks([(time.perf_counter() - tt) / n_e2e], dev)[0]
        # calls back to back on one stream (lid_topk_host_async): the library copies a call's inputs in on
        # its own copy stream while the previous call's kernels run, and the kernels run one after another.
        # Every step still copies its own inputs in and its own result out (into one of three pinned result
        # buffers), and the clock stops when the stream has drained.
        pouts = [(ho_i, ho_s)] + [(torch.empty_like(ho_i).pin_memory(), torch.empty_like(ho_s).pin_memory())
                                  for _ in range(2)]

        def pipelined(n):
            for i in range(n):
                oi, os_ = pouts[i % 3]
                lid.topk_host_async(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, oi, os_, inp.dtype, stream)
            stream.synchronize()

        pipelined(4)
        if world > 1:
            torch.distributed.barrier()
        tt = time.perf_counter()
        pipelined(n_e2e)
        e2e_s = max_over_ranks([(time.perf_counter() - tt) / n_e2e], dev)[0]
        h2d = hq.numel() * 2 + hk.numel() * 2 + hw.numel() * 4 + (0 if hm is None else hm.numel() * 2)
        d2h = ho_i.numel() * 4 + ho_s.numel() * 4
        res["e2e"] = {"value": whole_job_rate(inp.n_q * inp.n_kv, 1, world, e2e_s * 1e3), "unit": "pairs/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                      "steps": n_e2e,
                      "api": "lid_topk_host_async, calls back to back on one stream (pinned host buffers; every "
                             "step H2D of its inputs on the library's copy stream + kernels + D2H of its result; "
                             "clock stops after the stream drains)",
                      "sync_ms_per_step": sync_s * 1e3,
                      "sync_value": whole_job_rate(inp.n_q * inp.n_kv, 1, world, sync_s * 1e3),
                      "sync_api": "lid_topk_host (one call at a time, stream synchronised after each)"}
    del sets, outs, ws
    torch.cuda.empty_cache()
    return res


def attn_work(a):
    """(bytes, flops, attended pairs) of one sparse-attention call: the queries,
    the selection lists, every distinct selected row once, the f32 outputs;
    4 * Ha * Dc flops per attended (query, key) pair (the scores and the
    weighted sum of the rows)."""
    valid = (a.idx >= 0) & (a.idx < a.n_kv)
    if a.sel_score is not None:
        valid &= a.sel_score != -np.inf
    pairs = int(valid.sum())
    rows = int(np.unique(a.idx[valid]).size)
    nbytes = (a.qa_bits.nbytes + a.idx.nbytes + (0 if a.sel_score is None else a.sel_score.nbytes)
              + rows * a.Dc * a.kv_bits.itemsize + a.n_q * a.Ha * (a.Dc + 1) * 4)
    return nbytes, 4.0 * a.Ha * a.Dc * pairs, pairs


def measure_attn(args, name, a, dev, stream, sampler, world, steps):
    """Time `steps` calls of lid_sparse_attn on workload `name` (inputs `a`)."""
    import torch

    import sparse_attention_lightning_lid_gb300 as lid

    def to_dev(x, dt):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(dt)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(2 * l2 / a.nbytes) + (1 if a.nbytes < 2 * l2 else 0))
    base = (to_dev(a.qa_bits, torch.bfloat16), to_dev(a.kv_bits, torch.bfloat16),
            torch.from_numpy(a.idx).to(dev), torch.from_numpy(a.sel_score).to(dev))
    sets = [base] + [tuple(t.clone() for t in base) for _ in range(n_sets - 1)]
    outs = [(torch.empty((a.n_q, a.Ha, a.Dc), device=dev), torch.empty((a.n_q, a.Ha), device=dev))
            for _ in range(n_sets)]
    plan = lid.attn_plan(a.n_q, a.n_kv, a.Ha, a.Dc, a.top_k, lid.AttnOptions(path=args.attn_path))
    ws = torch.empty(max(1, plan["workspace_bytes"]), dtype=torch.uint8, device=dev)
    launches_per_step = 2 if plan["splits"] > 1 else 1

    aopt = lid.AttnOptions(path=args.attn_path)

    def step(i):
        qa, kv, idx, sc = sets[i % n_sets]
        o, l_ = outs[i % n_sets]
        lid.sparse_attn(qa, kv, idx, a.scale, sel_score=sc, out=o, lse=l_, ws=ws, stream=stream, options=aopt)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize()
    G = max(1, min(args.graph_steps, steps))
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(G):
                step(i)
        torch.cuda.synchronize()
    reps = max(1, steps // G)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    t0.record(stream)
    with torch.cuda.stream(stream):
        for r_ in range(reps):
            if graph is not None:
                graph.replay()
            else:
                for i in range(G):
                    step(r_ * G + i)
    t1.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    ms = max_over_ranks([t0.elapsed_time(t1)], dev)[0]
    steps_done = reps * G
    has_graph = graph is not None
    del sets, outs, ws, graph
    torch.cuda.empty_cache()
    return {"ms": ms, "steps": steps_done, "kern_ms": ms / steps_done, "plan": plan, "n_sets": n_sets, "G": G,
            "graph": has_graph,
            "launches": steps_done * launches_per_step, "clocks": sampler.window(h0, h1) if sampler else None}


def attn_entry(name, a, r, world):
    nbytes, flops, pairs = attn_work(a)
    peaks, peak_kind = load_peaks()
    us = r["kern_ms"] * 1e3
    ridge = (peaks["bf16_tflops"] * 1e12) / (peaks["hbm_gbs"] * 1e9)
    if flops / nbytes < ridge:
        ach = nbytes / (us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_kind": peak_kind + " (copy bandwidth)",
                "algorithmic_bytes_per_launch": nbytes}
    else:
        ach = flops / (us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"], "peak_kind": peak_kind + " (cuBLAS bf16 burst)",
                "algorithmic_flops_per_launch": flops}
    kname = "sparse_attn_tc_kernel" if r["plan"]["path"] == 2 else "sparse_attn_kernel"
    roof.update({"traffic": recorded_traffic(name),
                 "kernel": kname + (" + attn_combine_kernel" if r["plan"]["splits"] > 1 else ""),
                 "kernel_avg_us": us, "kernel_timing": "timed region / steps (back to back)",
                 "intensity_flop_per_byte": flops / nbytes, "ridge_flop_per_byte": ridge})
    return {"workload": WORKLOAD_TEXT[name], "steps": r["steps"], "ms_per_step": r["ms"] / r["steps"],
            "attended_pairs_per_s": whole_job_rate(pairs, r["steps"], world, r["ms"]),
            "tokens_per_s": whole_job_rate(a.n_q, r["steps"], world, r["ms"]),
            "kernel_avg_us": us, "roofline": roof, "gpu_launches": r["launches"], "clocks": r["clocks"],
            "plan": r["plan"], "dtype": "bf16",
            "l2": f"{r['n_sets']} rotating input set(s) ({r['n_sets'] * a.nbytes / 2**20:.0f} MiB > 2x L2)",
            "launch": f"CUDA graph of {r['G']} steps" if r["graph"] else "eager launches"}


def workload_entry(name, inp, r, world, ranges_np=None):
    """The per-workload record of the JSON line."""
    roof = roofline(inp, r["kern_ms"] * 1e3, ranges_np, name, traffic_ok=ranges_np is None)
    roof["kernel_timing"] = r["kern_src"]
    nbytes, flops, visible = algorithmic_work(inp, ranges_np)
    e = {"workload": WORKLOAD_TEXT[name], "steps": r["steps"], "ms_per_step": r["ms"] / r["steps"],
         "pairs_per_s": whole_job_rate(inp.n_q * inp.n_kv, r["steps"], world, r["ms"]),
         "rows_per_s": whole_job_rate(inp.n_q, r["steps"], world, r["ms"]),
         "visible_pairs_per_s": whole_job_rate(visible, r["steps"], world, r["ms"]),
         "kernel_avg_us": r["kern_ms"] * 1e3, "roofline": roof, "gpu_launches": r["launches"],
         "clocks": r["clocks"], "plan": r["plan"],
         "l2": f"{r['n_sets']} rotating input set(s) ({r['n_sets'] * inp.nbytes / 2**20:.0f} MiB > 2x L2)",
         "launch": f"CUDA graph of {r['G']} steps" if r["graph"] else "eager launches",
         "mask_form": "per-row visible ranges" if r["ranges"] else "dense f16 mask", "dtype": inp.dtype}
    if "eager_ms_per_step" in r:
        e["eager_ms_per_step"] = r["eager_ms_per_step"]
        e["eager_us_per_step_note"] = "the same steps launched eagerly (no graph), timed back to back"
    if "e2e" in r:
        e["e2e"] = r["e2e"]
    return e


def run_ours(args):
    import torch

    import sparse_attention_lightning_lid_gb300 as lid

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lid.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    sampler = ClockSampler(gpu_uuid(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    names = [args.workload] if args.workload != "all" else list(li.WORKLOADS) + ["multiseq_ranges"] + list(
        ATTN_WORKLOADS)
    headline = args.workload if args.workload != "all" else HEADLINE
    entries, results, inputs = {}, {}, {}
    for name in names:
        if name in ATTN_WORKLOADS:
            a = li.attn_workload(name)
            est = {"attn_decode": 15e-6, "attn_prefill": 110e-6}[name]
            steps = args.steps if name == headline else max(args.steps, int(MIN_TIMED_S / est) // 100 * 100)
            r = measure_attn(args, name, a, dev, stream, sampler, world, steps)
            results[name], inputs[name] = r, a
            entries[name] = attn_entry(name, a, r, world)
            continue
        # multiseq_ranges: the multi-sequence workload through lid_topk_ranges (each row's
        # visible range instead of the dense mask)
        base = "multiseq" if name == "multiseq_ranges" else name
        inp = li.workload(base)
        if name == "multiseq_ranges":
            ranges_np = li.workload_ranges(base)
        else:
            ranges_np = li.workload_ranges(name) if (args.ranges and name == args.workload) else None
        if name == headline:
            steps = args.steps
        else:  # about MIN_TIMED_S of timed work, at least --steps
            est = {"tiny": 10e-6, "decode": 10e-6, "prefill": 150e-6, "long": 4e-3, "multiseq": 80e-6,
                   "multiseq_ranges": 70e-6}.get(name, 1e-3)
            steps = max(args.steps, int(MIN_TIMED_S / est) // 100 * 100)
        r = measure(args, name, inp, dev, stream, sampler, world, steps, ranges_np,
                    eager=name.startswith("decode"), e2e=(name == headline and not args.no_e2e))
        results[name] = r
        inputs[name] = inp
        entries[name] = workload_entry(name, inp, r, world, ranges_np)
    if sampler:
        sampler.stop()
    if world > 1:
        torch.distributed.destroy_process_group()
    return {"world": world, "rank": rank, "headline": headline, "entries": entries, "results": results,
            "inputs": inputs}


# ---------------------------------------------------------------- oracle arm

def oracle_rows_for_budget(inp, seconds):
    """Rows of the workload the oracle can score in about `seconds`."""
    import oracle
    t = time.perf_counter()
    oracle.topk_inputs(inp, rows=[0])
    one = max(time.perf_counter() - t, 1e-3)
    return max(1, min(inp.n_q, int(seconds / one)))


def cpu_baseline(inp, budget_s=10.0):
    import oracle
    rows = oracle_rows_for_budget(inp, min(budget_s, 10.0) / 3)
    sel = np.arange(rows, dtype=np.int64)
    reps, total_pairs = 0, 0
    t = time.perf_counter()
    while True:
        oracle.topk_inputs(inp, rows=sel)
        reps += 1
        total_pairs += rows * inp.n_kv
        if time.perf_counter() - t > budget_s / 3 or reps >= 50:
            break
    el = time.perf_counter() - t
    return {"value": total_pairs / el, "unit": "pairs/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{reps} oracle call(s) on {rows} of {inp.n_q} query rows x {inp.n_kv} keys "
                      f"of the same workload ({el:.1f} s wall, fp64, full sort per row)",
            "cpu": cpu_model()}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args, inp, name):
    import oracle
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    rows = oracle_rows_for_budget(inp, 1.0)
    sel = np.arange(rows, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.topk_inputs(inp, rows=sel)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.topk_inputs(inp, rows=sel)
    el = time.perf_counter() - t
    value = args.steps * rows * inp.n_kv / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "pairs/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "rows_per_s": args.steps * rows / el,
        "config": {"workload": WORKLOAD_TEXT[name], "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"each step: {rows} of {inp.n_q} query rows x {inp.n_kv} keys",
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + list(WORKLOAD_TEXT))
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--splits", type=int, default=0, help="force the key-split count (0 = planned)")
    ap.add_argument("--kstages", type=int, default=0, help="force the K pipeline stages (0 = planned)")
    ap.add_argument("--early-tiles", type=int, default=0,
                    help="(one-launch path) tiles streamed before the certificates are published (0 = planned)")
    ap.add_argument("--attn-path", type=int, default=0,
                    help="(attention workloads) 0 planned, 1 warp-level MMA kernel, 2 tensor-core kernel")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ranges", action="store_true",
                    help="(with --workload) pass each row's visible key range (lid_topk_ranges form) "
                         "instead of the dense mask")
    args = ap.parse_args()

    if args.impl == "reference":
        import oracle
        oracle.build()
        name = args.workload if args.workload != "all" else HEADLINE
        if name in ATTN_WORKLOADS:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the top-k workloads"}))
            return 0
        return run_reference(args, li.workload("multiseq" if name == "multiseq_ranges" else name), name)

    r = run_ours(args)
    if r["rank"] != 0:
        return 0
    world = r["world"]
    name = r["headline"]
    head = r["entries"][name]
    res = r["results"][name]
    inp = r["inputs"][name]
    if name in ATTN_WORKLOADS:  # one attention workload on its own
        line = {"metric": "sparse attention: attended (query, key) pairs/s", "value": head["attended_pairs_per_s"],
                "unit": "pairs/s", "n_gpus": world, "steps": res["steps"], "warmup": args.warmup,
                "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD_TEXT[name], "l2": head["l2"], "launch": head["launch"],
                           "plan": head["plan"]},
                "roofline": head["roofline"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                "e2e": None, "workloads": r["entries"]}
        print(json.dumps(line))
        return 0
    line = {
        "metric": METRIC, "value": head["pairs_per_s"], "unit": "pairs/s", "n_gpus": world, "steps": res["steps"],
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": inp.dtype, "data": "synthetic",
        "rows_per_s": head["rows_per_s"], "visible_pairs_per_s": head["visible_pairs_per_s"],
        "config": {"workload": WORKLOAD_TEXT[name], "global_batch": inp.n_q * world, "n_kv": inp.n_kv,
                   "top_k": inp.top_k, "l2": head["l2"], "launch": head["launch"],
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "mask_form": head["mask_form"],
                   "plan": head["plan"]},
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "e2e": res.get("e2e"),
        "workloads": {k: v for k, v in r["entries"].items()},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
