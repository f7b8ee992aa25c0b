#!/usr/bin/env python
"""Benchmark of one paged-KV decode step on GB300.

A step is one pass of the whole hot path over one batch: append each
sequence's new K/V token through ``slot_mapping``, then decode attention over
the paged cache (with the split-K log-sum-exp merge when the plan splits; for
workloads whose sequences share prefix blocks, the shared-prefix decode).
Inputs are seeded synthetic caches (see ``workloads``) already resident in
HBM.  Every workload's KV cache is larger than the 129 MB L2, and consecutive
calls alternate between two copies of it, so no call finds the previous
call's lines in L2 and no flush is needed between steps.

Prints ONE JSON line on rank 0.  ``value`` is achieved HBM bandwidth over the
step's algorithmic bytes (K+V of every context token, counted once per
physical slot, + Q + O + block-table entries + context lengths + the append's
reads and writes), in GB/s, summed over ranks.  Without ``--config`` the
headline is the long-context layer (c4, the largest single-GPU workload) and
``per_config`` holds the same measurements for c2, c3, c5 and c5_bs32.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the same workload

Multi-GPU (N > 1, one process per GPU under torch.distributed.run): every rank
runs an independent replica of the workload (its own seed); there is no
collective on the data path, only a barrier and a max-reduction of the timing.
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

METRIC = "paged decode-attn achieved HBM GB/s (% of GB300 peak); decode tokens/s, 1 GPU"
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "c1": "tiny paged decode: B=2, context {37,50}+1, bs16, 4q/2kv heads, d64, fp16",
    "c2": "Llama-7B-shaped MHA layer: B=64, 32q/32kv heads, d128, bs16, context U[512,4096], fp16",
    "c3": "Llama-70B-shaped GQA-8 layer: B=32, 64q/8kv heads, d128, bs16, context 4096, bf16",
    "c4": "long-context split-K: B=8, 64q/8kv heads, d128, bs16, context U[32768,131072], bf16",
    "c5": "continuous-batching mix: B=256, 32q/8kv heads, d128, bs16, 2048-token shared prefix "
          "in 4 groups + lognormal suffix, bf16",
    "c5_bs32": "continuous-batching mix, bs32 variant",
}

# DRAM bytes (read + write) per launch of the decode path measured by ncu
# (profiles/), keyed by workload; valid only for the kernel sources they were
# measured on (digest of csrc/), else reported as null.
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
    #     --clock-control none -k regex:decode_kernel -s 4 -c 1 (the fused default step)
    "c4": {"digest": "cf3422a1a4f3f93b", "splits": 64, "shared": False, "fused": True,
           "bytes": 2818488320 + 7384064},
    "c2": {"digest": "cf3422a1a4f3f93b", "splits": 2, "shared": False, "fused": True,
           "bytes": 2312607744 + 4360192},
    "c3": {"digest": "cf3422a1a4f3f93b", "splits": 3, "shared": False, "fused": True,
           "bytes": 537545984 + 4047872},
    # shared-prefix path: decode_kernel (suffixes, and the merge of each unit by
    # its last CTA; -k regex:decode_kernel -s 4 -c 1) + prefix_kernel
    # (-k regex:prefix_kernel -s 2 -c 1); the plan kernel's few KB are not included
    "c5": {"digest": "cf3422a1a4f3f93b", "splits": 8, "shared": True, "fused": False,
           "bytes": (1536165632 + 5141504) + (35748096 + 16640)},
    "c5_bs32": {"digest": "cf3422a1a4f3f93b", "splits": 8, "shared": True, "fused": False,
                "bytes": (1536079616 + 5253632) + (35749120 + 9216)},
}


def _kernel_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_164_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(w, q_len: int = 1, kv_bytes: int = 2) -> dict:
    """Algorithmic bytes of one step of workload ``w`` (16-bit q, out and new
    tokens; ``kv_bytes`` per cached K/V element), with ``q_len`` query tokens
    per sequence (1: decode)."""
    import torch
    e = 2
    s = w.spec
    lens = w.context_lens.cpu().long()
    bt = w.block_tables.cpu().long()
    bs = s.block_size
    row = s.num_kv_heads * s.head_dim * kv_bytes     # one cached token's K (or V) row
    logical_tokens = int(lens.sum())
    # unique physical slots read (shared prefix pages count once per step)
    slots = []
    for b in range(s.num_seqs):
        n = int(lens[b])
        t = torch.arange(n)
        slots.append(bt[b, t // bs] * bs + t % bs)
    unique_tokens = int(torch.unique(torch.cat(slots)).numel()) if slots else 0
    pages = int(((lens + bs - 1) // bs).sum())
    qo = 2 * s.num_seqs * q_len * s.num_q_heads * s.head_dim * e
    meta = pages * 4 + s.num_seqs * 4
    decode = 2 * unique_tokens * row + qo + meta
    decode_logical = 2 * logical_tokens * row + qo + meta
    new_row = s.num_kv_heads * s.head_dim * e
    append = 2 * s.num_seqs * (new_row + row) + 8 * s.num_seqs   # read new K/V, write both; slots
    flops = 4 * logical_tokens * q_len * s.num_q_heads * s.head_dim
    return dict(decode=decode, decode_logical=decode_logical, append=append,
                step=decode + append, kv_unique=2 * unique_tokens * row, flops=flops,
                tokens=s.num_seqs * q_len)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while it runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_begin: float, t_end: float) -> dict:
        if self.proc is None or not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [l for (t, l) in self.lines if t_begin <= t <= t_end + 0.15]
        note = None
        if not inside:
            # the region was shorter than the sampling period: take the nearest sample
            nearest = min(self.lines, key=lambda tl: abs(tl[0] - (t_begin + t_end) / 2))
            inside = [nearest[1]]
            note = "timed region shorter than the sampling period; nearest sample used"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in inside:
            p = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except (ValueError, IndexError):
                continue
            for name, flag in zip(names, p[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
               "samples": len(inside)}
        if note:
            out["note"] = note
        return out


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(value: float, op: str, device=None) -> float:
    """max or sum of a scalar over ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def oracle_inputs(w):
    """The oracle's inputs for ``w`` (on the host): its caches with the step's new
    tokens appended by the oracle, q, block tables and context lengths."""
    import oracle
    from workloads import bits
    kc, vc = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    oracle.append(kc, vc, bits(w.k_new), bits(w.v_new), w.slot_mapping.cpu().numpy())
    return kc, vc, bits(w.q), w.block_tables.cpu().numpy(), w.context_lens.cpu().numpy()


def oracle_sample_rate(w, budget_s: float, seqs=None, inputs=None):
    """Times the fp64 oracle on a bounded sample of ``w``'s sequences.

    Returns (GB/s over the sample's algorithmic bytes, seconds, sample description,
    threads).  The sample is the first k sequences, k sized from a one-sequence
    calibration so the timed call takes about ``budget_s`` seconds.  ``inputs``:
    ``oracle_inputs(w)``, prepared once when the rate is taken repeatedly.
    """
    import numpy as np
    import oracle
    kc, vc, q, bt, cl = inputs if inputs is not None else oracle_inputs(w)
    s = w.spec
    row = s.num_kv_heads * s.head_dim * 2

    q_len = q.shape[1] if q.ndim == 4 else 1  # several query tokens: causal multi-query

    def run(idx):
        t0 = time.perf_counter()
        if q.ndim == 4:
            oracle.multi_query_attention(q[idx], kc, vc, bt[idx], cl[idx], w.scale, s.dtype)
        else:
            oracle.decode_attention(q[idx], kc, vc, bt[idx], cl[idx], w.scale, s.dtype)
        return time.perf_counter() - t0

    if seqs is None:
        t1 = run(np.arange(1))
        per_seq = max(t1, 1e-4)
        k = int(max(1, min(s.num_seqs, budget_s / per_seq)))
        seqs = np.arange(k)
    # repeat the sample until about budget_s of CPU work has been timed
    secs, reps = 0.0, 0
    while reps == 0 or secs < budget_s:
        secs += run(seqs)
        reps += 1
    secs /= reps
    toks = int(cl[seqs].sum())
    nbytes = 2 * toks * row + 2 * len(seqs) * q_len * s.num_q_heads * s.head_dim * 2
    what = f"multi-query attention ({q_len} query tokens)" if q.ndim == 4 else "decode attention"
    desc = (f"oracle {what} on the first {len(seqs)} of {s.num_seqs} sequences "
            f"({toks} context tokens) of the same workload, timed over {reps} runs")
    return nbytes / secs / 1e9, secs, desc, oracle.num_threads(), seqs


def run_reference(args):
    """The fp64 CPU oracle timed as the reference arm (rank 0 only)."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import torch
    from workloads import make_queries, make_workload
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    name = args.config or HEADLINE_CONFIG
    w = make_workload(name, device=dev)
    if args.q_len > 0:
        w.q = make_queries(w, args.q_len, seed=w.spec.seed + 101)
    w = w.to("cpu")
    # about --ref-seconds (150 s) of oracle work in all, whatever the step count
    # (0.2 to 10 s a step)
    per_step = max(0.2, min(10.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    inputs = oracle_inputs(w)
    seqs = None
    for _ in range(args.warmup):
        _, _, _, _, seqs = oracle_sample_rate(w, per_step, seqs, inputs)
    rates, secs_all = [], []
    desc, threads = "", 1
    for _ in range(args.steps):
        r, secs, desc, threads, seqs = oracle_sample_rate(w, per_step, seqs, inputs)
        rates.append(r)
        secs_all.append(secs)
    value = statistics.median(rates) if rates else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.median(secs_all), 3) if secs_all else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "description": WORKLOAD_TEXT[name],
                       "q_len": max(1, args.q_len)},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


HEADLINE_CONFIG = "c4"
PER_CONFIGS = ("c2", "c3", "c5", "c5_bs32")
# Copies of the KV cache that consecutive calls alternate between, so that no
# call finds the previous call's lines in L2 (each copy is far larger than L2).
KV_COPIES = 2


def _measure(name, args, device, rank, ws, cpu_seconds):
    """Builds workload ``name`` on ``device`` and times its step, its decode
    call, its append and its end-to-end step; returns the numbers (timings
    already reduced over ranks) and the JSON fields that describe them."""
    import torch

    import paged_kv_cache_164_gb300 as pkv
    from workloads import SPECS, make_queries, make_workload, to_head_major

    # --block-size: the workload with another page size
    overrides = {"block_size": args.block_size} if args.block_size else {}
    if ws > 1:  # an independent replica per rank
        w = make_workload(name, device=device, seed=SPECS[name].seed + 1000 * rank, **overrides)
    else:
        w = make_workload(name, device=device, **overrides)
    layout = args.layout
    if layout == "hnd":  # the same values in the head-major page layout
        w.k_cache = to_head_major(w.k_cache)
        w.v_cache = to_head_major(w.v_cache)
    s = w.spec
    # --q-len N: causal multi-query attention of N query tokens per sequence
    # (a prefill chunk or speculative verification) in place of the decode
    mq = args.q_len > 0
    if mq:
        w.q = make_queries(w, args.q_len, seed=s.seed + 101)
    # --kv fp8: the cache as E4M3 codes with one scale for K and one for V
    fp8 = args.kv == "fp8"
    k_scale = v_scale = 1.0
    if fp8:
        k_scale = float(w.k_cache.float().abs().max()) / 448.0
        v_scale = float(w.v_cache.float().abs().max()) / 448.0
        w.k_cache = (w.k_cache.float() / k_scale).clamp(-448, 448).to(
            torch.float8_e4m3fn).view(torch.uint8)
        w.v_cache = (w.v_cache.float() / v_scale).clamp(-448, 448).to(
            torch.float8_e4m3fn).view(torch.uint8)
    caches = [(w.k_cache, w.v_cache)]
    for _ in range(KV_COPIES - 1):
        caches.append((w.k_cache.clone(), w.v_cache.clone()))
    nbytes = step_bytes(w, args.q_len if mq else 1, 1 if fp8 else 2)
    mcl = w.max_context_len
    # Workloads whose sequences share prefix blocks use the shared-prefix decode
    # (each group's prefix read once for all members) unless told otherwise.
    shared = s.shared_prefix_groups > 0 and args.prefix_sharing and not mq
    # Host-side bounds of the group metadata, read once (each read syncs the device).
    max_group_size, max_prefix_len = w.max_group_size, w.max_prefix_len
    splits = pkv.decode_num_splits(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                   s.block_size, mcl, args.splits, kv=args.kv)
    mq_kernel, mq_parts = None, 0
    if mq:
        mq_kernel, mq_parts = pkv.multi_query_plan(s.num_seqs, args.q_len, s.num_q_heads,
                                                   s.num_kv_heads, s.head_dim, s.block_size, mcl)
        ws_bytes = pkv.multi_query_workspace_size(s.num_seqs, args.q_len, s.num_q_heads,
                                                  s.num_kv_heads, s.head_dim, s.block_size, mcl)
    elif shared:
        ws_bytes = pkv.prefix_shared_workspace_size(
            s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim, s.block_size, mcl,
            w.group_prefix_len.numel(), max_group_size, max_prefix_len)
    else:
        ws_bytes = pkv.workspace_size(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                      s.block_size, mcl, args.splits)
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    out = torch.empty_like(w.q)
    flag = pkv.new_error_flag(device)
    # append, decode, merge when split; the shared-prefix path: append, plan,
    # prefix (second stream) and decode (no merge launch)
    # The step's append is done by the decode kernel itself
    # (pkv_append_decode_attention, or its E4M3 form) on the plain path;
    # --unfused times the two calls (the append, then the decode) instead.
    fused = args.fused and not mq and not shared
    if mq:
        launches_per_step = 2 + (1 if mq_kernel == "tcgen05" or mq_parts > 1 else 0)
    else:
        launches_per_step = (4 if shared else (1 if fused else 2) + (1 if splits > 1 else 0))

    def decode_call(c, q, block_tables, context_lens, out=out):
        kc, vc = caches[c]
        if fp8:
            pkv.decode_attention_fp8(q, kc, vc, block_tables, context_lens, mcl,
                                     k_scale, v_scale, scale=w.scale, num_splits=args.splits,
                                     out=out, workspace=workspace, err_flag=flag, layout=layout)
        elif mq:
            pkv.multi_query_attention(q, kc, vc, block_tables, context_lens, mcl,
                                      scale=w.scale, out=out, workspace=workspace, err_flag=flag,
                                      layout=layout)
        elif shared:
            pkv.decode_attention_prefix_shared(
                q, kc, vc, block_tables, context_lens, mcl, w.group_start,
                w.group_prefix_len, max_group_size, max_prefix_len, scale=w.scale, out=out,
                workspace=workspace, err_flag=flag, layout=layout)
        else:
            pkv.decode_attention(q, kc, vc, block_tables, context_lens, mcl,
                                 scale=w.scale, num_splits=args.splits, out=out,
                                 workspace=workspace, err_flag=flag, layout=layout)

    def append_call(c, k_new, v_new, slot_mapping):
        kc, vc = caches[c]
        if fp8:
            pkv.append_fp8(k_new, v_new, kc, vc, slot_mapping, k_scale, v_scale,
                           err_flag=flag, layout=layout)
        else:
            pkv.append(k_new, v_new, kc, vc, slot_mapping, err_flag=flag, layout=layout)

    def fused_call(c, q, k_new, v_new, block_tables, context_lens, out=out):
        kc, vc = caches[c]
        if fp8:
            pkv.append_decode_attention_fp8(q, k_new, v_new, kc, vc, block_tables, context_lens,
                                            mcl, k_scale, v_scale, scale=w.scale,
                                            num_splits=args.splits, out=out,
                                            workspace=workspace, err_flag=flag, layout=layout)
        else:
            pkv.append_decode_attention(q, k_new, v_new, kc, vc, block_tables, context_lens,
                                        mcl, scale=w.scale, num_splits=args.splits, out=out,
                                        workspace=workspace, err_flag=flag, layout=layout)

    def step(c):
        if fused:
            fused_call(c, w.q, w.k_new, w.v_new, w.block_tables, w.context_lens)
            return
        append_call(c, w.k_new, w.v_new, w.slot_mapping)
        decode_call(c, w.q, w.block_tables, w.context_lens)

    for i in range(args.warmup):
        step(i % KV_COPIES)
    if pkv.check_error(flag) != 0:
        raise RuntimeError(f"{name}: device error flag set during warm-up")

    stream = torch.cuda.current_stream(device)

    def timed(fn, count):
        """ms per call of fn(i) over `count` calls back to back, with CUDA events
        on the launching stream and a synchronise on both sides."""
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(device)
        torch.cuda.synchronize(device)
        t0.record(stream)
        for i in range(count):
            fn(i)
        t1.record(stream)
        torch.cuda.synchronize(device)
        return t0.elapsed_time(t1) / count

    # Timed region: K whole steps back to back (the library chains its kernels
    # with programmatic dependent launch, so no event sits between them).
    run_step = lambda i: step(i % KV_COPIES)  # noqa: E731
    if args.graph:
        # one step per cache copy captured in a CUDA graph (the library's
        # set-up ran in the warm-up above), replayed in turn: one graph launch
        # per step
        graphs = []
        for c in range(KV_COPIES):
            side = torch.cuda.Stream(device)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                step(c)
            stream.wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step(c)
            graph.replay()
            graphs.append(graph)
        torch.cuda.synchronize(device)
        run_step = lambda i: graphs[i % KV_COPIES].replay()  # noqa: E731
    t_begin = time.time()
    ms_local = timed(run_step, args.steps)
    t_end = time.time()
    # The dominant kernel alone: K decode calls back to back (decode kernel and,
    # when the plan splits, its merge), for the roofline.
    for i in range(3):
        decode_call(i % KV_COPIES, w.q, w.block_tables, w.context_lens)
    decode_ms = timed(lambda i: decode_call(i % KV_COPIES, w.q, w.block_tables, w.context_lens),
                      args.steps)
    # The append alone (the scatter of the step's new K/V rows), timed the same way.
    for i in range(3):
        append_call(i % KV_COPIES, w.k_new, w.v_new, w.slot_mapping)
    append_ms = timed(lambda i: append_call(i % KV_COPIES, w.k_new, w.v_new, w.slot_mapping),
                      args.steps)
    ms_step = reduce_over_ranks(ms_local, "max", device)
    decode_ms = reduce_over_ranks(decode_ms, "max", device)
    append_ms = reduce_over_ranks(append_ms, "max", device)
    bytes_all = reduce_over_ranks(float(nbytes["step"]), "sum", device)
    tokens_all = reduce_over_ranks(float(nbytes["tokens"]), "sum", device)
    if pkv.check_error(flag) != 0:
        raise RuntimeError(f"{name}: device error flag set during the timed steps")

    # ---- end to end through the public API: pinned host inputs -> device -> host output
    # Every step copies its inputs from pinned host memory and its output back.
    # As a serving loop would: the inputs travel as one packed copy into one of
    # two device staging buffers on a copy stream, so step i+1's inputs move
    # while step i computes, and step i's output returns on another stream.
    # (the fused step derives each new token's slot itself: no slot mapping)
    names = ("q", "k_new", "v_new") + (() if fused else ("slot_mapping",)) + \
        ("block_tables", "context_lens")
    srcs = {k: getattr(w, k) for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (srcs[k].numel() * srcs[k].element_size() + 255) // 256 * 256
    host_buf = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dev_buf = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    views = []
    for sidx in range(2):
        v = {}
        for k in names:
            t = srcs[k]
            nb = t.numel() * t.element_size()
            host_buf[sidx][offs[k]:offs[k] + nb].copy_(
                t.contiguous().view(-1).view(torch.uint8).cpu())
            v[k] = dev_buf[sidx][offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        views.append(v)
    outs = [torch.empty_like(out) for _ in range(2)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(srcs[k].numel() * srcs[k].element_size() for k in names)
    d2h = out_h[0].numel() * out_h[0].element_size()
    h2d_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    in_free = [torch.cuda.Event() for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    state = {"i": 0}

    def e2e_step():
        i = state["i"]
        sidx = i % 2
        state["i"] += 1
        h2d_stream.wait_event(in_free[sidx])      # the step that last read this buffer is done
        with torch.cuda.stream(h2d_stream):
            dev_buf[sidx].copy_(host_buf[sidx], non_blocking=True)
        in_ready[sidx].record(h2d_stream)
        stream.wait_event(in_ready[sidx])
        stream.wait_event(out_free[sidx])          # this output buffer's copy-out is done
        v = views[sidx]
        if fused:
            fused_call(i % KV_COPIES, v["q"], v["k_new"], v["v_new"], v["block_tables"],
                       v["context_lens"], out=outs[sidx])
        else:
            append_call(i % KV_COPIES, v["k_new"], v["v_new"], v["slot_mapping"])
            decode_call(i % KV_COPIES, v["q"], v["block_tables"], v["context_lens"],
                        out=outs[sidx])
        in_free[sidx].record(stream)
        done[sidx].record(stream)
        d2h_stream.wait_event(done[sidx])
        with torch.cuda.stream(d2h_stream):
            out_h[sidx].copy_(outs[sidx], non_blocking=True)
        out_free[sidx].record(d2h_stream)

    def e2e_drain():
        for sidx in range(2):
            stream.wait_event(out_free[sidx])

    for _ in range(max(3, args.warmup // 2)):
        e2e_step()
    e2e_drain()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(device)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    d2h_stream.wait_event(e0)
    for _ in range(args.steps):
        e2e_step()
    e2e_drain()
    e1.record(stream)
    torch.cuda.synchronize(device)
    t_loops_end = time.time()
    e2e_ms = reduce_over_ranks(e0.elapsed_time(e1) / args.steps, "max", device)
    last = (state["i"] - 1) % 2
    if not torch.equal(out_h[last].to(device), out):
        raise RuntimeError(f"{name}: end-to-end output differs from the device output")

    traffic = None
    rec = NCU_TRAFFIC.get(name)
    if rec and rec.get("digest") == _kernel_digest() and rec.get("splits") == splits and \
            rec.get("shared") == shared and rec.get("fused") == fused and not mq and \
            layout == "nhd" and not args.block_size and not fp8:
        traffic = rec["bytes"]

    cpu = None
    if rank == 0 and cpu_seconds > 0:
        w_host = w.to("cpu")
        gbs, secs, desc, threads, _ = oracle_sample_rate(w_host, cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": round(secs, 3)}
        del w_host

    peak, _ = _peaks()
    value = bytes_all / (ms_step * 1e-3) / 1e9
    decode_gbs = nbytes["decode"] / (decode_ms * 1e-3) / 1e9
    kernel = (("prefix_kernel in multi-query mode (tcgen05) + merge_kernel"
               if mq_kernel == "tcgen05" else
               "decode_kernel in multi-query mode" + (" + merge_kernel" if mq_parts > 1 else ""))
              if mq else
              "plan_kernel, then prefix_kernel (on a second stream) beside decode_kernel "
              "(each unit merged by its last CTA)"
              if shared else "decode_kernel + merge_kernel")
    config = {"workload": name, "description": WORKLOAD_TEXT[name],
              "num_seqs": s.num_seqs, "num_q_heads": s.num_q_heads,
              "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim,
              "block_size": s.block_size, "context_tokens": int(w.context_lens.sum()),
              "max_context_len": mcl, "num_splits": mq_parts if mq else splits,
              "accumulate": "fp32", "shared_prefix_decode": shared,
              "q_len": args.q_len if mq else 1,
              "fused_append": fused, "cuda_graph": bool(args.graph),
              "layout": layout, "kv_cache": "e4m3" if fp8 else s.dtype,
              "kv_bytes_unique": nbytes["kv_unique"],
              "decode_bytes_per_step": nbytes["decode"],
              "decode_bytes_logical": nbytes["decode_logical"],
              "append_bytes_per_step": nbytes["append"],
              "l2": f"no flush: the KV cache ({nbytes['kv_unique'] / 1e9:.2f} GB) is larger than "
                    f"the 129 MB L2, and consecutive calls alternate between {KV_COPIES} copies "
                    "of it, so no call finds the previous call's lines in L2",
              "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU"}
    return {
        "name": name, "ms_step": ms_step, "value": value, "decode_ms": decode_ms,
        "append_ms": append_ms, "e2e_ms": e2e_ms, "bytes_all": bytes_all,
        "tokens_all": tokens_all, "nbytes": nbytes, "decode_gbs": decode_gbs, "peak": peak,
        "traffic": traffic, "kernel": kernel, "cpu": cpu, "config": config, "h2d": h2d,
        "d2h": d2h, "launches": launches_per_step * args.steps, "t_begin": t_begin,
        "t_end": t_end, "t_loops_end": t_loops_end,
        "dtype": f"e4m3 KV, {s.dtype} q" if fp8 else s.dtype,
    }


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_164_gb300 as pkv

    ws, rank, local = _dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    pkv.load()

    names = config_names(args)
    sampler = ClockSampler(device.index, period_ms=50) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    results = []
    for i, name in enumerate(names):
        secs = (args.cpu_seconds if i == 0 else args.cpu_seconds_per_config) \
            if args.cpu_baseline else 0.0
        results.append(_measure(name, args, device, rank, ws, secs))
        torch.cuda.empty_cache()
    if sampler:
        sampler.stop()

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return

    peak, peak_src = _peaks()
    head = results[0]

    def e2e_of(r):
        return {"value": round(r["bytes_all"] / (r["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(r["e2e_ms"], 5), "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"]}

    def roofline_of(r):
        return {"bound": "hbm", "achieved": round(r["decode_gbs"], 2), "peak": peak,
                "unit": "GB/s", "frac": round(r["decode_gbs"] / peak, 4),
                "traffic": r["traffic"],
                "kernel": r["kernel"] + " (one attention call, back to back)",
                "peak_source": f"{peak_src} hbm_gbs",
                "peak_kind": "a device-to-device copy (half reads, half writes); this path "
                             "only reads (KV, q) and writes little, so a call can read a few "
                             "percent above it"}

    per_config = {}
    for r in results[1:]:
        per_config[r["name"]] = {
            "value": round(r["value"], 2), "unit": "GB/s",
            "pct_of_peak": round(100.0 * r["value"] / (peak * ws), 2),
            "ms_per_step": round(r["ms_step"], 5),
            "tokens_per_s": round(r["tokens_all"] / (r["ms_step"] * 1e-3), 1),
            "decode_ms": round(r["decode_ms"], 5), "append_ms": round(r["append_ms"], 5),
            "roofline": roofline_of(r), "e2e": e2e_of(r), "cpu_baseline": r["cpu"],
            "gpu_launches": r["launches"], "dtype": r["dtype"], "config": r["config"],
            "clocks": sampler.summary(r["t_begin"], r["t_end"]) if sampler else None,
        }

    e2e = e2e_of(head)
    e2e["copies"] = ("per step: inputs packed in one pinned buffer, one H2D copy into one of two "
                     "device staging buffers on a copy stream (overlapping the previous step's "
                     "compute), output D2H on a second stream")
    line = {
        "metric": METRIC, "value": round(head["value"], 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(head["ms_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"], "data": "synthetic",
        "config": head["config"],
        "pct_of_peak": round(100.0 * head["value"] / (peak * ws), 2),
        "tokens_per_s": round(head["tokens_all"] / (head["ms_step"] * 1e-3), 1),
        "decode_ms": round(head["decode_ms"], 5),
        "append_ms": round(head["append_ms"], 5),
        "append_gbs": round(head["nbytes"]["append"] / (head["append_ms"] * 1e-3) / 1e9, 2),
        "roofline": roofline_of(head),
        "cpu_baseline": head["cpu"],
        "e2e": e2e,
        "gpu_launches": head["launches"],
        "clocks": sampler.summary(head["t_begin"], head["t_end"]) if sampler else None,
        "clocks_all_timed_loops": (sampler.summary(results[0]["t_begin"],
                                                   results[-1]["t_loops_end"])
                                   if sampler else None),
    }
    if per_config:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def config_names(args):
    """The workloads one run measures: without --config, the headline on the
    largest single-GPU workload (the long-context layer) and a line for each of
    the other workloads."""
    if args.config:
        return [args.config]
    return [HEADLINE_CONFIG] + ([] if args.no_per_config else list(PER_CONFIGS))


def check_args(args, ap):
    """Refuses, before any GPU work, the flag combinations a step cannot honour."""
    from workloads import SPECS

    for name in config_names(args):
        shared = SPECS[name].shared_prefix_groups > 0 and args.prefix_sharing and args.q_len == 0
        if args.kv == "fp8" and (args.q_len > 0 or shared):
            ap.error(f"{name}: --kv fp8 times the plain decode path only "
                     "(add --no-prefix-sharing for shared-prefix workloads)")
        if args.splits and shared:
            # the shared-prefix call plans its own suffix partitions
            ap.error(f"{name}: --splits does not apply to the shared-prefix step "
                     "(add --no-prefix-sharing to time the plain path)")
        if args.splits and args.q_len > 0:
            ap.error("--splits does not apply to the multi-query step "
                     "(it plans its own context partitions)")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--config", default=None, choices=sorted(WORKLOAD_TEXT),
                    help="one workload only (default: the long-context layer c4 as the "
                         "headline, plus a per_config line for c2, c3, c5 and c5_bs32)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="without --config: the headline workload only")
    ap.add_argument("--splits", type=int, default=0, help="KV partitions (0 = automatic)")
    ap.add_argument("--kv", choices=["16bit", "fp8"], default="16bit",
                    help="cache element type: the workload's 16-bit type or E4M3 codes")
    ap.add_argument("--layout", choices=["nhd", "hnd"], default="nhd",
                    help="page layout: token major [blocks][bs][H_kv][d] or head major "
                         "[blocks][H_kv][bs][d]")
    ap.add_argument("--block-size", type=int, default=0,
                    help="tokens per page (0 = the workload's own)")
    ap.add_argument("--unfused", dest="fused", action="store_false",
                    help="time the step as two calls, pkv_append then the decode, instead of "
                         "the decode launch appending the new tokens itself "
                         "(pkv_append_decode_attention, the default on the plain 16-bit path)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph")
    ap.add_argument("--q-len", type=int, default=0,
                    help="query tokens per sequence for causal multi-query attention "
                         "(0 = single-token decode)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="oracle time for the headline's cpu_baseline")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="oracle work in all for --impl reference (seconds)")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=3.0,
                    help="oracle time for each per_config cpu_baseline")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-prefix-sharing", dest="prefix_sharing", action="store_false",
                    help="decode shared-prefix workloads with the plain path")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    check_args(args, ap)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
