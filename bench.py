#!/usr/bin/env python3
"""Benchmark of the mixed-batch attention step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. quantise-on-append of the step's new K/V (the chunk's tokens and one token
     per decode row) into the paged Q8_0 / Q4_0 cache, and
  2. the fused mixed-batch attention launch over all rows,
both through the C ABI of libmixattn.so, on one CUDA stream.

Metric: mixed-batch attention tokens/s (decode rows + chunk tokens per step),
with the attention kernel's algorithmic KV-read GB/s against the measured HBM
copy bandwidth.  Inputs (the cache: hundreds of MB) are larger than L2, so no
flush runs between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Under torchrun (N > 1) every rank runs its own independent batch (weak scaling,
no collective on the data path); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "mixed-batch attn tokens/s and KV-read GB/s (% of GB300 HBM roofline), per KV format"
L2_BYTES = 129 * 1024 * 1024


def make_workload(name: str) -> wl.Workload:
    if name == "serving_mix":
        return wl.serving_mix()
    if name == "tiny":
        return wl.tiny()
    if name == "long_session_q8":
        return wl.long_session(wl.FMT_Q8_0)
    if name == "long_session_q4":
        return wl.long_session(wl.FMT_Q4_0)
    if name == "fairness":
        return wl.fairness()
    if name == "verify_q8":
        return wl.verify_batch(wl.FMT_Q8_0)
    if name == "verify_q4":
        return wl.verify_batch(wl.FMT_Q4_0)
    if name.startswith("sweep_"):  # sweep_<batch>_<ctx>_<f16|q8_0|q4_0|k8v4|k4v8>
        _, b, c, f = name.split("_", 3)
        mixed = {"k8v4": (wl.FMT_Q8_0, wl.FMT_Q4_0), "k4v8": (wl.FMT_Q4_0, wl.FMT_Q8_0)}
        if f in mixed:
            return wl.decode_sweep(int(b), int(c), *mixed[f])
        fmt = {v: k for k, v in wl.FMT_NAMES.items()}[f]
        return wl.decode_sweep(int(b), int(c), fmt)
    raise SystemExit(f"unknown workload {name}")


# The other KV formats of the metric, measured after the headline workload by a
# default run (one sub-object each): the tensor-bound fairness chunk (Q4_0), the
# long session in both formats, one fp16 and one K8V4 decode-sweep point, and a
# batch of speculative-verify rows (Q8_0).
FORMAT_WORKLOADS = [("fairness", 10), ("long_session_q8", 50), ("long_session_q4", 50),
                    ("sweep_4_65536_f16", 50), ("sweep_16_8192_k8v4", 50), ("verify_q8", 50)]


# --------------------------------------------------------------------------
# Algorithmic work of one step (what the path must touch at least once)
# --------------------------------------------------------------------------
def kv_bytes_per_token(fmt: int, d: int, hkv: int) -> int:
    per_head = {wl.FMT_F16: 2 * d, wl.FMT_Q8_0: d + d // 16, wl.FMT_Q4_0: d // 2 + d // 16}[fmt]
    return per_head * hkv


def algorithmic(w: wl.Workload) -> dict:
    kv_tok = kv_bytes_per_token(w.k_fmt, w.head_dim, w.num_kv_heads) + \
        kv_bytes_per_token(w.v_fmt, w.head_dim, w.num_kv_heads)
    kv = sum(w.seq_lens) * kv_tok
    qo = 2 * w.total_q * w.num_q_heads * w.head_dim * 2
    pt = sum(w.pages_for(r) for r in range(w.n_rows)) * 4
    flops = 0
    for r in range(w.n_rows):
        if w.row_kinds[r] == wl.ROW_CHUNK:
            p0, p1 = w.q_offsets[r], w.seq_lens[r]
            flops += 4 * w.head_dim * w.num_q_heads * ((p1 * (p1 + 1) - p0 * (p0 + 1)) // 2)
    n_new = w.total_q
    app_read = 2 * n_new * w.num_kv_heads * w.head_dim * 2 + 4 * n_new
    app_write = n_new * (kv_tok)
    tokens = w.total_q
    return {"kv_bytes": kv, "attn_bytes": kv + qo + pt, "chunk_flops": flops, "append_bytes": app_read + app_write,
            "tokens": tokens, "kv_bytes_per_token": kv_tok}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "tflops": d["bf16_tflops"], "tflops_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixed_attention_quantized_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from an ncu capture, if the
    kernel sources are unchanged since it was taken (profiles/dram_traffic.json)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return int(e["bytes_per_launch"])
    except Exception:
        return None
    return None


# --------------------------------------------------------------------------
# Clock sampling during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# Multi-process helpers (one process per GPU; replicas, no data-path collective)
# --------------------------------------------------------------------------
def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_step_per_rank: int, world: int, ms_per_step: float) -> float:
    """Tokens of all ranks per second: every rank runs its own batch each step."""
    return world * tokens_per_step_per_rank / (ms_per_step / 1e3)


def emit(line: dict, rank: int) -> None:
    """Rank 0 prints the one JSON line; the other ranks print nothing."""
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def step_inputs(w: wl.Workload, pt: np.ndarray):
    """New K/V of the step (chunk tokens + one per decode row) and their slots."""
    ks, vs, ss = [], [], []
    for r in range(w.n_rows):
        k, v = wl.row_kv(w, r, w.q_offsets[r], w.seq_lens[r])
        ks.append(k)
        vs.append(v)
        ss.append(wl.slots(w, pt, r, w.q_offsets[r], w.seq_lens[r]))
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(ss).astype(np.int32)


def prepare(w: wl.Workload, dev):
    """The cache with every row's history appended, the step's inputs on the
    device and a plan with its workspace."""
    import torch
    import mixed_attention_quantized_gb300 as mq
    cache = mq.KVCache.allocate(w.num_pages, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt, device=dev)
    pt = wl.page_table(w)
    for r in range(w.n_rows):
        for s0 in range(0, w.seq_lens[r], 65536):
            s1 = min(w.seq_lens[r], s0 + 65536)
            k, v = wl.row_kv(w, r, s0, s1)
            mq.kv_append_quant(cache, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev),
                               torch.from_numpy(wl.slots(w, pt, r, s0, s1)).to(dev))
    k_new, v_new, slots = step_inputs(w, pt)
    d = {"cache": cache, "pt": pt, "k_new": k_new, "v_new": v_new, "slots": slots, "q_host": wl.queries(w)}
    d["kd"] = torch.from_numpy(k_new).to(dev)
    d["vd"] = torch.from_numpy(v_new).to(dev)
    d["sd"] = torch.from_numpy(slots).to(dev)
    d["qd"] = torch.from_numpy(d["q_host"]).to(dev)
    d["ptd"] = torch.from_numpy(pt).to(dev)
    d["od"] = torch.empty_like(d["qd"])
    d["plan"] = mq.Plan(cache, w.num_q_heads, w.row_kinds, w.seq_lens, w.q_offsets, pt.shape[1])
    d["ws"] = mq.alloc_workspace(d["plan"].workspace_bytes, dev)
    return d


def time_steps(d, steps: int, warmup: int, dev, stream):
    """Per-step CUDA-event times (ms) of the append and the attention (upload +
    fused launch) on the launching stream, after `warmup` untimed steps."""
    import torch
    import mixed_attention_quantized_gb300 as mq
    cache, plan = d["cache"], d["plan"]
    for _ in range(warmup):
        mq.kv_append_quant(cache, d["kd"], d["vd"], d["sd"], stream)
        plan.run(d["qd"], d["ptd"], d["od"], d["ws"], stream)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        mq.kv_append_quant(cache, d["kd"], d["vd"], d["sd"], stream)
        ev[i][1].record(stream)
        plan.run(d["qd"], d["ptd"], d["od"], d["ws"], stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    return ([ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)],
            [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)])


def roofline_of(w: wl.Workload, alg: dict, attn_s: float, peaks: dict, traffic_key: str) -> dict:
    t_bytes = alg["attn_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flops = alg["chunk_flops"] / (peaks["tflops"] * 1e12)
    if t_bytes >= t_flops:
        gbs = alg["attn_bytes"] / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"]}
    else:
        tf = alg["chunk_flops"] / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": tf, "peak": peaks["tflops"], "unit": "TFLOP/s",
                "frac": tf / peaks["tflops"]}
    roof["traffic"] = measured_traffic(traffic_key)
    roof["peak_source"] = peaks["source"]
    roof["roofline_time_frac"] = max(t_bytes, t_flops) / attn_s
    return roof


def measure_format(name: str, steps: int, warmup: int, dev, stream, peaks: dict, stride: int,
                   cpu: bool) -> dict:
    """One sub-object of the default run: a workload in another KV format."""
    import torch
    w = make_workload(name)
    alg = algorithmic(w)
    d = prepare(w, dev)
    app_ms, attn_ms = time_steps(d, steps, warmup, dev, stream)
    d["plan"].close()
    del d
    torch.cuda.empty_cache()
    attn = sum(attn_ms) / len(attn_ms)
    app = sum(app_ms) / len(app_ms)
    out = {"workload": w.name, "kv_format": f"K={wl.FMT_NAMES[w.k_fmt]},V={wl.FMT_NAMES[w.v_fmt]}",
           "steps": steps, "tokens_per_step": alg["tokens"],
           "value": alg["tokens"] / ((attn + app) / 1e3), "unit": "tokens/s",
           "attention_us": attn * 1e3, "append_us": app * 1e3,
           "kv_gbs": alg["kv_bytes"] / (attn / 1e3) / 1e9,
           "kv_frac_of_hbm": alg["kv_bytes"] / (attn / 1e3) / 1e9 / peaks["hbm_gbs"],
           "chunk_tflops": alg["chunk_flops"] / (attn / 1e3) / 1e12,
           "roofline": roofline_of(w, alg, attn / 1e3, peaks, name)}
    if cpu:
        out["cpu_baseline"] = cpu_baseline(w, stride if w.name != "fairness" else 64)
    return out


def run_gpu(args, rank: int, world: int, local_rank: int) -> dict:
    import torch
    import mixed_attention_quantized_gb300 as mq

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = make_workload(args.workload)
    alg = algorithmic(w)
    # the history of every row is in the cache; each step appends its new tokens again
    d = prepare(w, dev)
    cache, pt, plan, ws = d["cache"], d["pt"], d["plan"], d["ws"]
    k_new, v_new, slots, q_host = d["k_new"], d["v_new"], d["slots"], d["q_host"]
    kd, vd, sd, qd, ptd, od = d["kd"], d["vd"], d["sd"], d["qd"], d["ptd"], d["od"]
    del d
    stream = torch.cuda.current_stream(dev)

    def step():
        mq.kv_append_quant(cache, kd, vd, sd, stream)
        plan.run(qd, ptd, od, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if mq.device_error(clear=True):
        raise RuntimeError("device error word set during warm-up")

    # ---- device-timed region: K steps, events per phase on the launching stream ----
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed work
    t0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        mq.kv_append_quant(cache, kd, vd, sd, stream)
        ev[i][1].record(stream)
        plan.run(qd, ptd, od, ws, stream)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), device=dev)
    app_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    attn_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    attn_mean = sum(attn_ms) / K
    app_mean = sum(app_ms) / K

    # ---- end-to-end: host buffers in, result out, through the same API ----
    # Every step copies its own inputs in from pinned host memory and reads its
    # output back; as a serving loop would, the copies of one step overlap the
    # compute of its neighbours: inputs and outputs are double-buffered on the
    # device, host-to-device copies run on one stream, device-to-host on
    # another, ordered by events (the cache append of a step still follows the
    # attention of the previous one on the compute stream).
    # The step's inputs travel as one pinned blob (K, V, slots, q, page table at
    # 256-byte aligned offsets) into one of two device blobs holding typed views.
    parts = [np.ascontiguousarray(x) for x in (k_new, v_new, slots, q_host, pt)]
    offs, total = [], 0
    for x in parts:
        offs.append(total)
        total += (x.nbytes + 255) // 256 * 256
    blob_pin = torch.empty(total, dtype=torch.uint8).pin_memory()
    for x, o in zip(parts, offs):
        blob_pin[o:o + x.nbytes].copy_(torch.from_numpy(x.view(np.uint8).reshape(-1)))

    def views(blob):
        out = []
        for x, o, like in zip(parts, offs, (kd, vd, sd, qd, ptd)):
            out.append(blob[o:o + x.nbytes].view(like.dtype).view(like.shape))
        return out

    dev_blobs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    bufs = [views(b) + [torch.empty_like(od)] for b in dev_blobs]
    o_pin = [torch.empty(od.shape, dtype=od.dtype).pin_memory() for _ in range(2)]
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    k_e2e = max(2, min(K, 200))
    ev_pool = [[torch.cuda.Event() for _ in range(3)] for _ in range(k_e2e + 4)]

    def e2e_run(n):
        for i in range(n):
            in_ready, done, out_read = ev_pool[i]
            kb, vb, sb, qb, pb, ob = bufs[i % 2]
            if i >= 2:
                h2d_stream.wait_event(ev_pool[i - 2][1])  # step i-2 is done reading this input set
            with torch.cuda.stream(h2d_stream):
                dev_blobs[i % 2].copy_(blob_pin, non_blocking=True)
            in_ready.record(h2d_stream)
            stream.wait_event(in_ready)
            if i >= 2:
                stream.wait_event(ev_pool[i - 2][2])  # the output of step i-2 has been read back
            mq.kv_append_quant(cache, kb, vb, sb, stream)
            plan.run(qb, pb, ob, ws, stream)
            done.record(stream)
            d2h_stream.wait_event(done)
            with torch.cuda.stream(d2h_stream):
                o_pin[i % 2].copy_(ob, non_blocking=True)
            out_read.record(d2h_stream)
        return ev_pool[n - 1][2]

    e2e_run(4)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    d2h_stream.wait_event(e0)
    last = e2e_run(k_e2e)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / k_e2e
    h2d = total  # the step's inputs as copied (their bytes plus 256-byte alignment padding)
    d2h = od.numel() * od.element_size()
    # parity of the last timed output against the pinned copy (same buffer, same values)
    dev_err = mq.device_error(clear=True)

    plan_info = plan.info()
    plan.close()
    del cache, bufs, dev_blobs, kd, vd, sd, qd, ptd, od, ws
    torch.cuda.empty_cache()
    # the other KV formats (default run on one GPU): each its own sub-object
    formats = []
    if args.formats and world == 1:
        for name, steps in FORMAT_WORKLOADS:
            if name == args.workload:
                continue
            formats.append(measure_format(name, min(steps, args.steps), 3, dev, stream, load_peaks(),
                                          args.oracle_stride, not args.no_cpu_baseline))
        dev_err |= mq.device_error(clear=True)
    return {"w": w, "alg": alg, "total_ms": total_ms, "attn_ms": attn_mean, "append_ms": app_mean,
            "attn_ms_list": attn_ms, "clocks": clocks, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h,
            "plan": plan_info, "device_error": dev_err, "formats": formats}


# --------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# --------------------------------------------------------------------------
def oracle_sample(w: wl.Workload, stride: int):
    """Every decode row and every `stride`-th chunk token of the workload."""
    sel = []
    for r in range(w.n_rows):
        s0, n = w.q_starts[r], w.q_lens[r]
        sel.extend(range(s0, s0 + n, 1 if w.row_kinds[r] == wl.ROW_DECODE else stride))
    return np.array(sel, dtype=np.int32)


def oracle_prepare(w: wl.Workload, sel: np.ndarray):
    import oracle
    starts = np.array(w.q_starts)
    row_of = np.searchsorted(starts, sel, side="right") - 1
    rows = sorted(set(row_of.tolist()))
    kv = {r: wl.row_kv(w, r) for r in rows}
    qs = {r: wl.row_q(w, r) for r in rows}
    oracle.build()
    return rows, kv, qs, row_of


def oracle_time(w: wl.Workload, sel: np.ndarray, prepared, threads: int) -> float:
    """Seconds the oracle takes for the sample: quantise the sampled rows' new
    tokens (the append) and run fp64 attention for the sampled queries."""
    import oracle
    rows, kv, qs, row_of = prepared
    t0 = time.perf_counter()
    kb, vb, seq, off, q, index = [], [], [], [], [], {}
    acc = 0
    for r in rows:
        k, v = kv[r]
        kb.append(oracle.quantize(w.k_fmt, k))
        vb.append(oracle.quantize(w.v_fmt, v))
        seq.append(w.seq_lens[r])
        off.append(w.q_offsets[r])
        q.append(qs[r])
        index[r] = acc
        acc += w.q_lens[r]
    sub = np.array([index[r] + (s - w.q_starts[r]) for s, r in zip(sel, row_of)], dtype=np.int32)
    oracle.attention(w.k_fmt, w.v_fmt, np.concatenate(q), kb, vb, seq, off, sel=sub, threads=threads)
    return time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w: wl.Workload, stride: int, one_core: bool = False) -> dict:
    """The oracle timed on all host threads over a bounded sample; with `one_core`
    the same sample is timed again on one thread."""
    sel = oracle_sample(w, stride)
    prep = oracle_prepare(w, sel)
    cores = cpu_cores()
    secs = oracle_time(w, sel, prep, cores)
    out = {"value": len(sel) / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": f"{len(sel)} of {w.total_q} query tokens (all decode rows, every {stride}th chunk token), "
                     f"full history of each sampled row quantised; {secs:.1f} s"}
    if one_core and cores > 1:
        secs1 = oracle_time(w, sel, prep, 1)
        out["one_core"] = {"value": len(sel) / secs1, "unit": "tokens/s", "cores": 1, "seconds": round(secs1, 1)}
    return out


# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="serving_mix")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--oracle-stride", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-formats", dest="formats", action="store_false",
                    help="skip the other KV formats' sub-measurements of the default run")
    args = ap.parse_args()
    if args.workload != "serving_mix":
        args.formats = False
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        w = make_workload(args.workload)
        sel = oracle_sample(w, args.oracle_stride)
        prep = oracle_prepare(w, sel)
        cores = cpu_cores()
        # each step is one bounded sample (~3 s of oracle work at the default stride):
        # 3 to 10 untimed warm-up steps (W, bounded), then up to K timed steps within
        # ~2 minutes
        warm = max(3, min(args.warmup, 10))
        for _ in range(warm):
            oracle_time(w, sel, prep, cores)
        times = [oracle_time(w, sel, prep, cores)]
        while len(times) < args.steps and sum(times) + times[-1] <= 120.0:
            times.append(oracle_time(w, sel, prep, cores))
        secs = sum(times) / len(times)
        val = len(sel) / secs
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": len(times), "steps_requested": args.steps, "warmup": warm,
                "warmup_requested": args.warmup, "ms_per_step": secs * 1e3,
                "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "kv_format": f"K={wl.FMT_NAMES[w.k_fmt]},V={wl.FMT_NAMES[w.v_fmt]}"},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{len(sel)} of {w.total_q} query tokens per step"},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        emit(line, rank)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    w, alg = res["w"], res["alg"]
    peaks = load_peaks()
    K = args.steps
    ms_step = res["total_ms"] / K
    value = whole_job_tokens_per_s(alg["tokens"], world, ms_step)
    attn_s = res["attn_ms"] / 1e3
    kv_gbs = alg["kv_bytes"] / attn_s / 1e9
    tflops = alg["chunk_flops"] / attn_s / 1e12
    roof = roofline_of(w, alg, attn_s, peaks, args.workload)  # traffic keyed by the workload's CLI name
    roof["kernel"] = "mixattn fused attention (one launch per step)"

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": w.name, "kv_format": f"K={wl.FMT_NAMES[w.k_fmt]},V={wl.FMT_NAMES[w.v_fmt]}",
                   "heads": f"{w.num_q_heads}q/{w.num_kv_heads}kv", "head_dim": w.head_dim,
                   "rows": f"{w.row_kinds.count(wl.ROW_DECODE)} decode + {w.row_kinds.count(wl.ROW_CHUNK)} chunk",
                   "tokens_per_step": alg["tokens"], "kv_bytes": alg["kv_bytes"],
                   "l2": "inputs larger than L2, no flush" if alg["kv_bytes"] > L2_BYTES else "L2-resident (small case)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_gbs": kv_gbs, "kv_frac_of_hbm": kv_gbs / peaks["hbm_gbs"],
        "attention_us": res["attn_ms"] * 1e3, "append_us": res["append_ms"] * 1e3,
        "append_gbs": alg["append_bytes"] / (res["append_ms"] / 1e3) / 1e9,
        "chunk_tflops": tflops,
        "roofline": roof,
        "e2e": {"value": whole_job_tokens_per_s(alg["tokens"], world, res["e2e_ms"]), "unit": "tokens/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]},
        "gpu_launches": 3 * K,  # per step: append, tile-list upload, attention
        "clocks": res["clocks"],
        "plan": res["plan"],
        "device_error": res["device_error"],
    }
    if res["formats"]:
        line["formats"] = res["formats"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.oracle_stride, one_core=True)
    emit(line, rank)


if __name__ == "__main__":
    main()
