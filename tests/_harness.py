"""Shared helpers of the GPU parity tests: build a cache on the device through
the library's append kernel, run the attention step through the C ABI, and
evaluate the oracle on the same seeded inputs (all rows or a sample)."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl

TOL = 2e-3  # max-abs error on fp16 outputs against fp64 attention over the dequantised cache


def torch():
    import torch as _t
    return _t


def build_cache(w: wl.Workload, fill: int = 0, append_tokens: int = 32768, pt=None):
    """Allocate the cache (planes filled with byte `fill`) and append every row's history."""
    t = torch()
    import mixed_attention_quantized_gb300 as mq
    cache = mq.KVCache.allocate(w.num_pages, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt, fill=fill)
    pt = wl.page_table(w) if pt is None else pt
    for r in range(w.n_rows):
        for s0 in range(0, w.seq_lens[r], append_tokens):
            s1 = min(w.seq_lens[r], s0 + append_tokens)
            k, v = wl.row_kv(w, r, s0, s1)
            slots = wl.slots(w, pt, r, s0, s1)
            mq.kv_append_quant(cache, t.from_numpy(k).cuda(), t.from_numpy(v).cuda(),
                               t.from_numpy(slots).cuda())
    return cache, pt


def run_attention(w: wl.Workload, cache, pt, q=None, window: int = 0):
    t = torch()
    import mixed_attention_quantized_gb300 as mq
    plan = mq.Plan(cache, w.num_q_heads, w.row_kinds, w.seq_lens, w.q_offsets, pt.shape[1], window=window)
    ws = mq.alloc_workspace(plan.workspace_bytes)
    qd = t.from_numpy(wl.queries(w)).cuda() if q is None else q
    o = t.full_like(qd, float("nan"))
    plan.run(qd, t.from_numpy(np.ascontiguousarray(pt)).cuda(), o, ws)
    t.cuda.synchronize()
    plan.close()
    return o.cpu().numpy()


def oracle_attention(w: wl.Workload, sel=None, threads: int = 0, window: int = 0) -> np.ndarray:
    """fp64 oracle for the packed query indices `sel` (default: all)."""
    total = w.total_q
    sel = np.arange(total) if sel is None else np.asarray(sel)
    starts = np.array(w.q_starts)
    row_of = np.searchsorted(starts, sel, side="right") - 1
    rows = sorted(set(row_of.tolist()))
    # a reduced batch holding only the rows the sample touches
    kb, vb, seq, off, qs = [], [], [], [], []
    new_index = {}
    acc = 0
    for r in rows:
        k, v = wl.row_kv(w, r)
        kb.append(oracle.quantize(w.k_fmt, k))
        vb.append(oracle.quantize(w.v_fmt, v))
        seq.append(w.seq_lens[r])
        off.append(w.q_offsets[r])
        qs.append(wl.row_q(w, r))
        new_index[r] = acc
        acc += w.q_lens[r]
    q = np.concatenate(qs, axis=0)
    sub_sel = np.array([new_index[r] + (s - w.q_starts[r]) for s, r in zip(sel, row_of)], dtype=np.int32)
    return oracle.attention(w.k_fmt, w.v_fmt, q, kb, vb, seq, off, sel=sub_sel, threads=threads, window=window)


def max_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    g = gpu.astype(np.float64)
    assert np.isfinite(g).all(), "non-finite outputs"
    return float(np.abs(g - ref).max())
