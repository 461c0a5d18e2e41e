"""Seeded synthetic inputs for the mixed-batch attention step.

This module only draws random numbers and lays out pages; it holds none of the
method's arithmetic (no quantisation, no attention).  The CUDA path (through
``mixed_attention_quantized_gb300``) and the CPU oracle (``oracle``) both take
their inputs from here, and from nowhere else.

Recipe (each workload mirrors one of the synthetic cases the attention step is
measured on; the reference pages measure whole models on prompts that are not
available here, so these stand in for them):

* Q, K, V are fp32 N(0, 1) draws rounded to fp16 (numpy PCG64).
* Every tensor is drawn in blocks of ``TOKEN_BLOCK`` tokens, each block from
  its own ``SeedSequence([seed, row, tensor, block])``, so any token range of
  any row can be regenerated on its own (sampled checks at full size).
* "K outlier channels": per kv head, ``n_outlier`` channel indices drawn from
  the workload seed have their K values multiplied by ``alpha`` before the
  rounding to fp16.
* Contexts are integers drawn uniformly (inclusive bounds) from the workload
  seed; the physical page pool is a seeded random permutation, so consecutive
  logical pages of a row land on scattered physical pages.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

FMT_F16, FMT_Q8_0, FMT_Q4_0 = 0, 1, 2
ROW_DECODE, ROW_CHUNK = 0, 1
FMT_NAMES = {FMT_F16: "f16", FMT_Q8_0: "q8_0", FMT_Q4_0: "q4_0"}
TOKEN_BLOCK = 4096
PAGE = 32
FP16_MAX = 65504.0  # largest finite fp16 value

# tensor ids for the seed sequences
_T_K, _T_V, _T_Q, _T_OUTLIER, _T_ROWS, _T_PAGES = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    k_fmt: int
    v_fmt: int
    seed: int
    row_kinds: List[int]
    seq_lens: List[int]
    q_offsets: List[int]
    n_outlier: int = 0
    alpha: float = 8.0
    page_size: int = PAGE
    spare_pages: int = 0
    v_gain: float = 1.0  # V values multiplied by this (then clipped to the fp16 range, +-65504)
    q_gain: float = 1.0  # queries multiplied by this (sharper scores)
    k_gain: float = 1.0  # K values multiplied by this (then clipped to the fp16 range)

    @property
    def n_rows(self) -> int:
        return len(self.seq_lens)

    @property
    def q_lens(self) -> List[int]:
        return [s - o for s, o in zip(self.seq_lens, self.q_offsets)]

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def q_starts(self) -> List[int]:
        out, acc = [], 0
        for n in self.q_lens:
            out.append(acc)
            acc += n
        return out

    def pages_for(self, r: int) -> int:
        return -(-self.seq_lens[r] // self.page_size)

    @property
    def max_pages(self) -> int:
        return max(self.pages_for(r) for r in range(self.n_rows))

    @property
    def num_pages(self) -> int:
        return sum(self.pages_for(r) for r in range(self.n_rows)) + self.spare_pages


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def outlier_channels(w: Workload) -> np.ndarray:
    """``[Hkv, n_outlier]`` channel indices whose K values are scaled by alpha."""
    if w.n_outlier <= 0:
        return np.zeros((w.num_kv_heads, 0), dtype=np.int64)
    rng = _rng(w.seed, _T_OUTLIER)
    return np.stack([rng.choice(w.head_dim, size=w.n_outlier, replace=False)
                     for _ in range(w.num_kv_heads)])


def _normal_f16(key: Tuple[int, ...], shape, scale_cols=None, gain: float = 1.0) -> np.ndarray:
    x = _rng(*key).standard_normal(size=shape, dtype=np.float32)
    if scale_cols is not None:
        x = x * scale_cols
    if gain != 1.0:
        x = np.clip(x * np.float32(gain), -FP16_MAX, FP16_MAX)
    return x.astype(np.float16)


def _blocked(w: Workload, r: int, tensor: int, start: int, stop: int, width_shape,
             scale_cols=None, gain: float = 1.0) -> np.ndarray:
    out = np.empty((stop - start,) + tuple(width_shape), dtype=np.float16)
    b0, b1 = start // TOKEN_BLOCK, (stop - 1) // TOKEN_BLOCK if stop > start else -1
    for b in range(b0, b1 + 1):
        lo, hi = b * TOKEN_BLOCK, (b + 1) * TOKEN_BLOCK
        blk = _normal_f16((w.seed, r, tensor, b), (TOKEN_BLOCK,) + tuple(width_shape), scale_cols, gain)
        s, e = max(lo, start), min(hi, stop)
        out[s - start:e - start] = blk[s - lo:e - lo]
    return out


def row_kv(w: Workload, r: int, start: int = 0, stop: Optional[int] = None):
    """fp16 K and V ``[stop - start, Hkv, D]`` of row r's tokens start..stop-1."""
    stop = w.seq_lens[r] if stop is None else stop
    shape = (w.num_kv_heads, w.head_dim)
    cols = None
    if w.n_outlier > 0:
        cols = np.ones(shape, dtype=np.float32)
        for g, chans in enumerate(outlier_channels(w)):
            cols[g, chans] = np.float32(w.alpha)
    k = _blocked(w, r, _T_K, start, stop, shape, cols, gain=w.k_gain)
    v = _blocked(w, r, _T_V, start, stop, shape, gain=w.v_gain)
    return k, v


def row_q(w: Workload, r: int) -> np.ndarray:
    """fp16 queries ``[q_len, Hq, D]`` of row r (positions q_offset .. seq_len-1)."""
    return _blocked(w, r, _T_Q, w.q_offsets[r], w.seq_lens[r], (w.num_q_heads, w.head_dim), gain=w.q_gain)


def queries(w: Workload) -> np.ndarray:
    """All queries packed row after row: ``[total_q, Hq, D]`` fp16."""
    return np.concatenate([row_q(w, r) for r in range(w.n_rows)], axis=0)


def page_table(w: Workload) -> np.ndarray:
    """``[n_rows, max_pages]`` int32 physical page ids; unused entries are -1."""
    perm = _rng(w.seed, _T_PAGES).permutation(w.num_pages).astype(np.int32)
    pt = np.full((w.n_rows, w.max_pages), -1, dtype=np.int32)
    acc = 0
    for r in range(w.n_rows):
        n = w.pages_for(r)
        pt[r, :n] = perm[acc:acc + n]
        acc += n
    return pt


def slots(w: Workload, pt: np.ndarray, r: int, start: int, stop: int) -> np.ndarray:
    """Physical slot (page * page_size + offset) of row r's tokens start..stop-1."""
    t = np.arange(start, stop, dtype=np.int64)
    return (pt[r, t // w.page_size].astype(np.int64) * w.page_size + t % w.page_size).astype(np.int32)


# --------------------------------------------------------------------------
# The measured workloads.
# --------------------------------------------------------------------------

def tiny(k_fmt: int = FMT_Q8_0, v_fmt: Optional[int] = None) -> Workload:
    """1 layer, 4 q / 1 kv heads, head_dim 64: decode ctx 100 and 300, chunk of 64 at 128."""
    return Workload("tiny", 4, 1, 64, k_fmt, k_fmt if v_fmt is None else v_fmt, seed=0,
                    row_kinds=[ROW_DECODE, ROW_DECODE, ROW_CHUNK],
                    seq_lens=[100, 300, 192], q_offsets=[99, 299, 128])


def serving_mix(k_fmt: int = FMT_Q8_0, v_fmt: Optional[int] = None, chunk: int = 2048,
                n_decode: int = 16) -> Workload:
    """32 q / 8 kv heads, D 128: 16 decode rows ctx U[1024, 32768] + a 2048-token chunk at 0."""
    seed = 1000
    ctx = _rng(seed, _T_ROWS).integers(1024, 32768, size=n_decode, endpoint=True)
    seq = [int(c) for c in ctx] + [chunk]
    return Workload("serving_mix", 32, 8, 128, k_fmt, k_fmt if v_fmt is None else v_fmt, seed,
                    row_kinds=[ROW_DECODE] * n_decode + [ROW_CHUNK], seq_lens=seq,
                    q_offsets=[s - 1 for s in seq[:-1]] + [0], n_outlier=3, alpha=8.0)


def long_session(k_fmt: int = FMT_Q8_0, v_fmt: Optional[int] = None,
                 long_ctx: int = 262144) -> Workload:
    """1 decode row at ctx 262144 + 15 decode rows ctx U[512, 8192]."""
    seed = 2000
    ctx = _rng(seed, _T_ROWS).integers(512, 8192, size=15, endpoint=True)
    seq = [long_ctx] + [int(c) for c in ctx]
    return Workload("long_session", 32, 8, 128, k_fmt, k_fmt if v_fmt is None else v_fmt, seed,
                    row_kinds=[ROW_DECODE] * 16, seq_lens=seq, q_offsets=[s - 1 for s in seq])


def append_batch(k_fmt: int = FMT_Q8_0, v_fmt: Optional[int] = None, n_new: int = 2048) -> Workload:
    """One fresh sequence of 2048 new tokens (the append timing of the long-session case)."""
    return Workload("append_2048", 32, 8, 128, k_fmt, k_fmt if v_fmt is None else v_fmt, seed=2500,
                    row_kinds=[ROW_CHUNK], seq_lens=[n_new], q_offsets=[0])


def fairness(k_fmt: int = FMT_Q4_0, v_fmt: Optional[int] = None, offset: int = 200000,
             chunk: int = 2048) -> Workload:
    """A 2048-token chunk at offset 200000 + 16 decode rows ctx U[2048, 16384], Q4_0 K and V."""
    seed = 3000
    ctx = _rng(seed, _T_ROWS).integers(2048, 16384, size=16, endpoint=True)
    seq = [int(c) for c in ctx] + [offset + chunk]
    return Workload("fairness", 32, 8, 128, k_fmt, k_fmt if v_fmt is None else v_fmt, seed,
                    row_kinds=[ROW_DECODE] * 16 + [ROW_CHUNK], seq_lens=seq,
                    q_offsets=[s - 1 for s in seq[:-1]] + [offset])


def verify_batch(k_fmt: int = FMT_Q8_0, v_fmt: Optional[int] = None, n_rows: int = 16) -> Workload:
    """Speculative-verify rows: 16 rows of 4..16 draft tokens each (causal, at the
    end of a context of U[8192, 32768] tokens), 32 q / 8 kv heads, D 128."""
    seed = 5000
    rng = _rng(seed, _T_ROWS)
    ctx = rng.integers(8192, 32768, size=n_rows, endpoint=True)
    nq = rng.integers(4, 16, size=n_rows, endpoint=True)
    seq = [int(c) + int(n) for c, n in zip(ctx, nq)]
    return Workload("verify", 32, 8, 128, k_fmt, k_fmt if v_fmt is None else v_fmt, seed,
                    row_kinds=[ROW_CHUNK] * n_rows, seq_lens=seq, q_offsets=[int(c) for c in ctx])


def decode_sweep(batch: int, ctx: int, fmt: int, v_fmt: Optional[int] = None) -> Workload:
    """``batch`` decode rows all at ``ctx``, 32 q / 8 kv heads, D 128 (K format
    ``fmt``; V format ``v_fmt``, default the same)."""
    idx = {1: 0, 4: 1, 16: 2, 64: 3}.get(batch, 4) * 2 + (0 if ctx <= 8192 else 1)
    seed = 4000 + idx
    return Workload(f"decode_sweep_b{batch}_ctx{ctx}", 32, 8, 128, fmt, fmt if v_fmt is None else v_fmt, seed,
                    row_kinds=[ROW_DECODE] * batch, seq_lens=[ctx] * batch,
                    q_offsets=[ctx - 1] * batch)


def custom(name: str, hq: int, hkv: int, d: int, k_fmt: int, v_fmt: int, seed: int,
           rows: List[Tuple[int, int, int]], n_outlier: int = 0, alpha: float = 8.0,
           spare_pages: int = 0, v_gain: float = 1.0, q_gain: float = 1.0,
           k_gain: float = 1.0) -> Workload:
    """Free-form workload; rows are (kind, seq_len, q_offset)."""
    return Workload(name, hq, hkv, d, k_fmt, v_fmt, seed, [r[0] for r in rows],
                    [r[1] for r in rows], [r[2] for r in rows], n_outlier, alpha,
                    spare_pages=spare_pages, v_gain=v_gain, q_gain=q_gain, k_gain=k_gain)
