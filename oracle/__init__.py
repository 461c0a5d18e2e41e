"""CPU oracle for the mixed-batch attention step over a block-quantised KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The CUDA library
never calls it and shares no code with it: the oracle has its own fp16
conversion, its own rounding and its own attention loop (``oracle.c``).

What it computes (page "自研RDNA高併發推論引擎 以AI Max+ 395為範例", §1 and §2):

* ``quantize`` / ``dequantize``: the Q8_0 (34-byte) and Q4_0 (18-byte)
  32-element blocks of the §2 modes table, plus the plain fp16 mode;
* ``attention``: causal softmax attention in fp64 over the dequantised cache
  for chunk rows (a query slice at a position offset) and decode rows (one
  query), the row kinds that share one ForwardBatch in §1.

Pins (``tests/test_oracle_*.py``): the §2 occupancy table's byte counts,
hand-derived blocks whose fp32 arithmetic is exact, numpy's IEEE fp16
conversion, brute-force rounding on the codec, closed forms (one key, equal
keys), torch's fp64 scaled-dot-product attention for the fp16 mode, and the
decode-row == last-chunk-row invariant.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_F16, FMT_Q8_0, FMT_Q4_0 = 0, 1, 2
QK = 32
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP, no FMA contraction) and return the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            i32p = ctypes.POINTER(ctypes.c_int32)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            lib.orc_f32_to_f16_array.argtypes = [f32p, u16p, ctypes.c_int64]
            lib.orc_f16_to_f32_array.argtypes = [u16p, f32p, ctypes.c_int64]
            lib.orc_block_bytes.argtypes = [ctypes.c_int]
            lib.orc_block_bytes.restype = ctypes.c_int
            lib.orc_quantize.argtypes = [ctypes.c_int, u16p, ctypes.c_int64, u8p]
            lib.orc_quantize.restype = ctypes.c_int
            lib.orc_dequantize.argtypes = [ctypes.c_int, u8p, ctypes.c_int64, f64p]
            lib.orc_dequantize.restype = ctypes.c_int
            lib.orc_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, i32p, i32p, u16p, u8p, i64p, u8p, i64p, ctypes.c_int,
                i32p, f64p, ctypes.c_int]
            lib.orc_attention.restype = ctypes.c_int
            lib.orc_attention_window.argtypes = lib.orc_attention.argtypes + [ctypes.c_int]
            lib.orc_attention_window.restype = ctypes.c_int
            lib.orc_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def block_bytes(fmt: int) -> int:
    """Bytes of one canonical 32-element block: 64 (fp16), 34 (Q8_0), 18 (Q4_0)."""
    n = _load().orc_block_bytes(int(fmt))
    if n < 0:
        raise ValueError(f"unknown KV format {fmt}")
    return n


def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_f32_to_f16_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_f16_to_f32_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), h.size)
    return out


def quantize(fmt: int, x) -> np.ndarray:
    """Quantise fp16 data (last dim a multiple of 32) into canonical blocks.

    Returns uint8 of shape ``x.shape[:-1] + (x.shape[-1] // 32, block_bytes)``.
    """
    x = np.ascontiguousarray(x, dtype=np.float16)
    if x.shape[-1] % QK:
        raise ValueError("last dimension must be a multiple of 32")
    nblk = x.size // QK
    bb = block_bytes(fmt)
    out = np.empty(nblk * bb, dtype=np.uint8)
    bits = x.view(np.uint16)
    rc = _load().orc_quantize(int(fmt), _ptr(bits, ctypes.c_uint16), nblk, _ptr(out, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("orc_quantize failed")
    return out.reshape(x.shape[:-1] + (x.shape[-1] // QK, bb))


def dequantize(fmt: int, blocks) -> np.ndarray:
    """Canonical blocks ``[..., nb, block_bytes]`` -> float64 ``[..., nb * 32]``."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    bb = block_bytes(fmt)
    if blocks.shape[-1] != bb:
        raise ValueError("last dimension must be the block size")
    nblk = blocks.size // bb
    out = np.empty(nblk * QK, dtype=np.float64)
    rc = _load().orc_dequantize(int(fmt), _ptr(blocks, ctypes.c_uint8), nblk, _ptr(out, ctypes.c_double))
    if rc != 0:
        raise RuntimeError("orc_dequantize failed")
    return out.reshape(blocks.shape[:-2] + (blocks.shape[-2] * QK,))


def attention(fmt_k: int, fmt_v: int, q, k_blocks, v_blocks, seq_lens, q_offsets,
              sel=None, threads: int = 0, window: int = 0) -> np.ndarray:
    """fp64 causal attention over the dequantised cache.

    window:    > 0 for sliding-window attention: the query at position p sees
               keys p - window + 1 .. p only; 0 (default) sees keys 0 .. p.

    q:         fp16 ``[total_q, Hq, D]``, rows packed in order.
    k_blocks:  list (one per row) of uint8 ``[seq_len, Hkv, D/32, bb]`` canonical blocks.
    v_blocks:  same for V.
    seq_lens, q_offsets: per row; row r owns ``seq_len - q_offset`` queries.
    sel:       packed query-token indices to evaluate (default: all).
    Returns float64 ``[len(sel), Hq, D]``.
    """
    q = np.ascontiguousarray(q, dtype=np.float16)
    total_q, hq, d = q.shape
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    q_offsets = np.ascontiguousarray(q_offsets, dtype=np.int32)
    n_rows = len(seq_lens)
    if d > 512:
        raise ValueError("head_dim above 512 is not supported by the oracle")
    hkv = k_blocks[0].shape[1]
    k_all = np.concatenate([np.ascontiguousarray(kb, dtype=np.uint8).ravel() for kb in k_blocks])
    v_all = np.concatenate([np.ascontiguousarray(vb, dtype=np.uint8).ravel() for vb in v_blocks])
    k_off = np.zeros(n_rows, dtype=np.int64)
    v_off = np.zeros(n_rows, dtype=np.int64)
    ak = av = 0
    for r in range(n_rows):
        if k_blocks[r].shape[0] < seq_lens[r] or v_blocks[r].shape[0] < seq_lens[r]:
            raise ValueError(f"row {r}: fewer cached tokens than seq_len")
        k_off[r], v_off[r] = ak, av
        ak += k_blocks[r].size
        av += v_blocks[r].size
    if int((seq_lens - q_offsets).sum()) != total_q:
        raise ValueError("q rows do not match sum(seq_len - q_offset)")
    if sel is None:
        sel = np.arange(total_q, dtype=np.int32)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    out = np.empty((len(sel), hq, d), dtype=np.float64)
    rc = _load().orc_attention_window(
        int(fmt_k), int(fmt_v), d, hq, hkv, n_rows, _ptr(seq_lens, ctypes.c_int32),
        _ptr(q_offsets, ctypes.c_int32), _ptr(q.view(np.uint16), ctypes.c_uint16),
        _ptr(k_all, ctypes.c_uint8), _ptr(k_off, ctypes.c_int64), _ptr(v_all, ctypes.c_uint8),
        _ptr(v_off, ctypes.c_int64), len(sel), _ptr(sel, ctypes.c_int32),
        _ptr(out, ctypes.c_double), int(threads), int(window))
    if rc != 0:
        raise RuntimeError(f"orc_attention failed ({rc})")
    return out


def max_threads() -> int:
    return int(_load().orc_max_threads())
